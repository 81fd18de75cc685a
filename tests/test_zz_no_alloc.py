"""The allocation-free sampling entry point, called through the C ABI.

spec_verify_sample_static keeps its per-row records in a static device array
inside the library, for callers that cannot allocate device memory while
they verify a round. Its outputs must equal those of spec_verify_sample with
a caller workspace, on two calls in a row (the array keeps the previous
call's contents, which must not leak into the next result). Collected last
(file name) so that a failure here stops a run only after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def _static_fn(lib):
    f = lib.spec_verify_sample_static
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.restype = I
    f.argtypes = [P, I, P, I, I, P, P, I, I, I, F, P, P, P, P, P, P]
    return f


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("name,over", [
    ("small", dict(B=16, ctx=("fixed", (64,) * 16), V=4099, logit_dtype="bf16")),
    ("llama3_8b_rows", dict(B=4, ctx=("fixed", (64,) * 4), V=128256, K=5, logit_dtype="bf16")),
])
def test_static_entry_point_matches_workspace_entry_point(name, over):
    assert torch.cuda.is_available()
    import speculative_verify_paged_gb300 as sv
    sv.build()
    lib = sv.load_library()
    fn = _static_fn(lib)
    cfg = workloads.CONFIGS["tiny"].with_(**over)
    s = workloads.make_sampling_inputs(cfg, seed=21, device="cuda")
    ref_tok, ref_nac, ref_p, ref_q = sv.spec_verify_sample(s["target_logits"], s["draft_logits"],
                                                           s["draft_tokens"], s["uniforms"])
    torch.cuda.synchronize()
    B, K = cfg.B, cfg.K
    outs = []
    for call in range(2):   # outputs allocated up front: the checked calls run with nothing new allocated
        outs.append((torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda"),
                     torch.full((B,), -7, dtype=torch.int32, device="cuda"),
                     torch.zeros((B, K), dtype=torch.float32, device="cuda"),
                     torch.zeros((B, K), dtype=torch.float32, device="cuda"),
                     torch.zeros(1, dtype=torch.int32, device="cuda")))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # a warm-up call: the first call on a device resolves the array's address
    warm = outs[0]
    assert fn(_ptr(s["target_logits"]), sv.SV_BF16, _ptr(s["draft_logits"]), sv.SV_BF16, 0,
              _ptr(s["draft_tokens"]), _ptr(s["uniforms"]), B, K, cfg.V, 1.0, _ptr(warm[0]), _ptr(warm[1]),
              _ptr(warm[2]), _ptr(warm[3]), _ptr(warm[4]), stream) == 0, lib.sv_last_error_string()
    torch.cuda.synchronize()
    for t, v in zip(warm, (-7, -7, 0, 0, 0)):
        t.fill_(v)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    alloc0 = torch.cuda.memory_allocated()
    for call in range(2):
        tok, nac, p, q, status = outs[call]
        rc = fn(_ptr(s["target_logits"]), sv.SV_BF16, _ptr(s["draft_logits"]), sv.SV_BF16, 0,
                _ptr(s["draft_tokens"]), _ptr(s["uniforms"]), B, K, cfg.V, 1.0, _ptr(tok), _ptr(nac),
                _ptr(p), _ptr(q), _ptr(status), stream)
        assert rc == 0, lib.sv_last_error_string()
        torch.cuda.synchronize()
        # nothing was allocated: neither through torch's caching allocator nor
        # on the device as a whole
        assert torch.cuda.memory_allocated() == alloc0
        assert torch.cuda.mem_get_info()[0] == free0, "device memory changed across the call"
        assert int(status.item()) == 0
        assert torch.equal(tok, ref_tok), "call %d: tokens differ" % call
        assert torch.equal(nac, ref_nac), "call %d: accepted lengths differ" % call
        assert np.allclose(p.cpu().numpy(), ref_p.cpu().numpy(), rtol=1e-5, atol=0)
        assert np.allclose(q.cpu().numpy(), ref_q.cpu().numpy(), rtol=1e-5, atol=0)


def test_static_entry_point_rejects_oversized_batches():
    import speculative_verify_paged_gb300 as sv
    sv.build()
    lib = sv.load_library()
    fn = _static_fn(lib)
    fake = ctypes.c_void_p(0x1000)
    rc = fn(fake, sv.SV_BF16, fake, sv.SV_BF16, 0, fake, fake, 30000, 4, 1000, 1.0, fake, fake, None, None, None,
            None)
    assert rc == 2   # SV_ERR_UNSUPPORTED
    assert b"static scratch" in lib.sv_last_error_string()
