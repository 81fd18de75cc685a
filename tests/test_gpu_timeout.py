"""Bounded device waits that run out, on the GPU, without a fault.

With the test hooks a launch withholds a signal (the attention producers
issue no K/V copies; CTA 0 of the sampling pass's float-float grid does not
arrive at its barriers), so the waits on it can only end by their limit
(set to 2 ms here). The waiting kernel must
set SV_DEV_TIMEOUT in the call's device status and return with nothing in
flight, and the next call on the same stream, with the hooks cleared, must
be correct.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oatt
from oracle import sampling as osamp
from parity_utils import attn_tolerance, compare_sampling

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sv():
    import speculative_verify_paged_gb300 as sv
    sv.load_library()
    yield sv
    sv.test_hooks(0, 0)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_attention_wait_runs_out_then_next_call_is_correct(sv, kv):
    cfg = workloads.CONFIGS["tiny"].with_(kv_dtype=kv, q_dtype="bf16", d_head=128, ctx=("fixed", (300, 77)))
    a = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in workloads.make_attention_inputs(cfg, 2).items()}
    args = (a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["seq_lens"], 1 / math.sqrt(cfg.d_head),
            a["k_scale"], a["v_scale"])
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    try:
        sv.test_hooks(2_000_000, sv.SV_TEST_WITHHOLD_COPIES)
        sv.spec_verify_attn(*args, status=st)
        torch.cuda.synchronize()
    finally:
        sv.test_hooks(0, 0)
    assert int(st.item()) & sv.SV_DEV_TIMEOUT
    st.zero_()
    out = sv.spec_verify_attn(*args, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in a.items()}
    ref = oatt.verify_attention(cpu["q"], cpu["k_cache"], cpu["v_cache"], cpu["block_table"], cpu["seq_lens"],
                                1 / math.sqrt(cfg.d_head), cfg.block_size, cfg.kv_dtype, cpu["k_scale"],
                                cpu["v_scale"])
    assert np.abs(out.float().cpu().numpy() - ref).max() <= attn_tolerance(kv)


def test_sampling_wait_runs_out_then_next_call_is_correct(sv):
    cfg = workloads.CONFIGS["tiny"].with_(B=8, ctx=("fixed", (64,) * 8), V=20000, logit_dtype="bf16")
    s = {k: v.to(DEV) for k, v in workloads.make_sampling_inputs(cfg, seed=4).items()}
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    try:
        sv.test_hooks(2_000_000, sv.SV_TEST_WITHHOLD_ARRIVALS)
        # the float-float pass runs for every sequence when forced
        sv.spec_verify_sample(s["target_logits"], s["draft_logits"], s["draft_tokens"], s["uniforms"], status=st,
                              force_exact=True)
        torch.cuda.synchronize()
    finally:
        sv.test_hooks(0, 0)
    assert int(st.item()) & sv.SV_DEV_TIMEOUT
    st.zero_()
    tok, nac, p, q = sv.spec_verify_sample(s["target_logits"], s["draft_logits"], s["draft_tokens"], s["uniforms"],
                                           status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    cpu = {k: v.cpu() for k, v in s.items()}
    ref = osamp.rejection_sample(cpu["target_logits"], cpu["draft_logits"], cpu["draft_tokens"], cpu["uniforms"])
    compare_sampling(tok.cpu().numpy(), nac.cpu().numpy(), ref, p.cpu().numpy(), q.cpu().numpy())
