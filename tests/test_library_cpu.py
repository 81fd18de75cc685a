"""The C ABI without a GPU: the library builds, loads, exports every symbol the
header declares, sizes workspaces, and rejects bad arguments on the host
before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    import speculative_verify_paged_gb300 as sv
    sv.build()
    return sv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^(?:const\s+)?(?:sv_status|size_t|char|void|int|unsigned long long)\s*\*?\s*(\w+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_three_operations():
    names = declared_functions()
    for n in ("kv_block_append", "spec_verify_attn", "spec_verify_sample", "sv_last_error_string",
              "spec_verify_attn_workspace_size", "spec_verify_sample_workspace_size", "sv_kernel_launches"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_launch_counter_starts_without_gpu_work(lib):
    # host-side count; no kernel has run in this CPU-only process
    assert lib.sv_kernel_launches() == 0


def test_workspace_sizes(lib):
    # sampling: one 48-byte record per (sequence, position), one 16-byte
    # (max, sum) pair per 8192-logit chunk of each row (each part 256-byte
    # rounded), then the finish grid's fixed scratch (barrier words; per
    # re-evaluated row and CTA two float-float sums; per re-evaluated draw and
    # CTA a float-float total and an index), then one 8-byte entry per
    # sequence for the list of sequences left to the float-float pass
    up = lambda x: (x + 255) // 256 * 256
    chunks = (128256 + 8191) // 8192
    fin = 256 + 32 * 160 * 16 + 32 * 160 * (8 + 4)
    assert lib.spec_verify_sample_workspace_size(64, 4, 128256) == (
        up(64 * 5 * 48) + up(64 * 5 * chunks * 16) + fin + up(64 * 8))
    assert lib.spec_verify_sample_workspace_size(0, 4, 10) == fin
    s = lib.spec_verify_attn_workspace_size(64, 5, 64, 8, 128, 512, 16)
    # (acc d + m + l) floats per (sequence, kv head, split, row); splits of at
    # least 16 blocks
    assert s >= 64 * 8 * 1 * 40 * (128 + 2) * 4
    assert s <= 64 * 8 * (512 // 16) * 40 * (128 + 2) * 4 + 4096
    # an explicit split size: ceil(512 / 7) splits
    s7 = lib.spec_verify_attn_workspace_size_ex(64, 5, 64, 8, 128, 512, 16, 7)
    assert s7 >= 64 * 8 * 74 * 40 * (128 + 2) * 4
    assert lib.spec_verify_attn_workspace_size(1, 5, 6, 4, 128, 8, 16) == 0   # H_q % H_kv


def test_host_validation_errors(lib):
    import speculative_verify_paged_gb300 as sv
    NULL = None
    # kv_block_append: null pointers
    rc = lib.kv_block_append(NULL, NULL, 1, NULL, NULL, 1, None, NULL, NULL, NULL, 4, NULL,
                             2, 5, 2, 128, 16, 10, NULL, NULL)
    assert rc == 1
    assert b"null" in lib.sv_last_error_string()
    # attention: H_q not a multiple of H_kv (pointers are never dereferenced)
    fake = ctypes.c_void_p(0x1000)
    rc = lib.spec_verify_attn(fake, 1, fake, fake, 1, None, NULL, NULL, fake, 4, fake,
                              2, 5, 6, 4, 128, 16, 10, 0.1, fake, 1, fake, 1 << 30, NULL, NULL)
    assert rc == 1 and b"H_q" in lib.sv_last_error_string()
    # attention: workspace too small
    rc = lib.spec_verify_attn(fake, 1, fake, fake, 1, None, NULL, NULL, fake, 4, fake,
                              2, 5, 8, 2, 128, 16, 10, 0.1, fake, 1, fake, 16, NULL, NULL)
    assert rc == 3
    # attention: unsupported dtype pairing
    rc = lib.spec_verify_attn(fake, 0, fake, fake, 1, None, NULL, NULL, fake, 4, fake,
                              2, 5, 8, 2, 128, 16, 10, 0.1, fake, 0, fake, 1 << 30, NULL, NULL)
    assert rc == 2
    # sampling: bad temperature, bad sizes, draft dtype mismatch, small workspace
    args = lambda T, B, K, V, ddt, ws: (fake, 1, fake, ddt, 0, fake, fake, B, K, V, T, fake, fake,
                                        NULL, NULL, fake, ws, NULL, NULL)
    assert lib.spec_verify_sample(*args(0.0, 2, 4, 100, 1, 1 << 20)) == 1
    assert lib.spec_verify_sample(*args(1.0, 2, 4, 0, 1, 1 << 20)) == 1
    assert lib.spec_verify_sample(*args(1.0, 2, 4, 100, 0, 1 << 20)) == 2
    assert lib.spec_verify_sample(*args(1.0, 2, 4, 100, 1, 16)) == 3
    # a good call leaves the error string empty only after success; the
    # message of the last failure is kept
    assert len(lib.sv_last_error_string()) > 0
    assert sv.SpecVerifyError(3, "x").status == 3


def test_topp_host_validation_and_workspace(lib):
    fake = ctypes.c_void_p(0x1000)
    NULL = None
    # top_p outside (0, 1], bad sizes, fp8 logits, a vocabulary above 2^28
    assert lib.spec_topp_filter(fake, 1, 4, 100, 1.0, 0.0, fake, NULL, NULL) == 1
    assert lib.spec_topp_filter(fake, 1, 4, 100, 1.0, 1.5, fake, NULL, NULL) == 1
    assert lib.spec_topp_filter(fake, 1, -1, 100, 1.0, 0.5, fake, NULL, NULL) == 1
    assert lib.spec_topp_filter(fake, 1, 4, 100, 0.0, 0.5, fake, NULL, NULL) == 1
    assert lib.spec_topp_filter(fake, 3, 4, 100, 1.0, 0.5, fake, NULL, NULL) == 2
    assert lib.spec_topp_filter(fake, 1, 4, (1 << 28) + 1, 1.0, 0.5, fake, NULL, NULL) == 2
    # workspace: filtered target rows (and draft rows), 256-byte rounded, in
    # front of the sampling workspace
    up = lambda x: (x + 255) // 256 * 256
    base = lib.spec_verify_sample_workspace_size(64, 4, 128256)
    assert lib.spec_verify_sample_topp_workspace_size(64, 4, 128256, 1, 0) == up(64 * 5 * 128256 * 2) + base
    assert lib.spec_verify_sample_topp_workspace_size(64, 4, 128256, 1, 1) == (
        up(64 * 5 * 128256 * 2) + up(64 * 4 * 128256 * 2) + base)
    assert lib.spec_verify_sample_topp_workspace_size(64, 4, 128256, 3, 0) == 0
    # sampling with top-p: draft_topp with probabilities, bad top_p, small workspace
    args = lambda tp, dtp, probs, ddt, ws: (fake, 1, fake, ddt, probs, fake, fake, 2, 4, 100, 1.0, tp, dtp,
                                            fake, fake, NULL, NULL, fake, ws, NULL, NULL)
    assert lib.spec_verify_sample_topp(*args(0.9, 1, 1, 0, 1 << 30)) == 1
    assert lib.spec_verify_sample_topp(*args(0.0, 0, 0, 1, 1 << 30)) == 1
    assert lib.spec_verify_sample_topp(*args(0.9, 0, 0, 1, 16)) == 3
    assert lib.spec_verify_sample_topp(*args(0.9, 0, 0, 0, 1 << 30)) == 2   # draft dtype mismatch


def test_tree_attention_host_checks(lib):
    fake = ctypes.c_void_p(0x1000)
    NULL = None
    base = lib.spec_verify_attn_workspace_size(64, 5, 64, 8, 128, 512, 16)
    # the ancestor masks: 8 bytes per node, 256-byte rounded, after the usual workspace
    assert lib.spec_verify_attn_tree_workspace_size(64, 5, 64, 8, 128, 512, 16) == base + (64 * 5 * 8 + 255) // 256 * 256
    args = lambda tree, n_new: (fake, 1, fake, fake, 1, None, NULL, NULL, fake, 64, fake, tree,
                                2, n_new, 8, 2, 128, 16, 100, 0.1, fake, 1, fake, 1 << 30, NULL, NULL)
    assert lib.spec_verify_attn_tree(*args(NULL, 5)) == 1          # no parents
    assert lib.spec_verify_attn_tree(*args(fake, 65)) == 2         # more than 64 nodes


def test_tree_sampling_workspace_and_host_checks(lib):
    fake = ctypes.c_void_p(0x1000)
    NULL = None
    assert lib.spec_verify_sample_tree_workspace_size(64, 5) == (64 * 2 * 5 * 16 + 255) // 256 * 256
    args = lambda n, ws: (fake, 1, fake, 1, 0, fake, fake, fake, 2, n, 100, 1.0, NULL, fake, fake, fake, fake, ws,
                          NULL, NULL)
    assert lib.spec_verify_sample_tree(*args(5, 16)) == 3        # workspace too small
    assert lib.spec_verify_sample_tree(*args(65, 1 << 20)) == 2  # more than 64 nodes


def test_product_path_has_no_cpu_fallback():
    """The binding raises when tensors are not on a CUDA device."""
    import torch

    import speculative_verify_paged_gb300 as sv
    x = torch.zeros(2, 5, 8, 16)
    with pytest.raises((ValueError, RuntimeError)):
        sv.spec_verify_sample(torch.zeros(2, 5, 100), torch.zeros(2, 4, 100),
                              torch.zeros(2, 4, dtype=torch.int32), torch.zeros(2, 5, 2))
    with pytest.raises((ValueError, RuntimeError)):
        sv.spec_verify_attn(x, x, x, torch.zeros(2, 4, dtype=torch.int32), torch.zeros(2, dtype=torch.int32))


def test_mla_host_checks_and_workspace(lib):
    fake = ctypes.c_void_p(0x1000)
    NULL = None
    args = lambda B, n, H, dc, dr, bs, qdt, ws: (fake, qdt, fake, 1, fake, 64, fake, B, n, H, dc, dr, bs, 100, 0.07,
                                                 fake, fake, ws, NULL, NULL)
    assert lib.spec_verify_attn_mla(*args(2, 5, 128, 256, 64, 16, 1, 1 << 30)) == 2   # d_c other than 512
    assert lib.spec_verify_attn_mla(*args(2, 5, 128, 512, 64, 32, 1, 1 << 30)) == 2   # block size
    assert lib.spec_verify_attn_mla(*args(2, 5, 128, 512, 64, 16, 0, 1 << 30)) == 2   # f32 queries
    assert lib.spec_verify_attn_mla(*args(2, 0, 128, 512, 64, 16, 1, 1 << 30)) == 1   # n_new = 0
    assert lib.spec_verify_attn_mla(*args(1, 8, 16, 512, 64, 16, 1, 16)) == 3         # split context, small workspace
    assert lib.spec_verify_attn_mla(*args(2, 5, 128, 512, 64, 16, 1, 0)) == 3         # no room for the order
    assert lib.spec_verify_attn_mla(*args(0, 5, 128, 512, 64, 16, 1, 0)) == 0         # empty batch
    # splits only when the batch leaves the GPU short of work: partial outputs
    # of 512 floats and an (m, l) pair per row and split, 256-byte rounded,
    # then the longest-first order of the sequences (up to 4096 of them)
    up = lambda x: (x + 255) // 256 * 256
    assert lib.spec_verify_attn_mla_workspace_size(64, 5, 128, 512) == 256
    assert lib.spec_verify_attn_mla_workspace_size(5000, 5, 128, 512) == 0
    S = 24   # 376 blocks in splits of 16
    assert lib.spec_verify_attn_mla_workspace_size(1, 8, 16, 376) == up(S * 128 * 512 * 4) + up(S * 128 * 2 * 4) + 256
    assert lib.kv_block_append_latent(fake, 1, fake, fake, 4, fake, 2, 5, 512, 16, 10, NULL, NULL) == 2
    assert lib.kv_block_append_latent(fake, 0, fake, fake, 4, fake, 2, 5, 576, 16, 10, NULL, NULL) == 2
