"""The seeded input generator: shapes, determinism, block-table validity."""
import torch

import workloads


def test_tiny_shapes_and_block_table():
    cfg = workloads.CONFIGS["tiny"]
    a = workloads.make_attention_inputs(cfg, seed=0)
    assert a["q"].shape == (2, 5, 4, 64) and a["q"].dtype == torch.float32
    assert a["seq_lens"].tolist() == [40, 64]
    t = a["block_table"]
    used = torch.cat([t[0, :3], t[1, :4]])
    assert (t[0, 3:] == -1).all()
    assert len(set(used.tolist())) == 7                 # distinct physical blocks
    assert a["num_blocks"] == 7 + cfg.spare_blocks
    assert int(used.max()) < a["num_blocks"]


def test_determinism_and_field_independence():
    cfg = workloads.CONFIGS["tiny"]
    a1 = workloads.make_attention_inputs(cfg, seed=3)
    a2 = workloads.make_attention_inputs(cfg, seed=3)
    for k in ("q", "k_cache", "v_cache", "block_table"):
        assert torch.equal(a1[k], a2[k])
    s1 = workloads.make_sampling_inputs(cfg, seed=3)
    s2 = workloads.make_sampling_inputs(cfg, seed=3)
    for k in s1:
        assert torch.equal(s1[k], s2[k])
    assert not torch.equal(workloads.make_attention_inputs(cfg, seed=4)["q"], a1["q"])


def test_uniform_lengths_in_range():
    cfg = workloads.CONFIGS["llama3_70b"]
    lens = workloads.seq_lens_for(cfg, 0)
    assert len(lens) == 64 and min(lens) >= 1024 and max(lens) <= 8192


def test_fp8_codes_never_nan():
    cfg = workloads.CONFIGS["tiny"].with_(kv_dtype="fp8_e4m3", q_dtype="bf16")
    a = workloads.make_attention_inputs(cfg, seed=0)
    assert a["k_cache"].dtype == torch.uint8
    assert not ((a["k_cache"] & 0x7F) == 0x7F).any()
    assert (a["k_scale"] > 0).all()


def test_fp8_codes_cover_every_finite_code():
    # the generator draws all 254 finite e4m3 patterns: zeros, subnormals
    # (exponent field 0) and the largest magnitudes (0x7E = 448, 0xFE = -448)
    codes = workloads._fp8_codes((200000,), 0, "k_pool", "cpu")
    seen = torch.bincount(codes.to(torch.int64), minlength=256)
    finite = [c for c in range(256) if c & 0x7F != 0x7F]
    assert all(int(seen[c]) > 0 for c in finite)
    assert int(seen[0x7F]) == 0 and int(seen[0xFF]) == 0
    # roughly uniform: 200000 / 254 ~ 787 per code
    assert int(seen[finite].min()) > 600 and int(seen[finite].max()) < 1000


def test_draft_tokens_in_range_and_mostly_likely_tokens():
    cfg = workloads.CONFIGS["tiny"]
    s = workloads.make_sampling_inputs(cfg, seed=0)
    x = s["draft_tokens"]
    assert x.shape == (2, 4) and int(x.min()) >= 0 and int(x.max()) < cfg.V
    assert s["uniforms"].shape == (2, 5, 2)
    assert float(s["uniforms"].min()) >= 0 and float(s["uniforms"].max()) < 1


def test_byte_model_matches_kv_formula():
    from oracle import theory
    cfg = workloads.CONFIGS["llama3_8b"]
    lens = workloads.seq_lens_for(cfg, 0)
    kv = 2 * sum(lens) * cfg.H_kv * cfg.d_head * 2
    # per-layer KV bytes of the batch = the pages' formula with N_layers = 1
    assert kv == theory.kv_cache_bytes(4096, 1, 8, 128, 2, batch=16)
    assert workloads.attention_bytes(cfg, lens) > kv
