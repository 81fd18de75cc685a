"""Pins for the fp8 e4m3 codec and the paged KV append oracle.

The e4m3 table is checked against values the OCP FP8 definition fixes
(largest finite 448, smallest subnormal 2^-9, NaN codes, monotone order),
against torch's float8_e4m3fn conversion (a library routine) inside the
finite range, and for round-to-nearest-even ties and saturation.
The append oracle is checked against the addressing of "KV Cache +
Speculative Decoding" section 6.2 (page pos // 16, slot pos % 16).
"""
import numpy as np
import pytest
import torch

from oracle import attention, fp8, kv_append


def test_code_table_fixed_points():
    v = fp8.code_values()
    assert v[0x00] == 0.0
    assert v[0x01] == 2.0 ** -9
    assert v[0x07] == 7 / 8 * 2.0 ** -6
    assert v[0x08] == 2.0 ** -6
    assert v[0x38] == 1.0
    assert v[0x7E] == 448.0
    assert v[0xFE] == -448.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.signbit(v[0x80]) and v[0x80] == 0.0
    assert np.isfinite(v).sum() == 254
    assert np.all(np.diff(v[:0x7F]) > 0)


def test_code_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    v = fp8.code_values()
    fin = np.isfinite(v)
    assert np.array_equal(v[fin], ref[fin])
    assert np.all(np.isnan(ref[~fin]))


def test_encode_roundtrip_all_finite_codes():
    v = fp8.code_values()
    fin = np.isfinite(v)
    codes = np.arange(256)[fin]
    assert np.array_equal(fp8.encode(v[fin].astype(np.float32)), codes.astype(np.uint8))


def test_encode_ties_to_even_and_saturation():
    assert fp8.encode(np.float32(1.0625)) == 0x38     # between 1.0 (0x38) and 1.125: even
    assert fp8.encode(np.float32(1.1875)) == 0x3A     # between 1.125 and 1.25: even 0x3A
    assert fp8.encode(np.float32(2.0 ** -10)) == 0x00   # half the smallest subnormal
    assert fp8.encode(np.float32(3 * 2.0 ** -10)) == 0x02
    assert fp8.encode(np.float32(-3 * 2.0 ** -10)) == 0x82
    assert fp8.encode(np.float32(500.0)) == 0x7E
    assert fp8.encode(np.float32(np.inf)) == 0x7E
    assert fp8.encode(np.float32(-np.inf)) == 0xFE
    assert fp8.encode(np.float32(np.nan)) == 0x7F
    assert fp8.encode(np.float32(464.0)) == 0x7E


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 100, 20000),
                        rng.normal(0, 1e-3, 20000)]).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode(x), ref)


def test_quantize_divides_in_fp32():
    x = np.float32(1.0)
    s = np.float32(3.0)
    assert fp8.quantize(x, s) == fp8.encode(np.float32(x / s))


@pytest.mark.parametrize("kv_dtype", ["f32", "bf16", "fp8_e4m3"])
def test_append_writes_positions_through_block_table(kv_dtype):
    import workloads
    cfg = workloads.CONFIGS["tiny"].with_(kv_dtype=kv_dtype,
                                          q_dtype="f32" if kv_dtype == "f32" else "bf16")
    inp = workloads.make_attention_inputs(cfg, seed=4)
    new = workloads.make_append_inputs(cfg, seed=4)
    kc, vc = kv_append.kv_block_append(inp["k_cache"], inp["v_cache"], new["k_new"], new["v_new"],
                                       inp["block_table"], inp["seq_lens"], 16, kv_dtype,
                                       inp["k_scale"], inp["v_scale"])
    touched = torch.zeros(kc.shape[:3], dtype=torch.bool)
    for b in range(cfg.B):
        L = int(inp["seq_lens"][b])
        for j in range(cfg.n_new):
            pos = L - cfg.n_new + j
            blk = int(inp["block_table"][b, pos // 16])
            for g in range(cfg.H_kv):
                touched[blk, g, pos % 16] = True
                for cache, src, sc in ((kc, new["k_new"], inp["k_scale"]), (vc, new["v_new"], inp["v_scale"])):
                    row = src[b, j, g].float()
                    if kv_dtype == "fp8_e4m3":
                        expect = torch.from_numpy(fp8.quantize(row.numpy(), np.float32(sc[g].item())))
                        assert torch.equal(cache[blk, g, pos % 16], expect)
                        # decoded value is within half an e4m3 step of x,
                        # or +-448 scale where x lies beyond (saturation)
                        dec = fp8.decode(expect.numpy()) * sc[g].item()
                        lim = 448.0 * np.float64(np.float32(sc[g].item()))
                        x = np.clip(row.double().numpy(), -lim, lim)
                        assert np.all(np.abs(dec - x) <= 0.0625 * np.abs(x) + 2 ** -10 * sc[g].item())
                        sat = np.abs(row.double().numpy()) > lim * (1 + 2 ** -4)
                        assert np.all(np.abs(np.abs(dec[sat]) - lim) <= 1e-12 * lim)
                    else:
                        assert torch.equal(cache[blk, g, pos % 16], row.to(cache.dtype))
    # nothing else changed
    assert torch.equal(kc[~touched], inp["k_cache"][~touched])
    assert torch.equal(vc[~touched], inp["v_cache"][~touched])
    # and the dense gather sees the new rows at the end of each sequence
    if kv_dtype != "fp8_e4m3":
        for b in range(cfg.B):
            L = int(inp["seq_lens"][b])
            Kd = attention.gather_dense(kc, inp["block_table"][b].numpy(), L, 16)
            assert np.array_equal(Kd[L - cfg.n_new:], new["k_new"][b].to(kc.dtype).double().numpy())


def test_bf16_rounding_known_values():
    x = torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -7], dtype=torch.float32)
    assert x.to(torch.bfloat16).float().tolist() == [1.0, 1 + 2 ** -6, 1 + 2 ** -7]
