"""Seeded synthetic inputs for the speculative verify step.

This module is shared by the oracle-side tests and the CUDA-side tests and
benchmark. It only draws random numbers and lays them out; it contains none of
the verify step's arithmetic (no softmax, no attention, no fp8 rounding, no
inverse CDF).

Shapes follow the workloads the pages talk about: LLaMA-3-8B / 70B GQA layer
shapes (H_q/H_kv/d_head = 32/8/128 and 64/8/128, "KV Cache + Speculative
Decoding" section 2.2 and 4.2), 128K-token contexts (walkerchi "KV Cache" page,
section 3.1), a 128K vocabulary and K = 4..8 drafts.

Recipe (all draws come from torch generators seeded per field, so each field is
reproducible on its own and independent of which other fields are drawn):
  * seq_lens: fixed list or integers uniform in [lo, hi] (inclusive). A length
    counts every KV position of the sequence, including the K+1 new ones.
  * block table: every sequence gets ceil(L/16) physical blocks taken from a
    random permutation of the pool; the pool also holds `spare_blocks` unused
    blocks full of finite garbage. Unused table entries are -1.
  * K/V pools, Q, new K/V rows: N(0, 1), rounded to the storage dtype.
  * fp8 e4m3 pools: random codes drawn uniformly from the 254 finite e4m3
    bit patterns (both zeros, the subnormals of exponent field 0 and the
    largest magnitudes, +-448, included; the two NaN patterns S.1111.111
    excluded), with per-kv-head fp32 scales amax / 448 for amax uniform in
    [2, 6] (the largest code then stands for a magnitude of 2 to 6, like
    N(0, 1) data quantised with a per-head amax).
  * target logits ~ N(0, 3^2); draft logits = target + N(0, sigma^2).
  * draft tokens: x_i = argmax(draft_logits_i / T + Gumbel noise), which draws
    x_i from softmax(draft_logits_i / T) without evaluating that softmax.
  * uniforms: float32 in [0, 1), layout [B, K+1, 2] (u for the accept test,
    v for the residual / bonus draw).
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Optional

import torch

BLOCK_SIZE = 16


@dataclasses.dataclass(frozen=True)
class VerifyConfig:
    name: str
    B: int
    H_q: int
    H_kv: int
    d_head: int
    kv_dtype: str          # "f32" | "bf16" | "fp8_e4m3"
    q_dtype: str           # "f32" | "bf16" (also the attention output dtype)
    ctx: tuple             # ("fixed", (L_0, L_1, ...)) or ("uniform", (lo, hi))
    K: int
    V: int
    logit_dtype: str       # "f32" | "bf16"
    sigma: float           # draft noise
    block_size: int = BLOCK_SIZE
    spare_blocks: int = 3
    temperature: float = 1.0

    @property
    def n_new(self) -> int:
        return self.K + 1

    @property
    def group(self) -> int:
        return self.H_q // self.H_kv

    def with_(self, **kw) -> "VerifyConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": VerifyConfig("tiny", B=2, H_q=4, H_kv=2, d_head=64, kv_dtype="f32",
                         q_dtype="f32", ctx=("fixed", (40, 64)), K=4, V=1000,
                         logit_dtype="f32", sigma=1.0),
    "llama3_8b": VerifyConfig("llama3_8b", B=16, H_q=32, H_kv=8, d_head=128,
                              kv_dtype="bf16", q_dtype="bf16",
                              ctx=("fixed", (4096,) * 16), K=5, V=128256,
                              logit_dtype="bf16", sigma=1.5),
    "llama3_70b": VerifyConfig("llama3_70b", B=64, H_q=64, H_kv=8, d_head=128,
                               kv_dtype="bf16", q_dtype="bf16",
                               ctx=("uniform", (1024, 8192)), K=4, V=128256,
                               logit_dtype="bf16", sigma=1.5),
    "long": VerifyConfig("long", B=1, H_q=64, H_kv=8, d_head=128, kv_dtype="bf16",
                         q_dtype="bf16", ctx=("fixed", (131072,)), K=7, V=128256,
                         logit_dtype="bf16", sigma=1.0),
    "fp8": VerifyConfig("fp8", B=128, H_q=32, H_kv=8, d_head=128,
                        kv_dtype="fp8_e4m3", q_dtype="bf16",
                        ctx=("uniform", (256, 2048)), K=8, V=152064,
                        logit_dtype="f32", sigma=1.0),
}

# the 70B-shaped workload is also run with these draft-noise levels
SIGMA_SWEEP_70B = (0.5, 1.5, 3.0)

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8_e4m3": torch.uint8}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPE[name]


def elem_bytes(name: str) -> int:
    return {"f32": 4, "bf16": 2, "fp8_e4m3": 1}[name]


def _gen(seed: int, field: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + zlib.crc32(field.encode())) % (2 ** 62))
    return g


def _normal(shape, seed, field, device, std=1.0, dtype=torch.float32):
    g = _gen(seed, field, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def seq_lens_for(cfg: VerifyConfig, seed: int) -> list:
    kind, params = cfg.ctx
    if kind == "fixed":
        assert len(params) == cfg.B
        lens = list(params)
    else:
        lo, hi = params
        g = _gen(seed, "seq_lens", "cpu")
        lens = torch.randint(lo, hi + 1, (cfg.B,), generator=g).tolist()
    assert all(L >= cfg.n_new for L in lens)
    return lens


def paged_layout(cfg: VerifyConfig, seed: int, seq_lens: Optional[list] = None,
                 max_blocks_per_seq: Optional[int] = None):
    """Block table (int32, -1 for unused entries) and pool size."""
    if seq_lens is None:
        seq_lens = seq_lens_for(cfg, seed)
    bs = cfg.block_size
    nblk = [(L + bs - 1) // bs for L in seq_lens]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(nblk)
    num_blocks = sum(nblk) + cfg.spare_blocks
    g = _gen(seed, "block_perm", "cpu")
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    table = torch.full((cfg.B, max_blocks_per_seq), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[off:off + n]
        off += n
    return table, num_blocks, seq_lens


def _fp8_codes(shape, seed, field, device):
    """Random e4m3 bit patterns, uniform over the 254 finite codes: a draw k in
    [0, 254) is the code k for k < 127 (0x00 .. 0x7E) and k + 1 above
    (0x80 .. 0xFE), which skips the NaN patterns 0x7F and 0xFF."""
    g = _gen(seed, field, device)
    k = torch.randint(0, 254, shape, generator=g, device=device, dtype=torch.int32)
    return (k + (k >= 127).to(torch.int32)).to(torch.uint8)


def make_attention_inputs(cfg: VerifyConfig, seed: int = 0, device="cpu",
                          seq_lens: Optional[list] = None):
    """Q, paged K/V pools, block table and lengths for one verify step."""
    table, num_blocks, seq_lens = paged_layout(cfg, seed, seq_lens)
    shape = (num_blocks, cfg.H_kv, cfg.block_size, cfg.d_head)
    out = {"seq_lens": torch.tensor(seq_lens, dtype=torch.int32, device=device),
           "block_table": table.to(device), "num_blocks": num_blocks}
    if cfg.kv_dtype == "fp8_e4m3":
        out["k_cache"] = _fp8_codes(shape, seed, "k_pool", device)
        out["v_cache"] = _fp8_codes(shape, seed, "v_pool", device)
        gk, gv = _gen(seed, "k_scale", "cpu"), _gen(seed, "v_scale", "cpu")
        out["k_scale"] = ((2 + 4 * torch.rand(cfg.H_kv, generator=gk)) / 448).to(device)
        out["v_scale"] = ((2 + 4 * torch.rand(cfg.H_kv, generator=gv)) / 448).to(device)
    else:
        dt = torch_dtype(cfg.kv_dtype)
        out["k_cache"] = _normal(shape, seed, "k_pool", device, dtype=dt)
        out["v_cache"] = _normal(shape, seed, "v_pool", device, dtype=dt)
        out["k_scale"] = None
        out["v_scale"] = None
    out["q"] = _normal((cfg.B, cfg.n_new, cfg.H_q, cfg.d_head), seed, "q", device,
                       dtype=torch_dtype(cfg.q_dtype))
    return out


def make_append_inputs(cfg: VerifyConfig, seed: int = 0, device="cpu"):
    """New K/V rows [B, K+1, H_kv, d] for the positions L-K-1 .. L-1."""
    dt = torch_dtype(cfg.q_dtype)
    shape = (cfg.B, cfg.n_new, cfg.H_kv, cfg.d_head)
    return {"k_new": _normal(shape, seed, "k_new", device, dtype=dt),
            "v_new": _normal(shape, seed, "v_new", device, dtype=dt)}


def make_sampling_inputs(cfg: VerifyConfig, seed: int = 0, device="cpu",
                         sigma: Optional[float] = None):
    """Target/draft logits, draft tokens and per-position uniforms."""
    sigma = cfg.sigma if sigma is None else sigma
    dt = torch_dtype(cfg.logit_dtype)
    B, K, V = cfg.B, cfg.K, cfg.V
    tgt32 = _normal((B, K + 1, V), seed, "target_logits", device, std=3.0)
    drf32 = tgt32[:, :K, :] + _normal((B, K, V), seed, "draft_noise", device, std=sigma)
    target = tgt32.to(dt)
    draft = drf32.to(dt)
    del tgt32, drf32
    # Gumbel-max draw of the draft tokens from softmax(draft / T)
    g = _gen(seed, "draft_gumbel", device)
    tokens = torch.empty((B, K), dtype=torch.int32, device=device)
    for i in range(K):
        u = torch.rand((B, V), generator=g, device=device, dtype=torch.float64)
        u.clamp_(min=1e-300)
        gumbel = -torch.log(-torch.log(u))
        score = draft[:, i, :].double() / cfg.temperature + gumbel
        tokens[:, i] = score.argmax(dim=1).to(torch.int32)
        del u, gumbel, score
    gu = _gen(seed, "uniforms", device)
    uniforms = torch.rand((B, K + 1, 2), generator=gu, device=device, dtype=torch.float32)
    return {"target_logits": target, "draft_logits": draft,
            "draft_tokens": tokens, "uniforms": uniforms}


def attention_bytes(cfg: VerifyConfig, seq_lens) -> int:
    """Algorithmic bytes of one attention launch: each KV byte once (plus the
    per-head fp8 scales), Q, O, the block table entries used and the lengths."""
    kv = 2 * sum(seq_lens) * cfg.H_kv * cfg.d_head * elem_bytes(cfg.kv_dtype)
    qo = 2 * cfg.B * cfg.n_new * cfg.H_q * cfg.d_head * elem_bytes(cfg.q_dtype)
    nblk = sum((L + cfg.block_size - 1) // cfg.block_size for L in seq_lens)
    extra = 4 * nblk + 4 * cfg.B
    if cfg.kv_dtype == "fp8_e4m3":
        extra += 2 * 4 * cfg.H_kv
    return kv + qo + extra


def sampling_bytes(cfg: VerifyConfig) -> int:
    """Algorithmic bytes of one sampling launch: every target and draft logit
    once, draft tokens, uniforms and the outputs."""
    lb = elem_bytes(cfg.logit_dtype)
    logits = cfg.B * ((cfg.K + 1) + cfg.K) * cfg.V * lb
    small = cfg.B * cfg.K * 4 + cfg.B * (cfg.K + 1) * 2 * 4 + cfg.B * (cfg.K + 1) * 4 + cfg.B * 4
    return logits + small


def append_bytes(cfg: VerifyConfig) -> int:
    n = cfg.B * cfg.n_new * cfg.H_kv * cfg.d_head
    return 2 * n * (elem_bytes(cfg.q_dtype) + elem_bytes(cfg.kv_dtype))
