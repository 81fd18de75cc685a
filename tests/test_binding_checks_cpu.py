"""Host-side argument checks of the Python binding (no GPU, no library call).

The latent (MLA) kernels index a pool [num_blocks, 16, d_c + d_r]; a pool of
any other shape, or index tensors that are not int32, must be rejected before
a pointer reaches the library (on a device they would send TMA boxes and
stores past the allocation). Each rejection is pinned with its own message.
"""
import pytest
import torch

import speculative_verify_paged_gb300 as sv

B, N_NEW, H, DC, DR, BS, NB = 2, 3, 4, 512, 64, 16, 10


def _mla_args(**over):
    a = dict(q_lat=torch.zeros(B, N_NEW, H, DC + DR, dtype=torch.bfloat16),
             cache=torch.zeros(NB, BS, DC + DR, dtype=torch.bfloat16),
             block_table=torch.zeros(B, 4, dtype=torch.int32),
             seq_lens=torch.full((B,), 20, dtype=torch.int32))
    a.update(over)
    return a


def _latent_args(**over):
    a = dict(c_new=torch.zeros(B, N_NEW, DC + DR, dtype=torch.bfloat16),
             cache=torch.zeros(NB, BS, DC + DR, dtype=torch.bfloat16),
             block_table=torch.zeros(B, 4, dtype=torch.int32),
             seq_lens=torch.full((B,), 20, dtype=torch.int32))
    a.update(over)
    return a


@pytest.mark.parametrize("over,msg", [
    (dict(cache=torch.zeros(NB, H, BS, DC + DR, dtype=torch.bfloat16)), "3|dims"),
    (dict(cache=torch.zeros(NB, 8, DC + DR, dtype=torch.bfloat16)), "slots per block"),
    (dict(cache=torch.zeros(NB, BS, DC, dtype=torch.bfloat16)), "rows hold"),
    (dict(block_table=torch.zeros(B, 4, dtype=torch.int64)), "block_table must be int32"),
    (dict(seq_lens=torch.full((B,), 20, dtype=torch.int64)), "seq_lens must be int32"),
    (dict(q_lat=torch.zeros(B, N_NEW, DC + DR, dtype=torch.bfloat16)), "q_lat must be"),
])
def test_mla_attention_rejects_bad_pools_and_index_types(over, msg):
    a = _mla_args(**over)
    with pytest.raises(ValueError, match=msg):
        sv.spec_verify_attn_mla(a["q_lat"], a["cache"], a["block_table"], a["seq_lens"], 0.07)


@pytest.mark.parametrize("over,msg", [
    (dict(cache=torch.zeros(NB, H, BS, DC + DR, dtype=torch.bfloat16)), "3|dims"),
    (dict(cache=torch.zeros(NB, 8, DC + DR, dtype=torch.bfloat16)), "slots per block"),
    (dict(cache=torch.zeros(NB, BS, DC + DR + 8, dtype=torch.bfloat16)), "rows hold"),
    (dict(block_table=torch.zeros(B, 4, dtype=torch.int64)), "block_table must be int32"),
    (dict(seq_lens=torch.full((B,), 20, dtype=torch.int16)), "seq_lens must be int32"),
    (dict(c_new=torch.zeros(B, N_NEW, 1, DC + DR, dtype=torch.bfloat16)), "c_new must be"),
])
def test_latent_append_rejects_bad_pools_and_index_types(over, msg):
    a = _latent_args(**over)
    with pytest.raises(ValueError, match=msg):
        sv.kv_block_append_latent(a["c_new"], a["cache"], a["block_table"], a["seq_lens"])


def test_index_tensors_of_the_other_entry_points_must_be_int32():
    f = torch.zeros(1, 2, 4, 64, dtype=torch.bfloat16)
    pool = torch.zeros(4, 4, 16, 64, dtype=torch.bfloat16)
    bt64 = torch.zeros(1, 2, dtype=torch.int64)
    lens = torch.full((1,), 8, dtype=torch.int32)
    with pytest.raises(ValueError, match="block_table must be int32"):
        sv.spec_verify_attn(f, pool, pool, bt64, lens)
    with pytest.raises(ValueError, match="block_table must be int32"):
        sv.kv_block_append(f, f, pool, pool, bt64, lens)
    logits = torch.zeros(1, 3, 50)
    with pytest.raises(ValueError, match="draft_tokens must be int32"):
        sv.spec_verify_sample(logits, logits[:, :2], torch.zeros(1, 2, dtype=torch.int64), torch.zeros(1, 3, 2))
