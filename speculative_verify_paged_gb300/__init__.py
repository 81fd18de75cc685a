"""Python binding of libspecverify (ctypes): argument marshalling only.

Every operation runs in the library's CUDA kernels; this module checks that
tensors are CUDA, contiguous and of the expected dtype, passes their device
pointers and the current torch stream, allocates outputs / workspaces with
torch when the caller gives none, and raises on a non-zero status. There is no
CPU fallback: if the library is missing or CUDA is unavailable, calls raise.

Entry points (names follow the C ABI in include/specverify.h):
  kv_block_append     paged write of the K+1 new K/V rows
  spec_verify_attn    paged GQA verify attention over the K+1 queries
  spec_verify_sample  fused rejection sampling (accept / residual / bonus)
  verify_step         the three in stream order (one verify round of one layer)
  tree_verify_step    the same for a draft tree, with the commit of the accepted path
  MultiLayerVerify    a round over many layers' pools, runnable as one CUDA graph
  spec_verify_attn_mla, kv_block_append_latent
                      the same verify attention for a latent (MLA) cache
  BlockManager        host block manager of the paged pool (sv_bm_*)
  copy_blocks         device page copies for copy-on-write (sv_copy_blocks)
"""
import ctypes
import math
import os

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SV_F32, SV_BF16, SV_F16, SV_FP8_E4M3 = 0, 1, 2, 3
SV_SAMPLE_FORCE_EXACT = 1
DEV_STATUS_BITS = {1: "BAD_SEQ_LEN", 2: "BAD_BLOCK", 4: "BAD_TOKEN", 8: "TIMEOUT", 16: "NONFINITE",
                   32: "BAD_TREE", 64: "BAD_WORK"}
_STATUS = {0: "SV_OK", 1: "SV_ERR_INVALID_ARG", 2: "SV_ERR_UNSUPPORTED", 3: "SV_ERR_WORKSPACE",
           4: "SV_ERR_CUDA", 5: "SV_ERR_TIMEOUT", 6: "SV_ERR_OUT_OF_BLOCKS"}
SV_ERR_OUT_OF_BLOCKS = 6

_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s: %s" % (_STATUS.get(status, status), msg))
        self.status = status


class OutOfBlocks(SpecVerifyError):
    """The block manager's pool has too few free pages for the call."""


class _Typical(ctypes.Structure):
    _fields_ = [("epsilon", ctypes.c_float), ("delta", ctypes.c_float)]


class _Layout(ctypes.Structure):
    _fields_ = [("block_stride", ctypes.c_int64), ("head_stride", ctypes.c_int64),
                ("slot_stride", ctypes.c_int64)]


def load_library(path: str = LIB_PATH):
    """Load (not build) the shared library and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libspecverify.so is not built (%s): call "
                           "speculative_verify_paged_gb300.build.build() first" % path)
    lib = ctypes.CDLL(path)
    P, I, Z, F, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_uint
    LP = ctypes.POINTER(_Layout)
    lib.sv_last_error_string.restype = ctypes.c_char_p
    lib.sv_last_error_string.argtypes = []
    lib.sv_kernel_launches.restype = ctypes.c_ulonglong
    lib.sv_kernel_launches.argtypes = []
    lib.sv_test_hooks.restype = None
    lib.sv_test_hooks.argtypes = [ctypes.c_ulonglong, ctypes.c_uint]
    lib.kv_block_append.restype = I
    lib.kv_block_append.argtypes = [P, P, I, P, P, I, LP, P, P, P, I, P, I, I, I, I, I, I, P, P]
    lib.spec_verify_attn_workspace_size.restype = Z
    lib.spec_verify_attn_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.spec_verify_attn_workspace_size_ex.restype = Z
    lib.spec_verify_attn_workspace_size_ex.argtypes = [I, I, I, I, I, I, I, I]
    attn_args = [P, I, P, P, I, LP, P, P, P, I, P, I, I, I, I, I, I, I, F, P, I, P, Z, P]
    lib.spec_verify_attn.restype = I
    lib.spec_verify_attn.argtypes = attn_args + [P]
    lib.spec_verify_attn_ex.restype = I
    lib.spec_verify_attn_ex.argtypes = attn_args + [I, P]
    lib.spec_verify_attn_tree_workspace_size.restype = Z
    lib.spec_verify_attn_tree_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.spec_verify_attn_tree.restype = I
    lib.spec_verify_attn_tree.argtypes = attn_args[:11] + [P] + attn_args[11:] + [P]
    lib.spec_verify_sample_workspace_size.restype = Z
    lib.spec_verify_sample_workspace_size.argtypes = [I, I, I]
    samp_args = [P, I, P, I, I, P, P, I, I, I, F, P, P, P, P, P, Z, P]
    lib.spec_verify_sample.restype = I
    lib.spec_verify_sample.argtypes = samp_args + [P]
    lib.spec_verify_sample_ex.restype = I
    lib.spec_verify_sample_ex.argtypes = samp_args + [U, P]
    lib.spec_topp_filter.restype = I
    lib.spec_topp_filter.argtypes = [P, I, I, I, F, F, P, P, P]
    lib.spec_verify_sample_topp_workspace_size.restype = Z
    lib.spec_verify_sample_topp_workspace_size.argtypes = [I, I, I, I, I]
    lib.spec_verify_sample_topp.restype = I
    lib.spec_verify_sample_topp.argtypes = [P, I, P, I, I, P, P, I, I, I, F, F, I, P, P, P, P, P, Z, P, P]
    lib.kv_tree_commit.restype = I
    lib.kv_tree_commit.argtypes = [P, P, I, LP, P, I, P, P, P, I, I, I, I, I, I, P, P]
    lib.spec_verify_sample_tree_workspace_size.restype = Z
    lib.spec_verify_sample_tree_workspace_size.argtypes = [I, I]
    lib.spec_verify_sample_tree.restype = I
    lib.spec_verify_sample_tree.argtypes = [P, I, P, I, I, P, P, P, I, I, I, F, P, P, P, P, P, Z, P, P]
    I64, BMP = ctypes.c_int64, ctypes.c_void_p
    lib.sv_bm_create.restype = I
    lib.sv_bm_create.argtypes = [I, I, ctypes.POINTER(ctypes.c_void_p)]
    lib.sv_bm_destroy.restype = None
    lib.sv_bm_destroy.argtypes = [BMP]
    lib.sv_bm_num_free.restype = I
    lib.sv_bm_num_free.argtypes = [BMP]
    lib.sv_bm_ref_count.restype = I
    lib.sv_bm_ref_count.argtypes = [BMP, I]
    lib.sv_bm_free_list.restype = I
    lib.sv_bm_free_list.argtypes = [BMP, P, I, ctypes.POINTER(I)]
    lib.sv_bm_allocate.restype = I
    lib.sv_bm_allocate.argtypes = [BMP, I64, I64]
    lib.sv_bm_free.restype = I
    lib.sv_bm_free.argtypes = [BMP, I64]
    lib.sv_bm_fork.restype = I
    lib.sv_bm_fork.argtypes = [BMP, I64, I64]
    lib.sv_bm_share_prefix.restype = I
    lib.sv_bm_share_prefix.argtypes = [BMP, I64, I64, I64]
    lib.sv_bm_extend.restype = I
    lib.sv_bm_extend.argtypes = [BMP, P, I, I, P, P, I, ctypes.POINTER(I)]
    lib.sv_bm_truncate.restype = I
    lib.sv_bm_truncate.argtypes = [BMP, I64, I64]
    lib.sv_bm_commit_verify.restype = I
    lib.sv_bm_commit_verify.argtypes = [BMP, P, I, I, P]
    lib.sv_bm_seq_len.restype = I
    lib.sv_bm_seq_len.argtypes = [BMP, I64, ctypes.POINTER(I64)]
    lib.sv_bm_block_table.restype = I
    lib.sv_bm_block_table.argtypes = [BMP, P, I, I, P, P]
    lib.sv_copy_blocks.restype = I
    lib.sv_copy_blocks.argtypes = [P, I, I64, I64, P, P, I, I, P, P]
    lib.kv_block_append_latent.restype = I
    lib.kv_block_append_latent.argtypes = [P, I, P, P, I, P, I, I, I, I, I, P, P]
    lib.spec_verify_attn_mla_workspace_size.restype = Z
    lib.spec_verify_attn_mla_workspace_size.argtypes = [I, I, I, I]
    lib.spec_verify_attn_mla.restype = I
    lib.spec_verify_attn_mla.argtypes = [P, I, P, I, P, I, P, I, I, I, I, I, I, I, F, P, P, Z, P, P]
    _lib = lib
    return lib


def _check(rc):
    if rc != 0:
        cls = OutOfBlocks if rc == SV_ERR_OUT_OF_BLOCKS else SpecVerifyError
        raise cls(rc, load_library().sv_last_error_string().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dtype_code(t: torch.Tensor, fp8: bool = False) -> int:
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float16:
        return SV_F16
    if t.dtype == torch.uint8 or t.dtype == getattr(torch, "float8_e4m3fn", None):
        return SV_FP8_E4M3
    raise TypeError("unsupported dtype %s" % t.dtype)


def _cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensor arguments must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensor arguments must be contiguous")


def _int32(**ts):
    for name, t in ts.items():
        if t is not None and t.dtype != torch.int32:
            raise ValueError("%s must be int32, not %s" % (name, t.dtype))


def _check_latent_pool(cache, d_total, block_size, what):
    """The latent kernels index a pool [num_blocks, block_size, d_total] (d_total =
    d_c + d_r values per token, no head axis); any other shape would send their
    TMA boxes and stores past the allocation."""
    if cache.dim() != 3:
        raise ValueError("%s: the latent pool must be [num_blocks, block_size, d_c + d_r], got %d dims"
                         % (what, cache.dim()))
    if cache.shape[1] != block_size:
        raise ValueError("%s: the latent pool holds %d slots per block, block_size is %d"
                         % (what, cache.shape[1], block_size))
    if cache.shape[2] != d_total:
        raise ValueError("%s: the latent pool rows hold %d values, the queries / new rows %d"
                         % (what, cache.shape[2], d_total))


def _layout_arg(layout):
    if layout is None:
        return None
    return ctypes.byref(_Layout(*[int(x) for x in layout]))


# --------------------------------------------------------------- append ---

def kv_block_append(k_new, v_new, k_cache, v_cache, block_table, seq_lens, k_scale=None,
                    v_scale=None, block_size=16, layout=None, status=None):
    """Write k_new/v_new [B, n_new, H_kv, d] at positions seq_lens-n_new .. seq_lens-1."""
    _int32(block_table=block_table, seq_lens=seq_lens)
    lib = load_library()
    _cuda(k_new, v_new, k_cache, v_cache, block_table, seq_lens, k_scale, v_scale, status)
    B, n_new, H_kv, d = k_new.shape
    num_blocks = k_cache.shape[0]
    _check(lib.kv_block_append(_ptr(k_new), _ptr(v_new), _dtype_code(k_new), _ptr(k_cache),
                               _ptr(v_cache), _dtype_code(k_cache), _layout_arg(layout),
                               _ptr(k_scale), _ptr(v_scale), _ptr(block_table),
                               block_table.shape[1], _ptr(seq_lens), B, n_new, H_kv, d, block_size,
                               num_blocks, _ptr(status), _stream()))


def kv_tree_commit(k_cache, v_cache, block_table, seq_lens, path_nodes, num_accepted, block_size=16,
                   layout=None, num_blocks=None, H_kv=None, status=None):
    """Move each sequence's accepted tree path (path_nodes [B, n_new], num_accepted [B])
    next to the root in the paged pools; pools [num_blocks, H_kv, bs, d] unless layout."""
    _int32(block_table=block_table, seq_lens=seq_lens, path_nodes=path_nodes, num_accepted=num_accepted)
    lib = load_library()
    _cuda(k_cache, v_cache, block_table, seq_lens, path_nodes, num_accepted, status)
    B, n_new = path_nodes.shape
    if layout is None:
        num_blocks, H_kv, d = k_cache.shape[0], k_cache.shape[1], k_cache.shape[3]
    else:
        if num_blocks is None or H_kv is None:
            raise ValueError("with an explicit layout pass num_blocks and H_kv")
        d = k_cache.shape[-1]
    _check(lib.kv_tree_commit(_ptr(k_cache), _ptr(v_cache), _dtype_code(k_cache, True), _layout_arg(layout),
                              _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(path_nodes),
                              _ptr(num_accepted), B, n_new, H_kv, d, block_size, num_blocks, _ptr(status),
                              _stream()))


# ------------------------------------------------------------ attention ---

def attn_workspace_size(B, n_new, H_q, H_kv, d_head, max_blocks_per_seq, block_size=16,
                        blocks_per_split=None):
    lib = load_library()
    if blocks_per_split is None:
        return lib.spec_verify_attn_workspace_size(B, n_new, H_q, H_kv, d_head, max_blocks_per_seq,
                                                   block_size)
    return lib.spec_verify_attn_workspace_size_ex(B, n_new, H_q, H_kv, d_head, max_blocks_per_seq,
                                                  block_size, blocks_per_split)


def alloc_workspace(nbytes, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def spec_verify_attn(q, k_cache, v_cache, block_table, seq_lens, softmax_scale=None, k_scale=None,
                     v_scale=None, block_size=16, out=None, workspace=None, status=None,
                     blocks_per_split=None, layout=None, num_blocks=None, H_kv=None, tree_parent=None):
    """Paged GQA verify attention. q [B, n_new, H_q, d]; caches [num_blocks, H_kv, bs, d],
    or, with `layout` = (block, head, slot) strides in elements, flat views whose first
    element is (block 0, head 0, slot 0) plus explicit num_blocks and H_kv.
    tree_parent (int32 [B, n_new], optional): the new positions are a draft tree in BFS
    order and each query sees only its ancestors among them."""
    _int32(block_table=block_table, seq_lens=seq_lens, tree_parent=tree_parent)
    lib = load_library()
    _cuda(q, k_cache, v_cache, block_table, seq_lens, k_scale, v_scale, out, workspace, status,
          tree_parent)
    B, n_new, H_q, d = q.shape
    if layout is None:
        num_blocks_, H_kv = k_cache.shape[0], k_cache.shape[1]
    else:
        if H_kv is None or num_blocks is None:
            raise ValueError("with an explicit layout pass num_blocks and H_kv")
        num_blocks_ = num_blocks
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    max_blocks = block_table.shape[1]
    if tree_parent is not None:
        if blocks_per_split is not None:
            raise ValueError("blocks_per_split is not available with tree_parent")
        need = lib.spec_verify_attn_tree_workspace_size(B, n_new, H_q, H_kv, d, max_blocks, block_size)
    else:
        need = attn_workspace_size(B, n_new, H_q, H_kv, d, max_blocks, block_size, blocks_per_split)
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    args = [_ptr(q), _dtype_code(q), _ptr(k_cache), _ptr(v_cache), _dtype_code(k_cache, True),
            _layout_arg(layout), _ptr(k_scale), _ptr(v_scale), _ptr(block_table), max_blocks,
            _ptr(seq_lens), B, n_new, H_q, H_kv, d, block_size, num_blocks_, float(softmax_scale),
            _ptr(out), _dtype_code(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _ptr(status)]
    if tree_parent is not None:
        _check(lib.spec_verify_attn_tree(*args[:11], _ptr(tree_parent), *args[11:], _stream()))
    elif blocks_per_split is None:
        _check(lib.spec_verify_attn(*args, _stream()))
    else:
        _check(lib.spec_verify_attn_ex(*args, int(blocks_per_split), _stream()))
    return out


# ------------------------------------------------------------------ MLA ---

def kv_block_append_latent(c_new, cache, block_table, seq_lens, block_size=16, status=None):
    """Write latent rows c_new [B, n_new, d_c + d_r] (bf16) at positions
    seq_lens - n_new .. seq_lens - 1 of the pool cache [num_blocks, bs, d_c + d_r]."""
    if c_new.dim() != 3:
        raise ValueError("kv_block_append_latent: c_new must be [B, n_new, d_c + d_r]")
    _check_latent_pool(cache, c_new.shape[-1], block_size, "kv_block_append_latent")
    _int32(block_table=block_table, seq_lens=seq_lens)
    if cache.dtype != c_new.dtype:
        raise ValueError("the latent pool and the new rows must have the same dtype (bf16)")
    lib = load_library()
    _cuda(c_new, cache, block_table, seq_lens, status)
    B, n_new, D = c_new.shape
    _check(lib.kv_block_append_latent(_ptr(c_new), _dtype_code(c_new), _ptr(cache), _ptr(block_table),
                                      block_table.shape[1], _ptr(seq_lens), B, n_new, D, block_size,
                                      cache.shape[0], _ptr(status), _stream()))


def mla_workspace_size(B, n_new, H, max_blocks_per_seq):
    return load_library().spec_verify_attn_mla_workspace_size(B, n_new, H, max_blocks_per_seq)


def spec_verify_attn_mla(q_lat, cache, block_table, seq_lens, softmax_scale, d_c=512, block_size=16, out=None,
                         workspace=None, status=None):
    """Absorbed MLA verify attention: q_lat [B, n_new, H, d_c + d_r] bf16 against
    the latent pool cache [num_blocks, bs, d_c + d_r] bf16; returns the latent
    outputs [B, n_new, H, d_c] (bf16), to be multiplied by each head's W_UV."""
    if q_lat.dim() != 4:
        raise ValueError("spec_verify_attn_mla: q_lat must be [B, n_new, H, d_c + d_r]")
    _check_latent_pool(cache, q_lat.shape[-1], block_size, "spec_verify_attn_mla")
    _int32(block_table=block_table, seq_lens=seq_lens)
    if out is not None and (out.dtype != q_lat.dtype or out.shape != q_lat.shape[:3] + (d_c,)):
        raise ValueError("out must be [B, n_new, H, d_c] in the queries' dtype")
    lib = load_library()
    _cuda(q_lat, cache, block_table, seq_lens, out, workspace, status)
    B, n_new, H, D = q_lat.shape
    if out is None:
        out = torch.empty((B, n_new, H, d_c), dtype=q_lat.dtype, device=q_lat.device)
    max_blocks = block_table.shape[1]
    if workspace is None:
        workspace = alloc_workspace(mla_workspace_size(B, n_new, H, max_blocks), q_lat.device)
    _check(lib.spec_verify_attn_mla(_ptr(q_lat), _dtype_code(q_lat), _ptr(cache), _dtype_code(cache),
                                    _ptr(block_table), max_blocks, _ptr(seq_lens), B, n_new, H, d_c, D - d_c,
                                    block_size, cache.shape[0], float(softmax_scale), _ptr(out), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _ptr(status), _stream()))
    return out


# ------------------------------------------------------------- sampling ---

SV_TEST_WITHHOLD_COPIES, SV_TEST_WITHHOLD_ARRIVALS = 1, 2
SV_DEV_TIMEOUT = 8


def test_hooks(wait_limit_ns=0, withhold=0):
    """Wait limit of later launches' device waits (0: the default second) and
    the signals they withhold (SV_TEST_WITHHOLD_*), for tests of the bounded
    waits."""
    load_library().sv_test_hooks(int(wait_limit_ns), int(withhold))


def kernel_launches():
    """Kernels the library has launched in this process (host-side count)."""
    return int(load_library().sv_kernel_launches())


def sample_workspace_size(B, K, V):
    return load_library().spec_verify_sample_workspace_size(B, K, V)


def topp_filter(logits, top_p, temperature=1.0, out=None, status=None):
    """Rows of `logits` [..., V] with -inf outside each row's top-p set."""
    lib = load_library()
    _cuda(logits, out, status)
    if out is None:
        out = torch.empty_like(logits)
    V = logits.shape[-1]
    rows = logits.numel() // V
    _check(lib.spec_topp_filter(_ptr(logits), _dtype_code(logits), rows, V, float(temperature),
                                float(top_p), _ptr(out), _ptr(status), _stream()))
    return out


def spec_verify_sample(target_logits, draft, draft_tokens, uniforms, draft_is_probs=False,
                       temperature=1.0, out_tokens=None, num_accepted=None, p_at_draft=None,
                       q_at_draft=None, workspace=None, status=None, force_exact=False,
                       want_probs=True, top_p=None, draft_top_p=False):
    """Rejection sampling of one verify round.

    target_logits [B, K+1, V]; draft [B, K, V] logits (same dtype) or f32
    probabilities; draft_tokens int32 [B, K]; uniforms f32 [B, K+1, 2].
    top_p (optional): sample from the top-p truncated target rows (and draft
    logit rows too with draft_top_p).
    Returns (out_tokens [B, K+1], num_accepted [B], p_at_draft, q_at_draft).
    """
    _int32(draft_tokens=draft_tokens, out_tokens=out_tokens, num_accepted=num_accepted)
    lib = load_library()
    _cuda(target_logits, draft, draft_tokens, uniforms, out_tokens, num_accepted, p_at_draft,
          q_at_draft, workspace, status)
    B, K1, V = target_logits.shape
    K = K1 - 1
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if want_probs and p_at_draft is None:
        p_at_draft = torch.empty((B, K), dtype=torch.float32, device=dev)
    if want_probs and q_at_draft is None:
        q_at_draft = torch.empty((B, K), dtype=torch.float32, device=dev)
    ddt = _dtype_code(draft) if draft is not None else SV_F32
    if top_p is not None:
        if force_exact:
            raise ValueError("force_exact is not available with top_p")
        ldt = _dtype_code(target_logits)
        need = lib.spec_verify_sample_topp_workspace_size(B, K, V, ldt, int(bool(draft_top_p)))
        if workspace is None:
            workspace = alloc_workspace(need, dev)
        _check(lib.spec_verify_sample_topp(
            _ptr(target_logits), ldt, _ptr(draft), ddt, int(bool(draft_is_probs)), _ptr(draft_tokens),
            _ptr(uniforms), B, K, V, float(temperature), float(top_p), int(bool(draft_top_p)),
            _ptr(out_tokens), _ptr(num_accepted), _ptr(p_at_draft), _ptr(q_at_draft), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(status), _stream()))
        return out_tokens, num_accepted, p_at_draft, q_at_draft
    if workspace is None:
        workspace = alloc_workspace(sample_workspace_size(B, K, V), dev)
    args = [_ptr(target_logits), _dtype_code(target_logits), _ptr(draft), ddt, int(bool(draft_is_probs)),
            _ptr(draft_tokens), _ptr(uniforms), B, K, V, float(temperature), _ptr(out_tokens),
            _ptr(num_accepted), _ptr(p_at_draft), _ptr(q_at_draft), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(status)]
    if force_exact:
        _check(lib.spec_verify_sample_ex(*args, SV_SAMPLE_FORCE_EXACT, _stream()))
    else:
        _check(lib.spec_verify_sample(*args, _stream()))
    return out_tokens, num_accepted, p_at_draft, q_at_draft


def spec_verify_sample_tree(target_logits, draft, tree_parent, tree_tokens, uniforms, draft_is_probs=False,
                            temperature=1.0, out_tokens=None, num_accepted=None, path_nodes=None, status=None,
                            workspace=None, typical=None):
    """Rejection sampling over a draft tree of n nodes (BFS order, node 0 the root).

    typical=(epsilon, delta) switches to typical acceptance (not exact; draft unused).

    target_logits [B, n, V]; draft [B, n, V] logits (same dtype) or f32 probabilities;
    tree_parent, tree_tokens int32 [B, n]; uniforms f32 [B, n, 2].
    Returns (out_tokens [B, n], num_accepted [B], path_nodes [B, n]).
    """
    lib = load_library()
    _cuda(target_logits, draft, tree_parent, tree_tokens, uniforms, out_tokens, num_accepted, path_nodes,
          status, workspace)
    B, n, V = target_logits.shape
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, n), dtype=torch.int32, device=dev)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if path_nodes is None:
        path_nodes = torch.empty((B, n), dtype=torch.int32, device=dev)
    ddt = _dtype_code(draft) if draft is not None else SV_F32
    if workspace is None:
        workspace = alloc_workspace(lib.spec_verify_sample_tree_workspace_size(B, n), dev)
    _check(lib.spec_verify_sample_tree(_ptr(target_logits), _dtype_code(target_logits), _ptr(draft), ddt,
                                       int(bool(draft_is_probs)), _ptr(tree_parent), _ptr(tree_tokens),
                                       _ptr(uniforms), B, n, V, float(temperature),
                                       None if typical is None else ctypes.byref(_Typical(*typical)),
                                       _ptr(out_tokens),
                                       _ptr(num_accepted), _ptr(path_nodes), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _ptr(status), _stream()))
    return out_tokens, num_accepted, path_nodes


# ----------------------------------------------------------- verify step ---

def verify_step(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, target_logits, draft,
                draft_tokens, uniforms, k_scale=None, v_scale=None, draft_is_probs=False,
                temperature=1.0, softmax_scale=None, attn_out=None, attn_workspace=None,
                sample_workspace=None, status=None):
    """One verify round of one layer: append the K+1 new K/V rows, attend, sample.

    Returns (attn_out, out_tokens, num_accepted). Rolling the cache back is the
    caller's job: next round's length is seq_lens - (K+1) + num_accepted + 1.
    """
    kv_block_append(k_new, v_new, k_cache, v_cache, block_table, seq_lens, k_scale, v_scale,
                    status=status)
    out = spec_verify_attn(q, k_cache, v_cache, block_table, seq_lens, softmax_scale, k_scale,
                           v_scale, out=attn_out, workspace=attn_workspace, status=status)
    toks, nacc, _, _ = spec_verify_sample(target_logits, draft, draft_tokens, uniforms,
                                          draft_is_probs, temperature, workspace=sample_workspace,
                                          status=status, want_probs=False)
    return out, toks, nacc


# ------------------------------------------------------- block manager ---

def _host_i64(xs):
    a = (ctypes.c_int64 * max(len(xs), 1))(*[int(x) for x in xs])
    return a, len(xs)


class BlockManager:
    """Host block manager of one paged pool (sv_bm_* in the library).

    Pages 0 .. num_blocks-1 of page_size tokens; sequences are named by int
    ids. Every method runs in the library's C++ code; errors raise
    SpecVerifyError (OutOfBlocks when the pool is too small), and a failed
    call changes nothing.
    """

    def __init__(self, num_blocks, page_size=16):
        self._lib = load_library()
        h = ctypes.c_void_p()
        _check(self._lib.sv_bm_create(int(num_blocks), int(page_size), ctypes.byref(h)))
        self._h = h
        self.num_blocks = int(num_blocks)
        self.page_size = int(page_size)

    def close(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            try:
                self._lib.sv_bm_destroy(h)
            except Exception:   # interpreter shutdown: the library may be gone already
                pass
        self._h = None

    def __del__(self):
        self.close()

    @property
    def num_free(self):
        return int(self._lib.sv_bm_num_free(self._h))

    def ref_count(self, block):
        return int(self._lib.sv_bm_ref_count(self._h, int(block)))

    def ref_counts(self):
        return [self.ref_count(b) for b in range(self.num_blocks)]

    def free_list(self):
        out = (ctypes.c_int32 * self.num_blocks)()
        n = ctypes.c_int()
        _check(self._lib.sv_bm_free_list(self._h, out, self.num_blocks, ctypes.byref(n)))
        return list(out[: n.value])

    def allocate(self, seq_id, n_tokens):
        _check(self._lib.sv_bm_allocate(self._h, int(seq_id), int(n_tokens)))

    def free(self, seq_id):
        _check(self._lib.sv_bm_free(self._h, int(seq_id)))

    def fork(self, src, dst):
        _check(self._lib.sv_bm_fork(self._h, int(src), int(dst)))

    def share_prefix(self, src, dst, n_tokens):
        _check(self._lib.sv_bm_share_prefix(self._h, int(src), int(dst), int(n_tokens)))

    def extend(self, seq_ids, n_new):
        """Pages for n_new more tokens of each sequence; returns the
        copy-on-write pairs [(src_page, dst_page), ...]."""
        ids, n = _host_i64(seq_ids)
        cap = max(n, 1)
        src, dst = (ctypes.c_int32 * cap)(), (ctypes.c_int32 * cap)()
        nc = ctypes.c_int()
        _check(self._lib.sv_bm_extend(self._h, ids, n, int(n_new), src, dst, cap, ctypes.byref(nc)))
        return [(src[i], dst[i]) for i in range(nc.value)]

    def truncate(self, seq_id, new_len):
        _check(self._lib.sv_bm_truncate(self._h, int(seq_id), int(new_len)))

    def commit_verify(self, seq_ids, n_new, num_accepted):
        """Rollback after a verify round of n_new = K+1 rows; num_accepted is a
        host sequence or tensor (a CUDA tensor is copied to the host)."""
        if isinstance(num_accepted, torch.Tensor):
            num_accepted = num_accepted.detach().cpu().tolist()
        ids, n = _host_i64(seq_ids)
        if len(num_accepted) != n:
            raise ValueError("one num_accepted per sequence")
        acc = (ctypes.c_int32 * max(n, 1))(*[int(a) for a in num_accepted])
        _check(self._lib.sv_bm_commit_verify(self._h, ids, n, int(n_new), acc))

    def seq_len(self, seq_id):
        out = ctypes.c_int64()
        _check(self._lib.sv_bm_seq_len(self._h, int(seq_id), ctypes.byref(out)))
        return out.value

    def block_table(self, seq_ids, max_blocks_per_seq, device=None):
        """(block_table int32 [n, max_blocks_per_seq] padded with -1, seq_lens
        int32 [n]) as CPU tensors, or copied to `device`."""
        ids, n = _host_i64(seq_ids)
        table = torch.empty((n, int(max_blocks_per_seq)), dtype=torch.int32)
        lens = torch.empty((n,), dtype=torch.int32)
        _check(self._lib.sv_bm_block_table(self._h, ids, n, int(max_blocks_per_seq),
                                           ctypes.c_void_p(table.data_ptr()),
                                           ctypes.c_void_p(lens.data_ptr())))
        if device is not None:
            table, lens = table.to(device), lens.to(device)
        return table, lens


def copy_blocks(pools, pairs, num_blocks, block_bytes=None, block_stride_bytes=None, status=None):
    """Copy page src onto page dst of every pool for each (src, dst) pair.

    pools: CUDA tensors whose first dimension is the page index (each page a
    contiguous slice), e.g. every layer's K and V pool; block sizes default to
    one page of pools[0]."""
    if not pairs or not pools:
        return
    lib = load_library()
    _cuda(*pools, status)
    dev = pools[0].device
    if block_stride_bytes is None:
        block_stride_bytes = pools[0].stride(0) * pools[0].element_size()
    if block_bytes is None:
        block_bytes = block_stride_bytes
    for p in pools:
        if p.shape[0] < num_blocks or p.stride(0) * p.element_size() != block_stride_bytes:
            raise ValueError("every pool needs num_blocks pages of block_stride_bytes")
    pp = (ctypes.c_void_p * len(pools))(*[p.data_ptr() for p in pools])
    idx = torch.tensor(pairs, dtype=torch.int32).reshape(-1, 2).t().contiguous().to(dev)
    _check(lib.sv_copy_blocks(pp, len(pools), int(block_stride_bytes), int(block_bytes),
                              _ptr(idx[0]), _ptr(idx[1]), idx.shape[1], int(num_blocks),
                              _ptr(status), _stream()))
    return idx


def tree_verify_step(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, tree_parent, target_logits,
                     draft, tree_tokens, uniforms, k_scale=None, v_scale=None, draft_is_probs=False,
                     temperature=1.0, softmax_scale=None, typical=None, status=None):
    """One tree-verify round of one layer, in stream order: append the n node rows,
    tree attention, tree sampling, then move each accepted path next to its root
    (kv_tree_commit). Returns (attn_out, out_tokens, num_accepted, path_nodes); the
    next round's length is seq_lens - n + num_accepted + 1 (BlockManager.commit_verify)."""
    kv_block_append(k_new, v_new, k_cache, v_cache, block_table, seq_lens, k_scale, v_scale, status=status)
    out = spec_verify_attn(q, k_cache, v_cache, block_table, seq_lens, softmax_scale, k_scale, v_scale,
                           status=status, tree_parent=tree_parent)
    toks, nacc, path = spec_verify_sample_tree(target_logits, draft, tree_parent, tree_tokens, uniforms,
                                               draft_is_probs, temperature, status=status, typical=typical)
    kv_tree_commit(k_cache, v_cache, block_table, seq_lens, path, nacc, status=status)
    return out, toks, nacc, path


class MultiLayerVerify:
    """One verify round over several layers on one stream: per layer, append its
    K+1 rows into its own paged pools and attend; then one sampling pass.

    layers: list of dicts with device tensors q, k_new, v_new, k_cache, v_cache
    (and optionally k_scale, v_scale), all layers sharing block_table and
    seq_lens (one page table for the whole model, one pool pair per layer).
    Inputs and outputs stay in these static buffers, so the round can be
    captured once as a CUDA graph (capture()) and replayed (replay()); run()
    launches it directly. Attention outputs: self.outs[layer]; sampling:
    self.out_tokens, self.num_accepted.
    """

    def __init__(self, layers, block_table, seq_lens, target_logits, draft, draft_tokens, uniforms,
                 draft_is_probs=False, temperature=1.0, block_size=16):
        self.layers = layers
        self.block_table, self.seq_lens = block_table, seq_lens
        self.target_logits, self.draft = target_logits, draft
        self.draft_tokens, self.uniforms = draft_tokens, uniforms
        self.draft_is_probs, self.temperature, self.block_size = draft_is_probs, temperature, block_size
        q0 = layers[0]["q"]
        B, n_new, H_q, d = q0.shape
        H_kv = layers[0]["k_cache"].shape[1]
        dev = q0.device
        self.outs = [torch.empty_like(l["q"]) for l in layers]
        self.attn_ws = alloc_workspace(attn_workspace_size(B, n_new, H_q, H_kv, d, block_table.shape[1],
                                                           block_size), dev)
        Bs, K1, V = target_logits.shape
        self.samp_ws = alloc_workspace(sample_workspace_size(Bs, K1 - 1, V), dev)
        self.out_tokens = torch.empty((Bs, K1), dtype=torch.int32, device=dev)
        self.num_accepted = torch.empty((Bs,), dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.graph = None

    def run(self):
        for l, out in zip(self.layers, self.outs):
            kv_block_append(l["k_new"], l["v_new"], l["k_cache"], l["v_cache"], self.block_table, self.seq_lens,
                            l.get("k_scale"), l.get("v_scale"), block_size=self.block_size, status=self.status)
            spec_verify_attn(l["q"], l["k_cache"], l["v_cache"], self.block_table, self.seq_lens, None,
                             l.get("k_scale"), l.get("v_scale"), block_size=self.block_size, out=out,
                             workspace=self.attn_ws, status=self.status)
        spec_verify_sample(self.target_logits, self.draft, self.draft_tokens, self.uniforms, self.draft_is_probs,
                           self.temperature, out_tokens=self.out_tokens, num_accepted=self.num_accepted,
                           workspace=self.samp_ws, status=self.status, want_probs=False)

    def capture(self):
        """Record the round once as a CUDA graph (after one direct run, which
        also sets the kernels' attributes outside the capture)."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.run()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.run()
        return self.graph

    def replay(self):
        self.graph.replay()


def build(verbose=False, force=False):
    """Compile the CUDA library in-tree (sm_103a)."""
    return _build.build(verbose=verbose, force=force)
