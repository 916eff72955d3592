"""ctypes binding of libbd.so (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it checks that tensors live on the GPU with the right
dtype and layout, passes their device pointers and the current CUDA stream,
and raises BDError on a non-OK status.  Torch is used for device memory and
streams only.  There is no CPU fallback: if libbd.so has not been built the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int32, c_size_t, c_void_p

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbd.so")

BD_F32, BD_BF16 = 0, 1
BD_MASK = -1
BD_PAGE_SIZE = 64
STATUS = {0: "BD_OK", 1: "BD_ERR_INVALID_ARG", 2: "BD_ERR_UNSUPPORTED", 3: "BD_ERR_CUDA",
          4: "BD_ERR_DEVICE_CHECK", 5: "BD_ERR_TIMEOUT", 6: "BD_ERR_WORKSPACE"}

# every symbol include/bd.h declares
EXPORTS = ("bd_block_attention_workspace", "bd_block_attention",
           "bd_confidence_commit_workspace", "bd_confidence_commit",
           "bd_append_block_kv", "bd_status_string", "bd_version", "bd_kernel_launches",
           "bd_confidence_commit_noalloc", "bd_sample_commit_workspace", "bd_sample_commit",
           "bd_embed_rmsnorm", "bd_qkv_projection_workspace", "bd_qkv_projection",
           "bd_out_projection_workspace", "bd_out_projection_residual",
           "bd_append_block_kv_layers", "bd_confidence_commit_regions",
           "bd_sample_commit_truncated_workspace", "bd_sample_commit_truncated",
           "bd_mlp_workspace", "bd_mlp_residual", "bd_debug_force_attention_kernel", "bd_debug_wait_timeout_selftest",
           "bd_confidence_shard_workspace", "bd_confidence_shard", "bd_commit_shards",
           "bd_merge_conf_records_host", "bd_merge_attention_partials_host",
           "bd_merge_attention_partials")

# bd_attention_kernel values of bd_debug_force_attention_kernel (test hook)
BD_ATTN = {"auto": 0, "pair": 1, "mma": 2, "simt": 3, "cluster": 4, "pair_cluster": 5}


class BDError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")
        self.status = status


class PagedKV(ctypes.Structure):
    """Mirror of bd_paged_kv."""
    _fields_ = [("dtype", c_int32), ("num_pages", c_int32), ("page_size", c_int32),
                ("num_kv_heads", c_int32), ("head_dim", c_int32),
                ("max_pages_per_seq", c_int32), ("k_pool", c_void_p),
                ("v_pool", c_void_p), ("page_table", c_void_p)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libbd.so once; raise if it is missing (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built; run "
                               "`python -m block_diffusion_decoding_denoise_gb300.build`")
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(PagedKV)
        sig = {
            "bd_block_attention_workspace": (c_size_t, [c_int32] * 6),
            "bd_block_attention": (c_int32, [P, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                             c_int32, c_void_p, c_void_p, c_void_p, c_float,
                                             c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]),
            "bd_confidence_commit_workspace": (c_size_t, [c_int32] * 5),
            "bd_confidence_commit": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_int32,
                                               c_void_p, c_void_p, c_float, c_void_p, c_void_p,
                                               c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                               c_void_p, c_void_p]),
            "bd_confidence_commit_regions": (c_int32, [c_int32, c_int32, c_int32, c_int32,
                                                       c_int32, c_void_p, c_void_p, c_void_p,
                                                       c_void_p, c_void_p, c_void_p, c_void_p,
                                                       c_void_p, c_void_p, c_size_t, c_void_p,
                                                       c_void_p]),
            "bd_append_block_kv": (c_int32, [P, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                             c_void_p, c_void_p, c_void_p]),
            "bd_status_string": (ctypes.c_char_p, [c_int32]),
            "bd_version": (c_int32, []),
            "bd_kernel_launches": (ctypes.c_uint64, []),
            "bd_debug_force_attention_kernel": (c_int32, [c_int32]),
            "bd_debug_wait_timeout_selftest": (c_int32, [c_void_p, c_void_p]),
            "bd_confidence_shard_workspace": (c_size_t, [c_int32] * 5),
            "bd_confidence_shard": (c_int32, [c_int32] * 6 + [c_void_p] * 5 + [c_size_t, c_void_p,
                                                                            c_void_p]),
            "bd_commit_shards": (c_int32, [c_int32] * 4 + [c_void_p, c_float] + [c_void_p] * 7),
            "bd_merge_conf_records_host": (c_int32, [c_int32, ctypes.c_int64, c_void_p, c_void_p]),
            "bd_merge_attention_partials_host": (c_int32, [c_int32, ctypes.c_int64, c_int32,
                                                           c_void_p, c_void_p, c_void_p, c_void_p]),
            "bd_merge_attention_partials": (c_int32, [c_int32, ctypes.c_int64, c_int32, c_void_p,
                                                      c_void_p, c_void_p, c_int32, c_void_p,
                                                      c_void_p]),
            "bd_confidence_commit_noalloc": (c_int32, [c_int32, c_int32, c_int32, c_int32,
                                                       c_int32, c_void_p, c_void_p, c_float,
                                                       c_void_p, c_void_p, c_void_p, c_void_p,
                                                       c_void_p, c_void_p, c_void_p]),
            "bd_sample_commit_workspace": (c_size_t, [c_int32] * 5),
            "bd_sample_commit": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_int32,
                                           c_void_p, c_void_p, c_float, c_float, ctypes.c_uint64,
                                           c_void_p, c_void_p, c_void_p, c_void_p,
                                           c_void_p, c_void_p, c_void_p, c_size_t, c_void_p,
                                           c_void_p]),
            "bd_sample_commit_truncated_workspace": (c_size_t, [c_int32] * 5),
            "bd_sample_commit_truncated": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_int32,
                                                     c_void_p, c_void_p, c_float, c_float,
                                                     c_int32, c_float, ctypes.c_uint64,
                                                     c_void_p, c_void_p, c_void_p, c_void_p,
                                                     c_void_p, c_void_p, c_void_p, c_size_t,
                                                     c_void_p, c_void_p]),
            "bd_mlp_workspace": (c_size_t, [c_int32] * 3),
            "bd_mlp_residual": (c_int32, [c_int32] * 3 + [c_void_p, c_void_p, c_void_p, c_float,
                                                         c_void_p, c_void_p, c_void_p, c_size_t,
                                                         c_void_p, c_void_p]),
            "bd_embed_rmsnorm": (c_int32, [c_int32, c_int32, c_int32, c_void_p, c_void_p,
                                           c_void_p, c_float, c_void_p, c_void_p, c_void_p,
                                           c_void_p]),
            "bd_qkv_projection_workspace": (c_size_t, [c_int32] * 5),
            "bd_qkv_projection": (c_int32, [c_int32] * 5 + [c_void_p] * 6 +
                                  [c_size_t, c_void_p, c_void_p]),
            "bd_out_projection_workspace": (c_size_t, [c_int32] * 3),
            "bd_out_projection_residual": (c_int32, [c_int32] * 3 + [c_void_p, c_void_p, c_float,
                                                                    c_void_p, c_void_p, c_void_p,
                                                                    c_size_t, c_void_p,
                                                                    c_void_p]),
            "bd_append_block_kv_layers": (c_int32, [P, c_int32, c_int32, c_int32, c_void_p,
                                                    c_void_p, c_void_p, c_void_p, c_void_p,
                                                    c_void_p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return BD_F32
    if t.dtype == torch.bfloat16:
        return BD_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(fn: str, status: int):
    if status != 0:
        raise BDError(fn, status)


def paged_kv(k_pool: torch.Tensor, v_pool: torch.Tensor, page_table: torch.Tensor) -> PagedKV:
    """bd_paged_kv for pools [num_pages, Hkv, 64, D] and a [B, max_pages] int32 table."""
    if k_pool.shape != v_pool.shape or k_pool.dim() != 4 or k_pool.dtype != v_pool.dtype:
        raise ValueError("k_pool and v_pool must both be [num_pages, Hkv, page_size, D]")
    if page_table.dim() != 2:
        raise ValueError("page_table must be [batch, max_pages_per_seq]")
    return PagedKV(_dtype_code(k_pool), k_pool.shape[0], k_pool.shape[2], k_pool.shape[1],
                   k_pool.shape[3], page_table.shape[1], _ptr(k_pool, name="k_pool"),
                   _ptr(v_pool, name="v_pool"), _ptr(page_table, torch.int32, "page_table"))


def bd_block_attention_workspace(batch, block_len, num_q_heads, num_kv_heads, head_dim,
                                 max_ctx) -> int:
    return int(load().bd_block_attention_workspace(batch, block_len, num_q_heads, num_kv_heads,
                                                   head_dim, max_ctx))


def bd_block_attention(kv: PagedKV, ctx_len, tokens, q, k_blk, v_blk, out, ws, max_ctx,
                       softmax_scale=None, dev_status=None, stream=None):
    B, L, Hq, D = q.shape
    scale = D ** -0.5 if softmax_scale is None else softmax_scale
    st = load().bd_block_attention(
        ctypes.byref(kv), _ptr(ctx_len, torch.int32, "ctx_len"),
        _ptr(tokens, torch.int32, "tokens"), B, L, Hq, max_ctx, _ptr(q, name="q"),
        _ptr(k_blk, name="k_blk"), _ptr(v_blk, name="v_blk"), scale, _ptr(out, name="out"),
        _ptr(ws, name="ws") if ws is not None and ws.numel() else None,
        0 if ws is None else ws.numel() * ws.element_size(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("bd_block_attention", st)


def bd_confidence_commit_workspace(dtype_code, batch, block_len, hidden, vocab) -> int:
    return int(load().bd_confidence_commit_workspace(dtype_code, batch, block_len, hidden, vocab))


def bd_confidence_commit(hidden_states, lm_head, threshold, tokens, p_max, argmax,
                         n_committed, n_masked, ws, dev_status=None, stream=None):
    B, L, H = hidden_states.shape
    V = lm_head.shape[0]
    if lm_head.shape[1] != H or lm_head.dtype != hidden_states.dtype:
        raise ValueError("lm_head must be [vocab, hidden] with the hidden states' dtype")
    st = load().bd_confidence_commit(
        _dtype_code(hidden_states), B, L, H, V, _ptr(hidden_states, name="hidden_states"),
        _ptr(lm_head, name="lm_head"), float(threshold), _ptr(tokens, torch.int32, "tokens"),
        _ptr(p_max, torch.float32, "p_max"), _ptr(argmax, torch.int32, "argmax"),
        _ptr(n_committed, torch.int32, "n_committed"), _ptr(n_masked, torch.int32, "n_masked"),
        _ptr(ws, name="ws"), ws.numel() * ws.element_size(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("bd_confidence_commit", st)


def bd_confidence_commit_regions(hidden_states, lm_head, thresholds, tokens, p_max, argmax,
                                 n_committed, n_masked, ws, dev_status=None, stream=None):
    """bd_confidence_commit with a per-position threshold array
    `thresholds` [B, L'] float32 on the device (region thresholds)."""
    B, L, H = hidden_states.shape
    V = lm_head.shape[0]
    if lm_head.shape[1] != H or lm_head.dtype != hidden_states.dtype:
        raise ValueError("lm_head must be [vocab, hidden] with the hidden states' dtype")
    if tuple(thresholds.shape) != (B, L):
        raise ValueError("thresholds must be [batch, block_len]")
    st = load().bd_confidence_commit_regions(
        _dtype_code(hidden_states), B, L, H, V, _ptr(hidden_states, name="hidden_states"),
        _ptr(lm_head, name="lm_head"), _ptr(thresholds, torch.float32, "thresholds"),
        _ptr(tokens, torch.int32, "tokens"),
        _ptr(p_max, torch.float32, "p_max"), _ptr(argmax, torch.int32, "argmax"),
        _ptr(n_committed, torch.int32, "n_committed"), _ptr(n_masked, torch.int32, "n_masked"),
        _ptr(ws, name="ws"), ws.numel() * ws.element_size(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("bd_confidence_commit_regions", st)


def bd_confidence_commit_noalloc(hidden_states, lm_head, threshold, tokens, p_max, argmax,
                                 n_committed, n_masked, dev_status=None, stream=None):
    """bd_confidence_commit with the library's fixed device scratch array in
    place of a caller workspace, for callers that cannot allocate (see bd.h)."""
    B, L, H = hidden_states.shape
    V = lm_head.shape[0]
    if lm_head.shape[1] != H or lm_head.dtype != hidden_states.dtype:
        raise ValueError("lm_head must be [vocab, hidden] with the hidden states' dtype")
    st = load().bd_confidence_commit_noalloc(
        _dtype_code(hidden_states), B, L, H, V, _ptr(hidden_states, name="hidden_states"),
        _ptr(lm_head, name="lm_head"), float(threshold), _ptr(tokens, torch.int32, "tokens"),
        _ptr(p_max, torch.float32, "p_max"), _ptr(argmax, torch.int32, "argmax"),
        _ptr(n_committed, torch.int32, "n_committed"), _ptr(n_masked, torch.int32, "n_masked"),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("bd_confidence_commit_noalloc", st)


def bd_sample_commit_workspace(dtype_code, batch, block_len, hidden, vocab) -> int:
    return int(load().bd_sample_commit_workspace(dtype_code, batch, block_len, hidden, vocab))


def bd_sample_commit(hidden_states, lm_head, threshold, temperature, seed, offset, tokens,
                     p_sel, sampled, n_committed, n_masked, ws, dev_status=None, stream=None):
    """`offset` is a one-element int64 CUDA tensor: the draw counter the call
    reads and advances by one (see bd.h)."""
    B, L, H = hidden_states.shape
    V = lm_head.shape[0]
    if lm_head.shape[1] != H or lm_head.dtype != hidden_states.dtype:
        raise ValueError("lm_head must be [vocab, hidden] with the hidden states' dtype")
    st = load().bd_sample_commit(
        _dtype_code(hidden_states), B, L, H, V, _ptr(hidden_states, name="hidden_states"),
        _ptr(lm_head, name="lm_head"), float(threshold), float(temperature),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(offset, torch.int64, "offset"),
        _ptr(tokens, torch.int32, "tokens"), _ptr(p_sel, torch.float32, "p_sel"),
        _ptr(sampled, torch.int32, "sampled"), _ptr(n_committed, torch.int32, "n_committed"),
        _ptr(n_masked, torch.int32, "n_masked"), _ptr(ws, name="ws"),
        ws.numel() * ws.element_size(), _ptr(dev_status, torch.int32, "dev_status"),
        _stream(stream))
    _check("bd_sample_commit", st)


def bd_sample_commit_truncated_workspace(dtype_code, batch, block_len, hidden, vocab) -> int:
    return int(load().bd_sample_commit_truncated_workspace(dtype_code, batch, block_len, hidden,
                                                           vocab))


def bd_sample_commit_truncated(hidden_states, lm_head, threshold, temperature, top_k, top_p,
                               seed, offset, tokens, p_sel, sampled, n_committed, n_masked, ws,
                               dev_status=None, stream=None):
    """bd_sample_commit with top-k / top-p truncation (see bd.h)."""
    B, L, H = hidden_states.shape
    V = lm_head.shape[0]
    if lm_head.shape[1] != H or lm_head.dtype != hidden_states.dtype:
        raise ValueError("lm_head must be [vocab, hidden] with the hidden states' dtype")
    st = load().bd_sample_commit_truncated(
        _dtype_code(hidden_states), B, L, H, V, _ptr(hidden_states, name="hidden_states"),
        _ptr(lm_head, name="lm_head"), float(threshold), float(temperature), int(top_k),
        float(top_p), int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(offset, torch.int64, "offset"),
        _ptr(tokens, torch.int32, "tokens"), _ptr(p_sel, torch.float32, "p_sel"),
        _ptr(sampled, torch.int32, "sampled"), _ptr(n_committed, torch.int32, "n_committed"),
        _ptr(n_masked, torch.int32, "n_masked"), _ptr(ws, name="ws"),
        ws.numel() * ws.element_size(), _ptr(dev_status, torch.int32, "dev_status"),
        _stream(stream))
    _check("bd_sample_commit_truncated", st)


def bd_append_block_kv(kv: PagedKV, k_blk, v_blk, ctx_len, n_masked=None, dev_status=None,
                       stream=None):
    B, L = k_blk.shape[0], k_blk.shape[1]
    st = load().bd_append_block_kv(
        ctypes.byref(kv), B, L, _ptr(k_blk, name="k_blk"), _ptr(v_blk, name="v_blk"),
        _ptr(ctx_len, torch.int32, "ctx_len"), _ptr(n_masked, torch.int32, "n_masked"),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("bd_append_block_kv", st)


def bd_status_string(status: int) -> str:
    return load().bd_status_string(status).decode()


def bd_version() -> int:
    return int(load().bd_version())


def bd_kernel_launches() -> int:
    return int(load().bd_kernel_launches())


def bd_debug_wait_timeout_selftest(dev_status, stream=None):
    """Test hook: one CTA whose bounded wait runs out (BD_ERR_TIMEOUT in dev_status)."""
    _check("bd_debug_wait_timeout_selftest",
           load().bd_debug_wait_timeout_selftest(_ptr(dev_status, torch.int32, "dev_status"),
                                                 _stream(stream)))


def bd_debug_force_attention_kernel(which: str):
    """Test hook: force one attention kernel ("auto" restores the choice by shape)."""
    _check("bd_debug_force_attention_kernel",
           load().bd_debug_force_attention_kernel(BD_ATTN[which]))


# --- decoder layer stack --------------------------------------------------------
def bd_embed_rmsnorm(tokens, embed, mask_embed, x, xn, eps=1e-6, dev_status=None, stream=None):
    rows = tokens.numel()
    V, H = embed.shape
    st = load().bd_embed_rmsnorm(
        rows, H, V, _ptr(tokens, torch.int32, "tokens"), _ptr(embed, torch.bfloat16, "embed"),
        _ptr(mask_embed, torch.bfloat16, "mask_embed"), float(eps),
        _ptr(x, torch.float32, "x"), _ptr(xn, torch.bfloat16, "xn"),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("bd_embed_rmsnorm", st)


def bd_qkv_projection_workspace(rows, hidden, num_q_heads, num_kv_heads, head_dim) -> int:
    return int(load().bd_qkv_projection_workspace(rows, hidden, num_q_heads, num_kv_heads,
                                                  head_dim))


def bd_qkv_projection(xn, w_qkv, q, k, v, ws, dev_status=None, stream=None):
    rows, H = xn.shape[0] * (xn.shape[1] if xn.dim() == 3 else 1), xn.shape[-1]
    Hq, D = q.shape[-2], q.shape[-1]
    Hkv = k.shape[-2]
    st = load().bd_qkv_projection(
        rows, H, Hq, Hkv, D, _ptr(xn, torch.bfloat16, "xn"), _ptr(w_qkv, torch.bfloat16, "w_qkv"),
        _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"),
        _ptr(ws, name="ws"), ws.numel() * ws.element_size(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("bd_qkv_projection", st)


def bd_out_projection_workspace(rows, in_features, hidden) -> int:
    return int(load().bd_out_projection_workspace(rows, in_features, hidden))


def bd_out_projection_residual(attn, w_o, x, xn, ws, eps=1e-6, dev_status=None, stream=None):
    H, Fin = w_o.shape
    rows = x.numel() // H
    st = load().bd_out_projection_residual(
        rows, Fin, H, _ptr(attn, torch.bfloat16, "attn"), _ptr(w_o, torch.bfloat16, "w_o"),
        float(eps), _ptr(x, torch.float32, "x"), _ptr(xn, torch.bfloat16, "xn"),
        _ptr(ws, name="ws"), ws.numel() * ws.element_size(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("bd_out_projection_residual", st)


def bd_mlp_workspace(rows, hidden, inter) -> int:
    return int(load().bd_mlp_workspace(rows, hidden, inter))


def bd_mlp_residual(xn, w_gate_up, w_down, x, xn_out, ws, eps=1e-6, dev_status=None,
                    stream=None):
    """x += bf16(silu(g) * u) w_down^T with [g | u] = xn w_gate_up^T, then
    xn_out = bf16(RMSNorm(x)) (see bd.h)."""
    H = w_down.shape[0]
    inter = w_down.shape[1]
    if tuple(w_gate_up.shape) != (2 * inter, H):
        raise ValueError("w_gate_up must be [2 * inter, hidden]")
    rows = x.numel() // H
    st = load().bd_mlp_residual(
        rows, H, inter, _ptr(xn, torch.bfloat16, "xn"),
        _ptr(w_gate_up, torch.bfloat16, "w_gate_up"), _ptr(w_down, torch.bfloat16, "w_down"),
        float(eps), _ptr(x, torch.float32, "x"), _ptr(xn_out, torch.bfloat16, "xn_out"),
        _ptr(ws, name="ws"), ws.numel() * ws.element_size(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("bd_mlp_residual", st)


def bd_append_block_kv_layers(kvs, k_blk, v_blk, ctx_len, n_masked=None, dev_status=None,
                              stream=None):
    """kvs: list of PagedKV (one per layer, shared page table); k_blk/v_blk
    [layers, B, L', Hkv, D]."""
    arr = (PagedKV * len(kvs))(*kvs)
    L_, B, L = k_blk.shape[0], k_blk.shape[1], k_blk.shape[2]
    if L_ != len(kvs):
        raise ValueError("k_blk must hold one block per layer")
    st = load().bd_append_block_kv_layers(
        arr, len(kvs), B, L, _ptr(k_blk, name="k_blk"), _ptr(v_blk, name="v_blk"),
        _ptr(ctx_len, torch.int32, "ctx_len"), _ptr(n_masked, torch.int32, "n_masked"),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("bd_append_block_kv_layers", st)


# --- one sequence split across GPUs (vocabulary slices, key slices) ------------
RECORD_INTS = 3          # bd_conf_record: float m, float s, int32 idx


def bd_confidence_shard_workspace(batch, block_len, hidden, vocab_shard) -> int:
    return int(load().bd_confidence_shard_workspace(BD_BF16, batch, block_len, hidden,
                                                    vocab_shard))


def bd_confidence_shard(h, w_shard, vocab_offset, tokens, records, ws, dev_status=None,
                        stream=None):
    """records: int32 CUDA tensor [batch * block_len, 3] (bd_conf_record)."""
    B, L, H = h.shape
    Vs = w_shard.shape[0]
    if records.dtype != torch.int32 or records.numel() != B * L * RECORD_INTS:
        raise TypeError("records must be int32 [batch * block_len, 3]")
    st = load().bd_confidence_shard(
        BD_BF16, B, L, H, Vs, int(vocab_offset), _ptr(h, torch.bfloat16, "h"),
        _ptr(w_shard, torch.bfloat16, "w_shard"), _ptr(tokens, torch.int32, "tokens"),
        _ptr(records, torch.int32, "records"), _ptr(ws, name="ws"), ws.numel(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("bd_confidence_shard", st)


def bd_commit_shards(records, vocab, threshold, tokens, p_max, argmax, n_committed, n_masked,
                     dev_status=None, stream=None):
    """records: int32 CUDA tensor [num_shards, batch * block_len, 3]."""
    B, L = tokens.shape
    S = records.shape[0]
    if records.dtype != torch.int32 or records.numel() != S * B * L * RECORD_INTS:
        raise TypeError("records must be int32 [num_shards, batch * block_len, 3]")
    st = load().bd_commit_shards(
        B, L, int(vocab), S, _ptr(records, torch.int32, "records"), float(threshold),
        _ptr(tokens, torch.int32, "tokens"), _ptr(p_max, torch.float32, "p_max"),
        _ptr(argmax, torch.int32, "argmax"), _ptr(n_committed, torch.int32, "n_committed"),
        _ptr(n_masked, torch.int32, "n_masked"), _ptr(dev_status, torch.int32, "dev_status"),
        _stream(stream))
    _check("bd_commit_shards", st)


def bd_merge_conf_records_host(records):
    """records: numpy structured array [num_shards, n] of (m f4, s f4, idx i4),
    C-contiguous; returns the merged [n] array."""
    import numpy as np
    rec = np.ascontiguousarray(records)
    S, n = rec.shape
    out = np.empty(n, dtype=rec.dtype)
    st = load().bd_merge_conf_records_host(S, n, rec.ctypes.data, out.ctypes.data)
    _check("bd_merge_conf_records_host", st)
    return out


def bd_merge_attention_partials_host(m, l, o):
    """m, l: float32 [num_shards, rows]; o: float32 [num_shards, rows, D] (host)."""
    import numpy as np
    m = np.ascontiguousarray(m, np.float32)
    l = np.ascontiguousarray(l, np.float32)
    o = np.ascontiguousarray(o, np.float32)
    S, R, D = o.shape
    out = np.empty((R, D), np.float32)
    st = load().bd_merge_attention_partials_host(S, R, D, m.ctypes.data, l.ctypes.data,
                                                 o.ctypes.data, out.ctypes.data)
    _check("bd_merge_attention_partials_host", st)
    return out


def bd_merge_attention_partials(m, l, o, out, stream=None):
    """Device merge: m, l [S, rows], o [S, rows, D] fp32 CUDA; out [rows, D] fp32/bf16."""
    S, R, D = o.shape
    st = load().bd_merge_attention_partials(
        S, R, D, _ptr(m, torch.float32, "m"), _ptr(l, torch.float32, "l"),
        _ptr(o, torch.float32, "o"), _dtype_code(out), _ptr(out, name="out"), _stream(stream))
    _check("bd_merge_attention_partials", st)
