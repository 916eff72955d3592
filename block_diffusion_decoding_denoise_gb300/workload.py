"""Seeded synthetic workloads for the block-diffusion denoise step.

This module only draws numbers: it holds none of the method's arithmetic
(no attention, no softmax, no commit rule).  Both the CUDA path and the CPU
oracle are fed from it, so it must stay independent of both.

Shapes follow the SDAR-1.7B decoder the MinerU-Diffusion decoder is
initialised from ("Rethinking Document OCR as Inverse Rendering via Diffusion
Decoding", reproduction paragraph: decoder initialised from SDAR-1.7B-Chat-b32,
block size 32) and the five workloads below:

  tiny_fp32        fp32, B=1, prefix 256, Hq 8 / Hkv 2, D 64, H 512, V 1024
  sdar_b1          bf16, B=1, prefix 4096, Hq 16 / Hkv 8, D 128, H 2048, V 151936
  serving_b64      bf16, B=64, prefix ~ U{2048..12288} per sequence
  longctx_b8       bf16, B=8, prefix 16384, 16 blocks (28-layer decoder shapes)
  tsweep_b32       bf16, B=32, prefix 8192, 16 blocks, T in {0.5,...,0.99}

Random streams: numpy PCG64 seeded with ``[seed, workload_id, stream_id]``;
large tensors are drawn in fixed 16 Mi-element chunks, each from its own
spawned child seed, so the bytes do not depend on the thread count.  fp32
draws are rounded to bf16 (round-to-nearest-even) for the bf16 workloads.

Planted hidden states (the confidence inputs): for every (sequence, block,
position) a target token t ~ U[0, V) is fixed; at every denoise step s a fresh
amplitude a ~ U(0, a_max) and fresh N(0,1) noise give
    h = a * W[t] / |W[t]| + noise,
so a step's h does not depend on the commit threshold.  States are drawn for
all L' possible steps of a block (the fallback rule commits at least one
position per step, so no block needs more than L' steps).
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

MASK = -1
PAGE_SIZE = 64

# stream ids (fixed forever: changing one changes every stored expectation)
S_Q, S_KBLK, S_VBLK, S_KPRE, S_VPRE, S_W = 1, 2, 3, 4, 5, 6
S_TGT, S_AMP, S_NOISE, S_PERM, S_PLEN = 7, 8, 9, 10, 11
S_EMB, S_EMASK, S_WQKV, S_WO = 12, 13, 14, 15
S_WGU, S_WDOWN = 16, 17
MLP_INTER = 6144          # SDAR-1.7B (Qwen3-1.7B family) intermediate size


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int
    dtype: str            # "f32" or "bf16"
    batch: int
    block_len: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    hidden: int
    vocab: int
    prefix: int           # fixed prefix length (or the upper bound when ragged)
    prefix_min: int       # == prefix unless lengths are drawn per sequence
    num_blocks: int
    threshold: float
    a_max: float = 12.0
    w_std: float = 0.02
    num_layers: int = 1

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 0, "f32", 1, 32, 8, 2, 64, 512, 1024,
                          256, 256, 1, 0.95),
    "sdar_b1": Workload("sdar_b1", 1, "bf16", 1, 32, 16, 8, 128, 2048, 151936,
                        4096, 4096, 1, 0.95),
    "serving_b64": Workload("serving_b64", 2, "bf16", 64, 32, 16, 8, 128, 2048,
                            151936, 12288, 2048, 1, 0.95),
    "longctx_b8": Workload("longctx_b8", 3, "bf16", 8, 32, 16, 8, 128, 2048,
                           151936, 16384, 16384, 16, 0.95, num_layers=28),
    "tsweep_b32": Workload("tsweep_b32", 4, "bf16", 32, 32, 16, 8, 128, 2048,
                           151936, 8192, 8192, 16, 0.95),
}

_CHUNK = 1 << 24


def _rng(seed: int, wid: int, stream: int, *extra: int) -> np.random.Generator:
    return np.random.default_rng([seed, wid, stream, *extra])


def normal_f32(shape, seed: int, wid: int, stream: int, *extra: int,
               std: float = 1.0) -> np.ndarray:
    """N(0, std^2) float32 array, drawn chunk-wise from spawned child seeds."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    nch = max(1, (n + _CHUNK - 1) // _CHUNK)
    children = np.random.SeedSequence([seed, wid, stream, *extra]).spawn(nch)

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(children[c]))
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        if std != 1.0:
            out[lo:hi] *= np.float32(std)

    if nch == 1:
        fill(0)
    else:
        with _cf.ThreadPoolExecutor(min(nch, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nch)))
    return out.reshape(shape)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32
    holding exactly representable bf16 values (NaN-free inputs assumed)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + r) & np.uint32(0xFFFF0000)).view(np.float32)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Values as they are stored for the workload's dtype (float32 container)."""
    return round_bf16(x) if dtype == "bf16" else np.ascontiguousarray(x, np.float32)


def prefix_lengths(w: Workload, seed: int = 0) -> np.ndarray:
    if w.prefix_min == w.prefix:
        return np.full(w.batch, w.prefix, dtype=np.int32)
    g = _rng(seed, w.wid, S_PLEN)
    return g.integers(w.prefix_min, w.prefix + 1, size=w.batch).astype(np.int32)


def lm_head(w: Workload, seed: int = 0) -> np.ndarray:
    """LM-head weight W [V, H], N(0, w_std^2), in storage precision."""
    return to_storage(normal_f32((w.vocab, w.hidden), seed, w.wid, S_W,
                                 std=w.w_std), w.dtype)


def prefix_kv(w: Workload, b: int, length: int, seed: int = 0, layer: int = 0):
    """Cached K and V of sequence b's prefix, each [length, Hkv, D], N(0,1)."""
    shp = (length, w.num_kv_heads, w.head_dim)
    k = normal_f32(shp, seed, w.wid, S_KPRE, b, layer)
    v = normal_f32(shp, seed, w.wid, S_VPRE, b, layer)
    return to_storage(k, w.dtype), to_storage(v, w.dtype)


def block_qkv(w: Workload, blk: int, seed: int = 0, layer: int = 0):
    """Q [B, L', Hq, D] and K, V [B, L', Hkv, D] of block `blk`, N(0,1)."""
    B, L = w.batch, w.block_len
    q = normal_f32((B, L, w.num_q_heads, w.head_dim), seed, w.wid, S_Q, blk, layer)
    k = normal_f32((B, L, w.num_kv_heads, w.head_dim), seed, w.wid, S_KBLK, blk, layer)
    v = normal_f32((B, L, w.num_kv_heads, w.head_dim), seed, w.wid, S_VBLK, blk, layer)
    return to_storage(q, w.dtype), to_storage(k, w.dtype), to_storage(v, w.dtype)


def planted_targets(w: Workload, blk: int, seed: int = 0) -> np.ndarray:
    """Target token t per (sequence, position) of block `blk`: [B, L'] int32."""
    g = _rng(seed, w.wid, S_TGT, blk)
    return g.integers(0, w.vocab, size=(w.batch, w.block_len)).astype(np.int32)


def planted_hidden(w: Workload, W: np.ndarray, blk: int, seed: int = 0,
                   steps: int | None = None, a_max: float | None = None):
    """Planted hidden states for every denoise step of block `blk`.

    Returns (h [steps, B, L', H] in storage precision, t [B, L'] int32).
    """
    steps = w.block_len if steps is None else steps
    a_max = w.a_max if a_max is None else a_max
    B, L, H = w.batch, w.block_len, w.hidden
    t = planted_targets(w, blk, seed)
    dirs = W[t.reshape(-1)].astype(np.float32)                   # [B*L, H]
    norms = np.sqrt((dirs.astype(np.float64) ** 2).sum(axis=1)).astype(np.float32)
    dirs /= norms[:, None]
    a = _rng(seed, w.wid, S_AMP, blk).uniform(0.0, a_max, size=(steps, B * L))
    noise = normal_f32((steps, B * L, H), seed, w.wid, S_NOISE, blk)
    h = noise + a.astype(np.float32)[:, :, None] * dirs[None]
    return to_storage(h.reshape(steps, B, L, H), w.dtype), t


def page_permutation(w: Workload, num_pages: int, seed: int = 0) -> np.ndarray:
    """A random permutation of the physical page ids [0, num_pages)."""
    return _rng(seed, w.wid, S_PERM).permutation(num_pages).astype(np.int32)


def pages_needed(length: int) -> int:
    return (length + PAGE_SIZE - 1) // PAGE_SIZE


def page_tables(w: Workload, ctx_capacity: np.ndarray, seed: int = 0):
    """Randomly permuted page tables.

    ctx_capacity[b] is the number of tokens sequence b must be able to hold.
    Returns (page_table [B, max_pages] int32, num_pages).  Unused entries are -1.
    """
    need = [pages_needed(int(c)) for c in ctx_capacity]
    num_pages = int(sum(need))
    perm = page_permutation(w, num_pages, seed)
    max_pages = max(need) if need else 0
    table = np.full((w.batch, max(1, max_pages)), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    return table, num_pages


# --- decoder-layer inputs (the 28-layer long-context workload) -----------------
def embed_table(w: Workload, seed: int = 0) -> np.ndarray:
    """Token embedding E [V, H], N(0,1), in storage precision."""
    return to_storage(normal_f32((w.vocab, w.hidden), seed, w.wid, S_EMB), w.dtype)


def mask_embedding(w: Workload, seed: int = 0) -> np.ndarray:
    """Embedding row of the mask token [H], N(0,1), in storage precision."""
    return to_storage(normal_f32((w.hidden,), seed, w.wid, S_EMASK), w.dtype)


def layer_weights(w: Workload, layer: int, seed: int = 0):
    """Projection weights of one decoder layer, N(0, w_std^2), storage precision:
    wqkv [(Hq + 2 Hkv) D, H] (rows: q heads, then k heads, then v heads) and
    wo [H, Hq D]."""
    nqkv = (w.num_q_heads + 2 * w.num_kv_heads) * w.head_dim
    wqkv = normal_f32((nqkv, w.hidden), seed, w.wid, S_WQKV, layer, std=w.w_std)
    wo = normal_f32((w.hidden, w.num_q_heads * w.head_dim), seed, w.wid, S_WO, layer,
                    std=w.w_std)
    return to_storage(wqkv, w.dtype), to_storage(wo, w.dtype)


def mlp_weights(w: Workload, layer: int, inter: int = MLP_INTER, seed: int = 0):
    """Weights of the optional gated MLP of one layer, N(0, w_std^2), storage
    precision: w_gate_up [2 inter, H] (gate rows, then up rows) and
    w_down [H, inter]."""
    wgu = normal_f32((2 * inter, w.hidden), seed, w.wid, S_WGU, layer, std=w.w_std)
    wd = normal_f32((w.hidden, inter), seed, w.wid, S_WDOWN, layer, std=w.w_std)
    return to_storage(wgu, w.dtype), to_storage(wd, w.dtype)

