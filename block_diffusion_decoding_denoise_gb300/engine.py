"""Denoise-loop driver over the libbd C ABI.

Holds the device state of one decoding batch (paged KV cache, token state,
workspaces) and runs the block loop:

    for each block:  tokens := MASK
                     repeat   bd_block_attention ; bd_confidence_commit
                     until    no position of any sequence is masked
                     bd_append_block_kv

("Rethinking Document OCR as Inverse Rendering via Diffusion Decoding",
paper.rainbus.top summary, method steps 2-4: blocks in order, every step
refines the current block, confident tokens are confirmed, the rest is
denoised again; the novelty paragraph's KV-cache reuse across blocks.)

The loop issues steps asynchronously and reads the per-sequence masked count
back only every `check_every` steps; kernels skip sequences that are already
finished, so speculative steps past the end cost only empty launches.  All
arithmetic runs in libbd's kernels; torch provides memory and streams.
"""
from __future__ import annotations

import numpy as np
import torch

from . import bd

MASK = bd.BD_MASK


class PagedCache:
    """K/V pools [num_pages, Hkv, 64, D] of one layer plus the page table."""

    def __init__(self, num_pages: int, num_kv_heads: int, head_dim: int, dtype,
                 page_table: np.ndarray, device="cuda"):
        self.k = torch.zeros(num_pages, num_kv_heads, bd.BD_PAGE_SIZE, head_dim,
                             dtype=dtype, device=device)
        self.v = torch.zeros_like(self.k)
        self.page_table_np = np.ascontiguousarray(page_table, dtype=np.int32)
        self.page_table = torch.from_numpy(self.page_table_np).to(device)
        self.kv = bd.paged_kv(self.k, self.v, self.page_table)

    @property
    def capacity(self) -> int:
        return self.page_table.shape[1] * bd.BD_PAGE_SIZE

    def load_prefix(self, b: int, k_prefix, v_prefix):
        """Place a sequence's cached K/V ([len, Hkv, D]) into its pages."""
        n = k_prefix.shape[0]
        if n == 0:
            return
        pos = np.arange(n)
        pages = torch.from_numpy(self.page_table_np[b][pos // bd.BD_PAGE_SIZE].astype(np.int64))
        slots = torch.from_numpy((pos % bd.BD_PAGE_SIZE).astype(np.int64))
        pages, slots = pages.to(self.k.device), slots.to(self.k.device)
        self.k[pages, :, slots, :] = torch.as_tensor(k_prefix).to(self.k.device, self.k.dtype)
        self.v[pages, :, slots, :] = torch.as_tensor(v_prefix).to(self.v.device, self.v.dtype)


class DenoiseEngine:
    """One batch of sequences decoding blocks of `block_len` tokens."""

    def __init__(self, lm_head: torch.Tensor, caches, ctx_len, *, batch: int, block_len: int,
                 num_q_heads: int, threshold: float, max_ctx: int):
        self.W = lm_head
        self.caches = caches if isinstance(caches, (list, tuple)) else [caches]
        self.B, self.L, self.Hq = batch, block_len, num_q_heads
        self.T = float(threshold)
        self.max_ctx = int(max_ctx)
        dev = lm_head.device
        c0 = self.caches[0]
        self.Hkv, self.D = c0.k.shape[1], c0.k.shape[3]
        self.dtype = lm_head.dtype
        self.V, self.H = lm_head.shape
        self.ctx_len = torch.as_tensor(np.asarray(ctx_len, np.int32)).to(dev)
        self.tokens = torch.full((batch, block_len), MASK, dtype=torch.int32, device=dev)
        self.p_max = torch.empty(batch, block_len, dtype=torch.float32, device=dev)
        self.argmax = torch.empty(batch, block_len, dtype=torch.int32, device=dev)
        self.n_committed = torch.zeros(block_len + 1, batch, dtype=torch.int32, device=dev)
        self.n_masked = torch.zeros(batch, dtype=torch.int32, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.attn_out = torch.empty(batch, block_len, num_q_heads, self.D, dtype=self.dtype,
                                    device=dev)
        code = bd.BD_BF16 if self.dtype == torch.bfloat16 else bd.BD_F32
        aws = bd.bd_block_attention_workspace(batch, block_len, num_q_heads, self.Hkv, self.D,
                                              self.max_ctx)
        cws = bd.bd_confidence_commit_workspace(code, batch, block_len, self.H, self.V)
        if cws == 0:
            raise ValueError("unsupported confidence-commit shape")
        self.attn_ws = torch.empty(max(aws, 1), dtype=torch.uint8, device=dev)
        self.conf_ws = torch.empty(cws, dtype=torch.uint8, device=dev)
        self._host_masked = torch.empty(batch, dtype=torch.int32, pin_memory=True)
        self._graphs = {}
        self.graph_kernel_launches = 0   # kernels launched by graph replays

    # -- one denoise step ---------------------------------------------------
    def step(self, h, q, k_blk, v_blk, n_committed_out=None, layer: int = 0):
        bd.bd_block_attention(self.caches[layer].kv, self.ctx_len, self.tokens, q, k_blk, v_blk,
                              self.attn_out, self.attn_ws, self.max_ctx,
                              dev_status=self.dev_status)
        bd.bd_confidence_commit(h, self.W, self.T, self.tokens, self.p_max, self.argmax,
                                self.n_committed[0] if n_committed_out is None
                                else n_committed_out, self.n_masked, self.conf_ws,
                                dev_status=self.dev_status)

    # -- CUDA graphs of step chunks -----------------------------------------
    def _chunk_graph(self, h_steps, q, k_blk, v_blk, s0: int, s1: int):
        """Graph of denoise steps [s0, s1) over these input buffers (captured once).

        Replaying it issues exactly the launches of the eager loop, with no
        host work per kernel."""
        key = (h_steps.data_ptr(), q.data_ptr(), k_blk.data_ptr(), v_blk.data_ptr(), s0, s1,
               self.step)
        entry = self._graphs.get(key)
        if entry is None:
            g = torch.cuda.CUDAGraph()
            n0 = bd.bd_kernel_launches()
            with torch.cuda.graph(g):
                for s in range(s0, s1):
                    self.step(h_steps[s], q, k_blk, v_blk, self.n_committed[s])
            entry = (g, bd.bd_kernel_launches() - n0)
            self._graphs[key] = entry
        return entry

    # -- one block ----------------------------------------------------------
    def decode_block(self, h_steps, q, k_blk, v_blk, check_every: int = 8,
                     graphs: bool = False, on_chunk=None):
        """Denoise the current block to completion and append its K/V.

        h_steps [S, B, L, H] (S >= block_len) holds each step's hidden
        states.  Steps run in chunks of `check_every` (replayed CUDA graphs
        when `graphs`); after each chunk the host reads the masked count and
        `on_chunk(s0, s1)` is called.  Returns the number of denoise steps
        issued; per-sequence step counts come from `steps_per_sequence()`.
        """
        self.tokens.fill_(MASK)
        self.n_committed.zero_()
        s = 0
        while True:
            s1 = min(self.L, s + check_every)
            if graphs:
                g, n_kernels = self._chunk_graph(h_steps, q, k_blk, v_blk, s, s1)
                g.replay()
                self.graph_kernel_launches += n_kernels
            else:
                for t in range(s, s1):
                    self.step(h_steps[t], q, k_blk, v_blk, self.n_committed[t])
            self._host_masked.copy_(self.n_masked, non_blocking=True)
            torch.cuda.current_stream().synchronize()
            if on_chunk is not None:
                on_chunk(s, s1)
            s = s1
            if int(self._host_masked.sum()) == 0 or s >= self.L:
                break
        bd.bd_append_block_kv(self.caches[0].kv, k_blk, v_blk, self.ctx_len, self.n_masked,
                              self.dev_status)
        return s

    def steps_per_sequence(self) -> np.ndarray:
        """Denoise steps each sequence took in the last block (>= 1 commit each)."""
        return (self.n_committed.cpu().numpy() > 0).sum(axis=0)

    def check_status(self):
        st = int(self.dev_status.item())
        if st != 0:
            raise bd.BDError("device check", st)
