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

import gc

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
                 num_q_heads: int, threshold: float, max_ctx: int,
                 temperature: float | None = None, seed: int = 0, decoder=None,
                 top_k: int = 0, top_p: float = 1.0):
        """`threshold`: one number, or a [batch, block_len] array of
        per-position thresholds (region thresholds, greedy only:
        bd_confidence_commit_regions).
        `temperature` None: greedy confidence (bd_confidence_commit); a
        number: sampled tokens (bd_sample_commit) with key `seed` and a device
        draw counter that every step advances, also under graph replay;
        `top_k` > 0 or `top_p` < 1 truncate the sampled distribution
        (bd_sample_commit_truncated).
        `decoder` (a DecoderStack sharing this engine's ctx_len): every step
        runs the layer stack over the current tokens (its attention replaces
        the single-layer attention call), and a finished block is run through
        the stack once more with its committed tokens to produce the K/V that
        every layer appends."""
        self.decoder = decoder
        self.W = lm_head
        self.caches = caches if isinstance(caches, (list, tuple)) else [caches]
        self.B, self.L, self.Hq = batch, block_len, num_q_heads
        dev = lm_head.device
        self.thresholds = None
        if np.ndim(threshold) == 0:
            self.T = float(threshold)
        else:
            if temperature is not None:
                raise ValueError("per-position thresholds are a greedy-commit option")
            thr = np.asarray(threshold, np.float32)
            if thr.shape != (batch, block_len):
                raise ValueError("per-position thresholds must be [batch, block_len]")
            self.T = None
            self.thresholds = torch.as_tensor(thr).to(dev)
        self.max_ctx = int(max_ctx)
        c0 = self.caches[0]
        self.Hkv, self.D = c0.k.shape[1], c0.k.shape[3]
        self.dtype = lm_head.dtype
        self.V, self.H = lm_head.shape
        self.ctx_len = (decoder.ctx_len if decoder is not None
                        else torch.as_tensor(np.asarray(ctx_len, np.int32)).to(dev))
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
        self.temperature = None if temperature is None else float(temperature)
        self.seed = int(seed)
        self.draw_counter = torch.zeros(1, dtype=torch.int64, device=dev)
        self.top_k, self.top_p = int(top_k), float(top_p)
        self.truncated = self.top_k > 0 or self.top_p < 1.0
        if self.truncated and self.temperature is None:
            raise ValueError("top-k / top-p truncation needs a sampling temperature")
        query = (bd.bd_confidence_commit_workspace if self.temperature is None
                 else bd.bd_sample_commit_truncated_workspace if self.truncated
                 else bd.bd_sample_commit_workspace)
        cws = query(code, batch, block_len, self.H, self.V)
        if cws == 0:
            raise ValueError("unsupported confidence-commit shape")
        self.attn_ws = torch.empty(max(aws, 1), dtype=torch.uint8, device=dev)
        self.conf_ws = torch.empty(cws, dtype=torch.uint8, device=dev)
        self._host_masked = torch.empty(batch, dtype=torch.int32, pin_memory=True)
        self._graphs = {}
        self.graph_kernel_launches = 0   # kernels launched by graph replays

    # -- one denoise step ---------------------------------------------------
    def step(self, h, q, k_blk, v_blk, n_committed_out=None, layer: int = 0):
        if self.decoder is not None:
            self.decoder.forward(self.tokens, attn_tokens=self.tokens)
        else:
            bd.bd_block_attention(self.caches[layer].kv, self.ctx_len, self.tokens, q, k_blk,
                                  v_blk, self.attn_out, self.attn_ws, self.max_ctx,
                                  dev_status=self.dev_status)
        self.commit(h, self.n_committed[0] if n_committed_out is None else n_committed_out)

    def append_block(self, k_blk, v_blk):
        """Append the finished block's K/V (every layer's, with a decoder)."""
        if self.decoder is not None:
            self.decoder.forward(self.tokens)
            self.decoder.append(self.n_masked)
        else:
            bd.bd_append_block_kv(self.caches[0].kv, k_blk, v_blk, self.ctx_len, self.n_masked,
                                  self.dev_status)

    def commit(self, h, n_committed_out):
        """The confidence/commit call of one step (greedy or sampled)."""
        if self.thresholds is not None:
            bd.bd_confidence_commit_regions(h, self.W, self.thresholds, self.tokens, self.p_max,
                                            self.argmax, n_committed_out, self.n_masked,
                                            self.conf_ws, dev_status=self.dev_status)
        elif self.temperature is None:
            bd.bd_confidence_commit(h, self.W, self.T, self.tokens, self.p_max, self.argmax,
                                    n_committed_out, self.n_masked, self.conf_ws,
                                    dev_status=self.dev_status)
        elif self.truncated:
            bd.bd_sample_commit_truncated(h, self.W, self.T, self.temperature, self.top_k,
                                          self.top_p, self.seed, self.draw_counter, self.tokens,
                                          self.p_max, self.argmax, n_committed_out,
                                          self.n_masked, self.conf_ws,
                                          dev_status=self.dev_status)
        else:
            bd.bd_sample_commit(h, self.W, self.T, self.temperature, self.seed,
                                self.draw_counter, self.tokens, self.p_max, self.argmax,
                                n_committed_out, self.n_masked, self.conf_ws,
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
            # Python's cyclic garbage collector must not run inside the capture:
            # freeing another object's CUDA graphs or memory there invalidates it
            gc.collect()
            was_enabled = gc.isenabled()
            gc.disable()
            try:
                g = torch.cuda.CUDAGraph()
                n0 = bd.bd_kernel_launches()
                with torch.cuda.graph(g):
                    for s in range(s0, s1):
                        self.step(h_steps[s], q, k_blk, v_blk, self.n_committed[s])
            finally:
                if was_enabled:
                    gc.enable()
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
        self.append_block(k_blk, v_blk)
        return s

    def steps_per_sequence(self) -> np.ndarray:
        """Denoise steps each sequence took in the last block (>= 1 commit each)."""
        return (self.n_committed.cpu().numpy() > 0).sum(axis=0)

    def check_status(self):
        st = int(self.dev_status.item())
        if st == 0 and self.decoder is not None:
            st = int(self.decoder.dev_status.item())
        if st != 0:
            raise bd.BDError("device check", st)


class DecoderStack:
    """The layer stack that feeds the block attention in the long-context
    workload: embedding + RMSNorm, then per layer QKV projection, block
    attention over that layer's paged cache and output projection with the
    residual add (bd_embed_rmsnorm, bd_qkv_projection, bd_block_attention,
    bd_out_projection_residual), and the gated MLP (bd_mlp_residual) for
    layers given as (wqkv, wo, w_gate_up, w_down).  All layers share one page
    table and one ctx_len; a finished block's K/V of every layer is appended
    by one bd_append_block_kv_layers call."""

    def __init__(self, embed: torch.Tensor, mask_embed: torch.Tensor, layers, caches, ctx_len,
                 *, batch: int, block_len: int, num_q_heads: int, max_ctx: int,
                 eps: float = 1e-6):
        self.E, self.e_mask = embed, mask_embed
        self.layers = list(layers)                 # [(wqkv, wo[, w_gate_up, w_down])] bf16
        self.caches = list(caches)                 # [PagedCache] sharing one page table
        assert len(self.layers) == len(self.caches)
        self.ctx_len = ctx_len
        self.B, self.L, self.Hq = batch, block_len, num_q_heads
        c0 = self.caches[0]
        self.Hkv, self.D = c0.k.shape[1], c0.k.shape[3]
        self.H = embed.shape[1]
        self.max_ctx, self.eps = int(max_ctx), float(eps)
        dev = embed.device
        rows = batch * block_len
        nl = len(self.layers)
        self.x = torch.empty(rows, self.H, dtype=torch.float32, device=dev)
        self.xn = torch.empty(rows, self.H, dtype=torch.bfloat16, device=dev)
        self.q = torch.empty(batch, block_len, num_q_heads, self.D, dtype=torch.bfloat16,
                             device=dev)
        self.k = torch.empty(nl, batch, block_len, self.Hkv, self.D, dtype=torch.bfloat16,
                             device=dev)
        self.v = torch.empty_like(self.k)
        self.attn = torch.empty_like(self.q)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        qws = bd.bd_qkv_projection_workspace(rows, self.H, num_q_heads, self.Hkv, self.D)
        ows = bd.bd_out_projection_workspace(rows, num_q_heads * self.D, self.H)
        aws = bd.bd_block_attention_workspace(batch, block_len, num_q_heads, self.Hkv, self.D,
                                              self.max_ctx)
        if qws == 0 or ows == 0:
            raise ValueError("unsupported decoder shape")
        mws = 0
        for lw in self.layers:
            if len(lw) > 2:
                mws = max(mws, bd.bd_mlp_workspace(rows, self.H, lw[3].shape[1]))
                if mws == 0:
                    raise ValueError("unsupported MLP shape")
        self.ws = torch.empty(max(qws, ows, mws, 1), dtype=torch.uint8, device=dev)
        self.attn_ws = torch.empty(max(aws, 1), dtype=torch.uint8, device=dev)
        # every layer addresses its pool through one shared page table
        for c in self.caches[1:]:
            if not np.array_equal(c.page_table_np, c0.page_table_np):
                raise ValueError("decoder layers must share one page table")
        self.kvs = [bd.paged_kv(c.k, c.v, c0.page_table) for c in self.caches]

    def forward(self, tokens, attn_tokens=None):
        """Run the stack over the block whose state is `tokens` [B, L'].
        `attn_tokens` (or None) lets the attention skip finished sequences.
        Leaves x (after the last layer) and every layer's block K/V in
        self.x, self.k, self.v."""
        bd.bd_embed_rmsnorm(tokens, self.E, self.e_mask, self.x, self.xn, self.eps,
                            self.dev_status)
        for l, lw in enumerate(self.layers):
            wqkv, wo = lw[0], lw[1]
            bd.bd_qkv_projection(self.xn, wqkv, self.q, self.k[l], self.v[l], self.ws,
                                 self.dev_status)
            bd.bd_block_attention(self.kvs[l], self.ctx_len, attn_tokens, self.q, self.k[l],
                                  self.v[l], self.attn, self.attn_ws, self.max_ctx,
                                  dev_status=self.dev_status)
            bd.bd_out_projection_residual(self.attn, wo, self.x, self.xn, self.ws, self.eps,
                                          self.dev_status)
            if len(lw) > 2:
                bd.bd_mlp_residual(self.xn, lw[2], lw[3], self.x, self.xn, self.ws, self.eps,
                                   self.dev_status)

    def append(self, n_masked=None):
        """Append the block K/V of the last forward to every layer's cache."""
        bd.bd_append_block_kv_layers(self.kvs, self.k, self.v, self.ctx_len, n_masked,
                                     self.dev_status)
