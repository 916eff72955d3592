"""Shared helpers of the GPU parity tests: feed one seeded workload to the CUDA
library (through the C ABI) and to the CPU oracle, and compare.

Tolerances:
  attention outputs and p_max: max-abs 1e-4 for fp32 inputs, 2e-2 for bf16
  inputs (bf16 outputs carry a rounding error of up to 2^-9 relative).
  token ids and step counts: bit-exact, except at positions where the
  oracle's top-2 probability margin or |p_max - T| is below 1e-3 (and, for
  the fallback's choice of position, where the two most confident masked
  positions differ by less than 1e-3).  Exempt positions are counted; on an
  exempt divergence the comparison continues from the GPU's tokens
  (lockstep), so later steps stay comparable.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
from block_diffusion_decoding_denoise_gb300 import bd
from block_diffusion_decoding_denoise_gb300 import workload as wl
from block_diffusion_decoding_denoise_gb300.engine import PagedCache

EXEMPT = 1e-3


def tol_for(dtype: str) -> float:
    return 1e-4 if dtype == "f32" else 2e-2


def torch_dtype(dtype: str):
    return torch.float32 if dtype == "f32" else torch.bfloat16


def dev(x: np.ndarray, dtype: str):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda", torch_dtype(dtype))


@dataclasses.dataclass
class Setup:
    w: wl.Workload
    plen: np.ndarray
    k_pre: list
    v_pre: list
    cache: PagedCache
    ctx_len: torch.Tensor
    max_ctx: int


def make_cache(w: wl.Workload, seed=0, plen=None, extra_blocks=1) -> Setup:
    plen = wl.prefix_lengths(w, seed) if plen is None else np.asarray(plen, np.int32)
    cap = plen + w.block_len * extra_blocks
    table, npg = wl.page_tables(w, cap, seed)
    cache = PagedCache(max(npg, 1), w.num_kv_heads, w.head_dim, torch_dtype(w.dtype), table)
    ks, vs = [], []
    for b in range(w.batch):
        k, v = wl.prefix_kv(w, b, int(plen[b]), seed)
        ks.append(k)
        vs.append(v)
        cache.load_prefix(b, torch.from_numpy(k), torch.from_numpy(v))
    ctx = torch.from_numpy(plen.astype(np.int32)).cuda()
    return Setup(w, plen, ks, vs, cache, ctx, int(cap.max()))


def gpu_attention(s: Setup, q, k_blk, v_blk, tokens=None):
    w = s.w
    out = torch.full((w.batch, w.block_len, w.num_q_heads, w.head_dim), float("nan"),
                     dtype=torch_dtype(w.dtype), device="cuda")
    nws = bd.bd_block_attention_workspace(w.batch, w.block_len, w.num_q_heads, w.num_kv_heads,
                                          w.head_dim, s.max_ctx)
    ws = torch.zeros(max(nws, 1), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.bd_block_attention(s.cache.kv, s.ctx_len, tokens, dev(q, w.dtype), dev(k_blk, w.dtype),
                          dev(v_blk, w.dtype), out, ws, s.max_ctx, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out.float().cpu().numpy()


def oracle_attention(s: Setup, b, q, k_blk, v_blk):
    return oracle.current_block_attention(q[b], s.k_pre[b], s.v_pre[b], k_blk[b], v_blk[b])


@dataclasses.dataclass
class StepStats:
    steps_gpu: np.ndarray
    steps_oracle: np.ndarray
    final_gpu: np.ndarray
    final_oracle: np.ndarray
    exempt_positions: int = 0
    lockstep_adoptions: int = 0
    max_pmax_err: float = 0.0
    max_rel_pmax_err: float = 0.0
    argmax_compared: int = 0
    argmax_mismatch_nonexempt: int = 0
    commit_mismatch_nonexempt: int = 0
    rows_checked: int = 0


class ConfRunner:
    """Runs bd_confidence_commit step by step on device buffers."""

    def __init__(self, w: wl.Workload, W: np.ndarray, threshold):
        """`threshold`: a number (bd_confidence_commit) or a [B, L'] array of
        per-position thresholds (bd_confidence_commit_regions)."""
        self.w, self.T = w, threshold
        self.W = dev(W, w.dtype)
        B, L = w.batch, w.block_len
        self.T_dev = None
        if np.ndim(threshold) > 0:
            self.T_dev = torch.from_numpy(np.asarray(threshold, np.float32).copy()).cuda()
        code = bd.BD_F32 if w.dtype == "f32" else bd.BD_BF16
        n = bd.bd_confidence_commit_workspace(code, B, L, w.hidden, w.vocab)
        assert n > 0
        self.ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        self.tokens = torch.full((B, L), -1, dtype=torch.int32, device="cuda")
        self.p_max = torch.empty(B, L, dtype=torch.float32, device="cuda")
        self.argmax = torch.empty(B, L, dtype=torch.int32, device="cuda")
        self.ncom = torch.empty(B, dtype=torch.int32, device="cuda")
        self.nmask = torch.empty(B, dtype=torch.int32, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def set_tokens(self, tokens: np.ndarray):
        self.tokens.copy_(torch.from_numpy(tokens.astype(np.int32)))

    def step(self, h_dev):
        if self.T_dev is not None:
            bd.bd_confidence_commit_regions(h_dev, self.W, self.T_dev, self.tokens, self.p_max,
                                            self.argmax, self.ncom, self.nmask, self.ws,
                                            dev_status=self.status)
        else:
            bd.bd_confidence_commit(h_dev, self.W, self.T, self.tokens, self.p_max, self.argmax,
                                    self.ncom, self.nmask, self.ws, dev_status=self.status)
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0, bd.STATUS.get(int(self.status.item()))
        return (self.tokens.cpu().numpy().astype(np.int64), self.p_max.cpu().numpy(),
                self.argmax.cpu().numpy().astype(np.int64), self.ncom.cpu().numpy(),
                self.nmask.cpu().numpy())


def lockstep_block(w: wl.Workload, W: np.ndarray, h_steps: np.ndarray, threshold,
                   tokens0: np.ndarray | None = None, check_oracle_full: bool = True):
    """Denoise one block on the GPU and compare every step with the oracle.
    `threshold` is a number or a [B, L'] array of per-position thresholds."""
    B, L = w.batch, w.block_len
    T = np.broadcast_to(np.asarray(threshold, np.float64), (B, L))
    tol = tol_for(w.dtype)
    run = ConfRunner(w, W, threshold)
    tokens = np.full((B, L), -1, np.int64) if tokens0 is None else tokens0.astype(np.int64)
    run.set_tokens(tokens)
    Wd = W.astype(np.float64)
    wmax = float(np.sqrt((Wd ** 2).sum(axis=1)).max())
    steps_gpu = np.zeros(B, np.int64)
    stats = StepStats(steps_gpu, None, None, None)
    s = 0
    while (tokens == -1).any():
        assert s < h_steps.shape[0], "block did not finish"
        active = (tokens == -1).any(axis=1)
        h_dev = dev(h_steps[s], w.dtype)
        g_tok, g_p, g_a, g_nc, g_nm = run.step(h_dev)
        exp_tok, o_p, o_a, chosen, conf, (bi, ii) = oracle.denoise_step(
            tokens, h_steps[s].astype(np.float64), Wd, threshold)
        # confidence of the masked rows
        stats.rows_checked += len(bi)
        err = np.abs(g_p[bi, ii] - o_p[bi, ii])
        stats.max_pmax_err = max(stats.max_pmax_err, float(err.max()))
        assert err.max() <= tol, f"p_max error {err.max()} > {tol} at step {s}"
        # relative bound of fp32 logits (tests/_engine_parity.py states it)
        K = Wd.shape[1]
        gam = K * 2.0 ** -24 / (1 - K * 2.0 ** -24)
        eps = 2 * gam * np.sqrt((h_steps[s][bi, ii].astype(np.float64) ** 2).sum(axis=1)) * wmax
        rel = err / o_p[bi, ii]
        stats.max_rel_pmax_err = max(stats.max_rel_pmax_err, float(rel.max()))
        assert (rel <= np.expm1(2 * eps) + (Wd.shape[0] + 3) * 2.0 ** -24).all(), \
            f"relative p_max error {rel.max():.3e} above its bound at step {s}"
        unmasked = tokens != -1
        assert (g_p[unmasked] == -1).all() and (g_a[unmasked] == -1).all()
        margin = conf["top2_prob_margin"]
        near_t = np.abs(conf["p_max"] - T[bi, ii]) < EXEMPT
        am_exempt = margin < EXEMPT
        bad_am = (g_a[bi, ii] != o_a[bi, ii]) & ~am_exempt
        stats.argmax_compared += int((~am_exempt).sum())
        stats.argmax_mismatch_nonexempt += int(bad_am.sum())
        assert not bad_am.any(), f"argmax mismatch at non-exempt rows, step {s}"
        # commit decisions
        exempt_pos = np.zeros((B, L), bool)
        exempt_pos[bi, ii] = am_exempt | near_t
        for b in range(B):                                   # fallback near-ties
            mb = tokens[b] == -1
            if mb.any() and not (o_p[b][mb] >= T[b][mb]).any() and mb.sum() > 1:
                ps = np.sort(o_p[b][mb])
                if ps[-1] - ps[-2] < EXEMPT:
                    exempt_pos[b] |= mb & (o_p[b] > ps[-1] - EXEMPT)
        diff = g_tok != exp_tok
        stats.exempt_positions += int((diff & exempt_pos).sum())
        bad = diff & ~exempt_pos
        stats.commit_mismatch_nonexempt += int(bad.sum())
        assert not bad.any(), f"commit mismatch at non-exempt positions, step {s}: {np.argwhere(bad)}"
        if diff.any():
            stats.lockstep_adoptions += 1
        # bookkeeping outputs
        assert np.array_equal(g_nc, (g_tok != tokens).sum(axis=1))
        assert np.array_equal(g_nm, (g_tok == -1).sum(axis=1))
        assert ((g_nc >= 1) | ~active).all()
        steps_gpu += active
        tokens = g_tok
        s += 1
    stats.final_gpu = tokens
    stats.steps_gpu = steps_gpu
    if check_oracle_full:
        o_tok, o_steps, _ = oracle.decode_block(h_steps.astype(np.float64), Wd, threshold,
                                                 tokens0)
        stats.final_oracle, stats.steps_oracle = o_tok, o_steps
        if stats.exempt_positions == 0:
            assert np.array_equal(o_tok, tokens)
            assert np.array_equal(o_steps, steps_gpu)
    return stats


class SampleRunner:
    """Runs bd_sample_commit step by step on device buffers."""

    def __init__(self, w: wl.Workload, W: np.ndarray, threshold: float, temperature: float,
                 seed: int, top_k: int = 0, top_p: float = 1.0):
        """top_k > 0 or top_p < 1: bd_sample_commit_truncated."""
        self.w, self.T, self.temp, self.seed = w, threshold, temperature, seed
        self.top_k, self.top_p = top_k, top_p
        self.truncated = top_k > 0 or top_p < 1.0
        self.W = dev(W, w.dtype)
        B, L = w.batch, w.block_len
        code = bd.BD_F32 if w.dtype == "f32" else bd.BD_BF16
        query = (bd.bd_sample_commit_truncated_workspace if self.truncated
                 else bd.bd_sample_commit_workspace)
        n = query(code, B, L, w.hidden, w.vocab)
        assert n > 0
        self.ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        self.tokens = torch.full((B, L), -1, dtype=torch.int32, device="cuda")
        self.p_sel = torch.empty(B, L, dtype=torch.float32, device="cuda")
        self.sampled = torch.empty(B, L, dtype=torch.int32, device="cuda")
        self.ncom = torch.empty(B, dtype=torch.int32, device="cuda")
        self.nmask = torch.empty(B, dtype=torch.int32, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.offset = torch.zeros(1, dtype=torch.int64, device="cuda")

    def set_tokens(self, tokens: np.ndarray):
        self.tokens.copy_(torch.from_numpy(tokens.astype(np.int32)))

    def step(self, h_dev, offset: int | None = None):
        """One call; `offset` sets the device draw counter first (None: keep it)."""
        if offset is not None:
            self.offset.fill_(offset)
        before = int(self.offset.item())
        if self.truncated:
            bd.bd_sample_commit_truncated(h_dev, self.W, self.T, self.temp, self.top_k,
                                          self.top_p, self.seed, self.offset, self.tokens,
                                          self.p_sel, self.sampled, self.ncom, self.nmask,
                                          self.ws, dev_status=self.status)
        else:
            bd.bd_sample_commit(h_dev, self.W, self.T, self.temp, self.seed, self.offset,
                                self.tokens, self.p_sel, self.sampled, self.ncom, self.nmask,
                                self.ws, dev_status=self.status)
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0, bd.STATUS.get(int(self.status.item()))
        assert int(self.offset.item()) == before + 1      # the call advanced the counter
        return (self.tokens.cpu().numpy().astype(np.int64), self.p_sel.cpu().numpy(),
                self.sampled.cpu().numpy().astype(np.int64), self.ncom.cpu().numpy(),
                self.nmask.cpu().numpy())


def lockstep_sampled_block(w: wl.Workload, W: np.ndarray, h_steps: np.ndarray, threshold: float,
                           temperature: float, seed: int, tokens0: np.ndarray | None = None,
                           max_steps: int | None = None, top_k: int = 0, top_p: float = 1.0):
    """Sampled denoising of one block (offset = step index) on the GPU, every
    step compared with the oracle's sampled step on the same token state.

    Exemptions: a drawn token may differ where the oracle's two best
    perturbed keys are within 1e-3; a commit decision may differ there, where
    |p_sel - T| < 1e-3, or where the fallback's two best candidates are
    within 1e-3.  With truncation, also where either drawn token lies within
    1e-3 of the oracle's threshold theta (its membership of the kept set can
    flip with the GPU's fp32 logits), and the row's p_sel where the entries
    within 1e-3 of theta hold 1e-3 of the kept mass or more, or where the
    top-p running mass passes p within 1e-3.  The comparison then continues
    from the GPU's tokens."""
    B, L = w.batch, w.block_len
    T = np.broadcast_to(np.asarray(threshold, np.float64), (B, L))
    tol = tol_for(w.dtype)
    truncated = top_k > 0 or top_p < 1.0
    run = SampleRunner(w, W, threshold, temperature, seed, top_k, top_p)
    tokens = np.full((B, L), -1, np.int64) if tokens0 is None else tokens0.astype(np.int64)
    run.set_tokens(tokens)
    Wd = W.astype(np.float64)
    stats = StepStats(np.zeros(B, np.int64), None, None, None)
    s = 0
    while (tokens == -1).any() and (max_steps is None or s < max_steps):
        assert s < h_steps.shape[0], "block did not finish"
        active = (tokens == -1).any(axis=1)
        g_tok, g_p, g_s, g_nc, g_nm = run.step(dev(h_steps[s], w.dtype), offset=s)
        exp_tok, o_p, o_s, chosen, res, (bi, ii) = oracle.denoise_step_sampled(
            tokens, h_steps[s].astype(np.float64), Wd, threshold, temperature, seed, s,
            top_k=top_k, top_p=top_p)
        stats.rows_checked += len(bi)
        unmasked = tokens != -1
        assert (g_p[unmasked] == -1).all() and (g_s[unmasked] == -1).all()
        key_exempt = res["key_gap"] < EXEMPT
        p_exempt = np.zeros(len(bi), bool)
        if truncated:
            hr = h_steps[s][bi, ii].astype(np.float64)
            z_g = (hr * Wd[g_s[bi, ii]]).sum(axis=1) / temperature
            z_o = (hr * Wd[o_s[bi, ii]]).sum(axis=1) / temperature
            th = res["theta"]
            band_tok = (np.abs(z_g - th) < EXEMPT) | (np.abs(z_o - th) < EXEMPT)
            p_exempt = (res["band_mass"] >= EXEMPT) | (res["p_margin"] < EXEMPT)
            key_exempt = key_exempt | band_tok | p_exempt
        same = g_s[bi, ii] == o_s[bi, ii]
        bad = ~same & ~key_exempt
        stats.argmax_mismatch_nonexempt += int(bad.sum())
        assert not bad.any(), f"sampled token mismatch at non-exempt rows, step {s}"
        err = np.abs(g_p[bi, ii] - o_p[bi, ii])[same & ~p_exempt]
        if err.size:
            stats.max_pmax_err = max(stats.max_pmax_err, float(err.max()))
            assert err.max() <= tol, f"p_sel error {err.max()} > {tol} at step {s}"
        exempt_pos = np.zeros((B, L), bool)
        exempt_pos[bi, ii] = key_exempt | (np.abs(o_p[bi, ii] - T[bi, ii]) < EXEMPT)
        for b in range(B):
            mb = tokens[b] == -1
            if mb.any() and not (o_p[b][mb] >= T[b][mb]).any() and mb.sum() > 1:
                ps = np.sort(o_p[b][mb])
                if ps[-1] - ps[-2] < EXEMPT:
                    exempt_pos[b] |= mb & (o_p[b] > ps[-1] - EXEMPT)
        diff = g_tok != exp_tok
        stats.exempt_positions += int((diff & exempt_pos).sum())
        bad = diff & ~exempt_pos
        stats.commit_mismatch_nonexempt += int(bad.sum())
        assert not bad.any(), f"commit mismatch at non-exempt positions, step {s}: {np.argwhere(bad)}"
        if diff.any():
            stats.lockstep_adoptions += 1
        assert np.array_equal(g_nc, (g_tok != tokens).sum(axis=1))
        assert np.array_equal(g_nm, (g_tok == -1).sum(axis=1))
        assert ((g_nc >= 1) | ~active).all()
        stats.steps_gpu += active
        tokens = g_tok
        s += 1
    stats.final_gpu = tokens
    return stats
