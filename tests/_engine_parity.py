"""Harness of the product-loop parity tests: run DenoiseEngine.decode_block
(the loop bench.py times) over successive blocks and check every step of it
against the oracle.

What the engine does beyond one library call at a time: steps run in chunks
of 8 replayed as CUDA graphs (programmatic dependent launches between the
kernels); the host reads the masked count only between chunks, so steps past
the end of a block are issued speculatively and must change nothing; each
sequence's step count comes from the per-step commit counts; a finished
block's K/V is appended, and the next block's attention must read it.

Recording: a wrapper around the engine's step copies the token state, p_max
and argmax after every step into per-step device buffers (the copies are
captured into the same graphs).  A second engine without the wrapper decodes
the same blocks, and its final tokens and step counts must equal the recorded
run's bit for bit, so the recording changes nothing that is compared.

Per block and step, for the checked sequences (lockstep: the oracle starts
every step from the GPU's token state):
  p_max    max-abs 2e-2 for bf16 inputs, 1e-4 for fp32 (the target
           statement), and a relative bound r_row derived below;
  argmax   equal wherever the oracle's top-2 probability margin is >= 1e-3
           (the target statement's exemption), and also wherever its top-2
           logit gap exceeds 2 eps_row (then no fp32 rounding can swap them);
  commits  every position's outcome equal to the oracle's commit rule,
           except where the target statement exempts it (top-2 margin or
           |p_max - T| below 1e-3; the fallback's two best candidates within
           1e-3) AND the bound below cannot decide it;
  no-ops   a step issued after a sequence finished changes none of its
           tokens and counts no commit;
  steps    each sequence's step count equals the number of steps in which it
           still had a masked position; where no exempt divergence was
           adopted, it equals the oracle's own decode from the same start.
Decisions compared outside the exemptions are counted; the tests assert the
counts, so a workload where everything is exempt cannot pass silently.

The bound.  The GPU forms each logit l_v = sum_k h_k W_vk in fp32 from the
same (bf16 or fp32) input values the oracle reads.  With fp32 accumulation of
K terms, |dl_v| <= gamma_K sum_k |h_k W_vk| <= gamma_K |h|_2 |W_v|_2, gamma_K =
K u / (1 - K u), u = 2^-24 (Higham, Accuracy and Stability of Numerical
Algorithms, 2nd ed., section 3.1).  The tensor pipe's internal accumulation
order is not documented, so the bound is doubled:
    eps_row = 2 gamma_K |h_row|_2 max_v |W_v|_2.
p_max = 1 / sum_v exp(l_v - l_max): every logit off by at most eps_row moves
the sum by a factor within exp(+-2 eps_row); the fp32 sum of V positive
terms in any order adds at most (V - 1) u relative; so
    r_row = exp(2 eps_row) - 1 + (V + 3) u.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import os
import weakref

import numpy as np
import torch

import oracle
from block_diffusion_decoding_denoise_gb300 import workload as wl
from block_diffusion_decoding_denoise_gb300.engine import DecoderStack, DenoiseEngine, PagedCache

EXEMPT = 1e-3
U32 = 2.0 ** -24


def torch_dtype(dtype):
    return torch.float32 if dtype == "f32" else torch.bfloat16


def dev(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to("cuda", torch_dtype(dtype))


# ----------------------------------------------------------------------------
# oracle side: memoised confidence of single rows
# ----------------------------------------------------------------------------
class ConfMemo:
    """oracle.confidence of single rows, computed once per (tag, step, b, i):
    a row's planted hidden state does not depend on the threshold or on the
    token state, so runs at several thresholds share the work."""

    def __init__(self, W: np.ndarray):
        self.W64 = np.asarray(W, dtype=np.float64)
        self.V, self.K = W.shape
        self.wmax = float(np.sqrt((self.W64 ** 2).sum(axis=1)).max())
        self.gamma = self.K * U32 / (1.0 - self.K * U32)
        self.memo = {}
        self.threads = max(1, min(16, os.cpu_count() or 1))

    def rows(self, tag, s, h_step: np.ndarray, bi, ii):
        """Confidence of rows (bi, ii) of h_step [B, L, H]: dict of arrays."""
        keys = [(tag, s, int(b), int(i)) for b, i in zip(bi, ii)]
        todo = [j for j, k in enumerate(keys) if k not in self.memo]
        if todo:
            hr = np.asarray(h_step, dtype=np.float64)[np.asarray(bi)[todo], np.asarray(ii)[todo]]
            chunk = 16
            parts = [(j0, hr[j0:j0 + chunk]) for j0 in range(0, len(todo), chunk)]

            def run(part):
                return part[0], oracle.confidence(part[1], self.W64)
            if len(parts) > 1 and self.threads > 1:
                with cf.ThreadPoolExecutor(self.threads) as ex:
                    res = list(ex.map(run, parts))
            else:
                res = [run(p) for p in parts]
            for j0, c in res:
                hn = np.sqrt((hr[j0:j0 + chunk] ** 2).sum(axis=1))
                for r in range(len(c["p_max"])):
                    eps = 2.0 * self.gamma * hn[r] * self.wmax
                    self.memo[keys[todo[j0 + r]]] = (
                        float(c["p_max"][r]), int(c["argmax"][r]),
                        float(c["top2_prob_margin"][r]), float(c["top2_logit_gap"][r]), eps)
        out = np.array([self.memo[k] for k in keys], dtype=np.float64).reshape(-1, 5)
        return {"p_max": out[:, 0], "argmax": out[:, 1].astype(np.int64),
                "margin": out[:, 2], "lgap": out[:, 3], "eps": out[:, 4]}


@dataclasses.dataclass
class Counts:
    rows: int = 0                      # masked rows compared (p_max, argmax)
    argmax_ns: int = 0                 # argmax compared outside the 1e-3 exemption
    argmax_rig: int = 0                # argmax decided by the logit-gap bound
    decisions: int = 0                 # masked positions whose commit outcome was compared
    decisions_ns: int = 0              # ... outside the target statement's exemptions
    decisions_rig: int = 0             # ... decided by the bound
    commits_ns: int = 0                # oracle commits compared outside the exemptions
    adoptions: int = 0                 # exempt divergences adopted (lockstep)
    speculative_steps: int = 0         # steps issued after a sequence had finished
    max_abs_pmax: float = 0.0
    max_rel_pmax: float = 0.0
    max_rel_over_bound: float = 0.0    # max of (relative p_max error / r_row)
    steps_checked: int = 0

    def add(self, o: "Counts"):
        for f in dataclasses.fields(self):
            a, b = getattr(self, f.name), getattr(o, f.name)
            setattr(self, f.name, max(a, b) if f.name.startswith("max_") else a + b)


def _set_determined(p, T, r):
    """True when the commit set of one sequence's masked positions is the same
    for every p' with |p' - p| <= r p (the bound): membership of each position
    in {p >= T} is fixed, and when the set is empty the fallback's choice is
    fixed as well."""
    lo, hi = p * (1.0 - r), p * (1.0 + r)
    if not ((lo >= T) | (hi < T)).all():
        return False
    if (lo >= T).any():
        return True
    j = int(np.argmax(p))
    others = np.arange(len(p)) != j
    return bool((lo[j] > hi[others]).all())


def check_step(w, memo: ConfMemo, tag, s, h_step, before, after, g_p, g_a, ncom_s, T, seqs,
               counts: Counts, abs_tol):
    """Compare one recorded engine step with the oracle's step from the same
    token state, for sequences `seqs`.  Returns the per-sequence flag
    'an exempt divergence was adopted'."""
    B, L = before.shape
    Tm = np.broadcast_to(np.asarray(T, np.float64), (B, L))
    adopted = np.zeros(B, bool)
    # every sequence: commit count and no-op steps
    done = ~(before == -1).any(axis=1)
    assert (after[done] == before[done]).all(), f"step {s}: a finished sequence changed"
    assert (ncom_s[done] == 0).all(), f"step {s}: a finished sequence counted commits"
    counts.speculative_steps += int(done.sum())
    assert np.array_equal(ncom_s, (after != before).sum(axis=1)), f"step {s}: n_committed"
    assert ((after == before) | (before == -1)).all(), f"step {s}: a confirmed token changed"
    for b in seqs:
        m = np.nonzero(before[b] == -1)[0]
        if len(m) == 0:
            continue
        counts.steps_checked += 1
        c = memo.rows(tag, s, h_step, np.full(len(m), b), m)
        po, ao = c["p_max"], c["argmax"]
        eps = c["eps"]
        r = np.expm1(2.0 * eps) + (memo.V + 3) * U32
        gp, ga = g_p[b, m].astype(np.float64), g_a[b, m]
        assert (g_p[b][before[b] != -1] == -1).all() and (g_a[b][before[b] != -1] == -1).all()
        # p_max
        err = np.abs(gp - po)
        rel = err / po
        counts.rows += len(m)
        counts.max_abs_pmax = max(counts.max_abs_pmax, float(err.max()))
        counts.max_rel_pmax = max(counts.max_rel_pmax, float(rel.max()))
        counts.max_rel_over_bound = max(counts.max_rel_over_bound, float((rel / r).max()))
        assert err.max() <= abs_tol, f"step {s} seq {b}: p_max error {err.max()} > {abs_tol}"
        assert (rel <= r).all(), (f"step {s} seq {b}: relative p_max error {rel.max():.3e} "
                                  f"above its bound {r[np.argmax(rel / r)]:.3e}")
        # argmax
        am_ns = c["margin"] >= EXEMPT
        am_rig = c["lgap"] > 2.0 * eps
        counts.argmax_ns += int(am_ns.sum())
        counts.argmax_rig += int(am_rig.sum())
        bad = (ga != ao) & (am_ns | am_rig)
        assert not bad.any(), (f"step {s} seq {b}: argmax differs at decided rows "
                               f"{m[bad].tolist()} (gpu {ga[bad].tolist()}, "
                               f"oracle {ao[bad].tolist()})")
        # commit decisions
        pfull = np.full(L, -1.0)
        afull = np.full(L, -1, np.int64)
        pfull[m], afull[m] = po, ao
        exp_tok, _ = oracle.commit(before[b:b + 1], pfull[None], afull[None], Tm[b:b + 1])
        exp_tok = exp_tok[0]
        ex_ns = np.zeros(L, bool)
        ex_ns[m] = (c["margin"] < EXEMPT) | (np.abs(po - Tm[b, m]) < EXEMPT)
        if not (po >= Tm[b, m]).any() and len(m) > 1:
            ps = np.sort(po)
            if ps[-1] - ps[-2] < EXEMPT:
                ex_ns[m] |= po > ps[-1] - EXEMPT
        set_det = _set_determined(po, Tm[b, m], r)
        tok_det = np.zeros(L, bool)
        tok_det[m] = c["lgap"] > 2.0 * eps
        counts.decisions += len(m)
        counts.decisions_ns += int((~ex_ns[m]).sum())
        counts.decisions_rig += len(m) if set_det else 0
        counts.commits_ns += int(((exp_tok[m] != -1) & ~ex_ns[m]).sum())
        diff = after[b] != exp_tok
        for i in np.nonzero(diff)[0]:
            both = after[b][i] != -1 and exp_tok[i] != -1
            rig = tok_det[i] if both else set_det
            assert ex_ns[i] and not rig, (
                f"step {s} seq {b} position {i}: gpu {after[b][i]}, oracle {exp_tok[i]} "
                f"(p_max {pfull[i]:.6g}, T {Tm[b, i]}, margin {c['margin'][list(m).index(i)]:.3g})")
        if diff.any():
            adopted[b] = True
            counts.adoptions += 1
    return adopted


# ----------------------------------------------------------------------------
# GPU side: engines
# ----------------------------------------------------------------------------
class Recorder:
    """Wraps an engine's step to copy tokens, p_max and argmax after every step
    into per-step buffers (also inside graph capture); for a decoder engine it
    also keeps the final residual stream of step 0."""

    def __init__(self, eng: DenoiseEngine):
        self._eng = weakref.ref(eng)               # no reference cycle through eng.step
        L, B = eng.L, eng.B
        self.tok = torch.full((L, B, L), -2, dtype=torch.int32, device="cuda")
        self.p = torch.zeros(L, B, L, dtype=torch.float32, device="cuda")
        self.a = torch.zeros(L, B, L, dtype=torch.int32, device="cuda")
        self.x0 = None
        if eng.decoder is not None:
            self.x0 = torch.zeros_like(eng.decoder.x)
        self.stride = eng.n_committed.stride(0) * eng.n_committed.element_size()
        eng.step = self.step

    def step(self, h, q, k, v, ncom=None, layer=0):
        e = self._eng()
        s = (ncom.data_ptr() - e.n_committed.data_ptr()) // self.stride
        DenoiseEngine.step(e, h, q, k, v, ncom, layer)
        self.tok[s].copy_(e.tokens)
        self.p[s].copy_(e.p_max)
        self.a[s].copy_(e.argmax)
        if s == 0 and self.x0 is not None:
            self.x0.copy_(e.decoder.x)

    def reset(self):
        self.tok.fill_(-2)


@dataclasses.dataclass
class BlockRecord:
    issued: int
    tok: np.ndarray       # [issued, B, L]
    p: np.ndarray
    a: np.ndarray
    ncom: np.ndarray      # [L + 1, B]
    steps: np.ndarray     # [B]
    final: np.ndarray     # [B, L]
    attn: np.ndarray | None
    ctx: np.ndarray
    x0: np.ndarray | None = None
    x_app: np.ndarray | None = None
    k_app: np.ndarray | None = None
    v_app: np.ndarray | None = None


def single_layer_setup(w, nblk, seed=0):
    """Paged cache with every sequence's prefix, room for nblk blocks."""
    plen = wl.prefix_lengths(w, seed)
    cap = plen + nblk * w.block_len
    table, npg = wl.page_tables(w, cap, seed)
    cache = PagedCache(npg, w.num_kv_heads, w.head_dim, torch_dtype(w.dtype), table)
    pre = []
    for b in range(w.batch):
        k, v = wl.prefix_kv(w, b, int(plen[b]), seed)
        cache.load_prefix(b, torch.from_numpy(k), torch.from_numpy(v))
        pre.append((k, v))
    return plen, cap, cache, pre


def run_blocks(eng: DenoiseEngine, blocks, ctx0, rec: Recorder | None, graphs=True,
               check_every=8):
    """Decode the blocks in order through eng.decode_block; returns one
    BlockRecord per block."""
    eng.ctx_len.copy_(ctx0)
    out = []
    for (h, q, k, v) in blocks:
        if rec is not None:
            rec.reset()
        issued = eng.decode_block(h, q, k, v, check_every=check_every, graphs=graphs)
        torch.cuda.synchronize()
        eng.check_status()
        r = BlockRecord(issued=issued, tok=None, p=None, a=None,
                        ncom=eng.n_committed.cpu().numpy(), steps=eng.steps_per_sequence(),
                        final=eng.tokens.cpu().numpy().astype(np.int64),
                        attn=eng.attn_out.float().cpu().numpy() if eng.decoder is None else None,
                        ctx=eng.ctx_len.cpu().numpy())
        if rec is not None:
            r.tok = rec.tok[:issued].cpu().numpy().astype(np.int64)
            r.p = rec.p[:issued].cpu().numpy()
            r.a = rec.a[:issued].cpu().numpy().astype(np.int64)
            assert (r.tok >= -1).all(), "a recorded step did not run"
            if rec.x0 is not None:
                r.x0 = rec.x0.cpu().numpy()
        if eng.decoder is not None:
            d = eng.decoder
            r.x_app = d.x.cpu().numpy()
            r.k_app = d.k.float().cpu().numpy()
            r.v_app = d.v.float().cpu().numpy()
        out.append(r)
    return out


def check_block(w, memo, tag, h_steps, rec: BlockRecord, T, seqs, counts: Counts):
    """Every recorded step of one block against the oracle (lockstep), plus the
    step counts.  Returns the sequences where an exempt divergence was adopted."""
    B, L = w.batch, w.block_len
    abs_tol = 1e-4 if w.dtype == "f32" else 2e-2
    before = np.full((B, L), -1, np.int64)
    active_steps = np.zeros(B, np.int64)
    adopted = np.zeros(B, bool)
    for s in range(rec.issued):
        active_steps += (before == -1).any(axis=1)
        adopted |= check_step(w, memo, tag, s, h_steps[s], before, rec.tok[s], rec.p[s],
                              rec.a[s], rec.ncom[s], T, seqs, counts, abs_tol)
        before = rec.tok[s]
    assert not (before == -1).any(), "the block did not finish"
    assert np.array_equal(before, rec.final)
    assert np.array_equal(rec.steps, active_steps), (rec.steps, active_steps)
    assert (rec.ncom[rec.issued:] == 0).all()
    # with no adopted divergence the trajectory is the oracle's own decode
    plain = [b for b in seqs if not adopted[b]]
    for b in plain:
        o_tok, o_steps = oracle_decode_seq(memo, tag, h_steps, b, T, L)
        assert np.array_equal(o_tok, rec.final[b]), f"seq {b}: final tokens differ from the oracle"
        assert o_steps == rec.steps[b], f"seq {b}: {rec.steps[b]} steps, oracle {o_steps}"
    return adopted


def oracle_decode_seq(memo, tag, h_steps, b, T, L):
    """The oracle's own decode of sequence b from an all-masked block (through
    the memo, so rows computed during the lockstep comparison are reused)."""
    tok = np.full((1, L), -1, np.int64)
    Tb = np.broadcast_to(np.asarray(T, np.float64), (h_steps.shape[1], L))[b:b + 1]
    s = 0
    while (tok == -1).any():
        m = np.nonzero(tok[0] == -1)[0]
        c = memo.rows(tag, s, h_steps[s], np.full(len(m), b), m)
        p = np.full((1, L), -1.0)
        a = np.full((1, L), -1, np.int64)
        p[0, m], a[0, m] = c["p_max"], c["argmax"]
        tok, _ = oracle.commit(tok, p, a, Tb)
        s += 1
    return tok[0], s
