"""CPU oracle for one denoise step of block-wise masked-diffusion decoding.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, fp64 statement of
what the GPU library computes.  Only the test suite, the package smoke check
and the benchmark's CPU-baseline leg may import it; the product path never
does, and it shares no code with the CUDA sources (it imports numpy only).

Sources (cited by title and section throughout):
  [RS]   "MinerU-Diffusion: Rethinking Document OCR as Inverse Rendering via
         Diffusion Decoding" -- Chinese paper summary (paper.rainbus.top),
         method paragraph: step 2 (block factorisation), step 3 (block-attention
         diffusion decoding), step 4 (confidence-threshold dynamic scheduling),
         step 6 (inference settings); novelty paragraph (KV-cache reuse).
  [HL]   "MinerU-Diffusion reads documents with diffusion decoding instead of
         left to right" (hysenlabs review), section "The idea: OCR as inverse
         rendering" (black = confirmed, red = updating, yellow = masked; the
         block-attention mask of the training figure) and its FAQ.
  [BLOG] the authors' announcement post (gitcode.csdn.net), Fig. 1 and Fig. 2
         captions (same mask, same token states).

Readings where the pages are silent or loose (each one is also listed with the
design notes of this repository):
  R1  "confidence exceeds T" is implemented as p_max >= T.
  R2  when no masked position reaches T, the single masked position with the
      largest p_max is committed; ties go to the lowest position.
  R3  argmax ties go to the lowest token id.
  R4  "top-k=0, temperature=1.0, top-p=1.0" is read as greedy argmax, with the
      confidence taken as the maximum of softmax(logits) at temperature 1.
  R5  committed ("confirmed") tokens are never revised.
  R6  the attention scale is 1/sqrt(D); no rotary embedding (positions play no
      part in the mask); grouped-query heads: query head h reads KV head
      h // (Hq / Hkv).
  R7  all positions of the current block attend to all positions of the block,
      masked or not.

Every function below is pinned by the `-m "not gpu"` tests in tests/ against
closed forms, library routines on special cases, invariants and brute force.
"""
from __future__ import annotations

import numpy as np

MASK = -1


# ---------------------------------------------------------------------------
# (1) Block-attention mask and attention        [RS] step 3; [HL]; [BLOG] Fig. 2
# ---------------------------------------------------------------------------
def block_mask(block_id: np.ndarray) -> np.ndarray:
    """Explicit L x L block-attention mask.

    block_id[j] is the block index of position j (the visual/prompt prefix is
    block 0, the first output block is 1, ...).  Position i may attend to j iff
    j lies in the same block (bidirectional) or an earlier one (causal across
    blocks): mask[i, j] = block_id[j] <= block_id[i].  Later blocks are never
    visible.
    """
    block_id = np.asarray(block_id)
    return block_id[None, :] <= block_id[:, None]


def block_attention(q, k, v, block_id, rows, scale=None):
    """Naive masked attention for the query positions `rows`.

    q [S, Hq, D], k and v [S, Hkv, D] (any float, computed in fp64),
    block_id [S].  Query head h uses KV head h // (Hq // Hkv) (R6).
    Returns out [len(rows), Hq, D] (fp64):
        out[r, h] = softmax_j(q[i,h] . k[j,g] * scale  over mask[i, j]) @ v[:, g]
    with the softmax written out as max-subtract, exp, sum, divide.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    assert Hq % Hkv == 0 and k.shape == (S, Hkv, D) and v.shape == (S, Hkv, D)
    group = Hq // Hkv
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    rows = np.asarray(rows, dtype=np.int64)
    allowed = block_mask(block_id)[rows]                      # [R, S]
    out = np.empty((len(rows), Hq, D), dtype=np.float64)
    for h in range(Hq):
        g = h // group
        s = (q[rows, h, :] @ k[:, g, :].T) * scale             # [R, S]
        s = np.where(allowed, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        p = e / e.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, g, :]
    return out


def current_block_attention(q_blk, k_cache, v_cache, k_blk, v_blk, scale=None):
    """Attention of one sequence's current block against its cache.

    The sequence is laid out as [cached tokens (prefix and finished blocks) |
    current block]; every cached token sits in an earlier block than the
    current one, and no later block exists yet, so block_mask() over that
    layout is the whole rule.  q_blk [L', Hq, D]; k/v_cache [C, Hkv, D];
    k/v_blk [L', Hkv, D].  Returns [L', Hq, D] fp64.
    """
    C, L = k_cache.shape[0], k_blk.shape[0]
    Hq, D = q_blk.shape[1], q_blk.shape[2]
    k = np.concatenate([np.asarray(k_cache, np.float64), np.asarray(k_blk, np.float64)])
    v = np.concatenate([np.asarray(v_cache, np.float64), np.asarray(v_blk, np.float64)])
    q = np.zeros((C + L, Hq, D))
    q[C:] = q_blk
    block_id = np.concatenate([np.zeros(C, np.int64), np.ones(L, np.int64)])
    return block_attention(q, k, v, block_id, np.arange(C, C + L), scale)


# ---------------------------------------------------------------------------
# (2) Vocabulary projection and confidence                [RS] steps 4 and 6
# ---------------------------------------------------------------------------
def confidence(h, W, row_chunk: int = 64):
    """Full-logit softmax confidence for each row of h.

    h [M, H], W [V, H].  logits l = h W^T (fp64).  The softmax is formed
    explicitly, p = exp(l - max l) / sum(exp(l - max l)), and
        p_max  = max_v p_v           (R4)
        argmax = lowest v with l_v == max l   (R3)
    Also returned, for the parity exemptions: the gap between the two largest
    probabilities and between the two largest logits of each row.
    Returns dict of arrays p_max, argmax, top2_prob_margin, top2_logit_gap.
    """
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    M = h.shape[0]
    p_max = np.empty(M)
    argmax = np.empty(M, dtype=np.int64)
    pmarg = np.empty(M)
    lgap = np.empty(M)
    for r0 in range(0, M, row_chunk):
        l = h[r0:r0 + row_chunk] @ W.T                         # [m, V]
        lmax = l.max(axis=1, keepdims=True)
        e = np.exp(l - lmax)
        p = e / e.sum(axis=1, keepdims=True)
        p_max[r0:r0 + row_chunk] = p.max(axis=1)
        argmax[r0:r0 + row_chunk] = np.argmax(l, axis=1)       # first = lowest id
        if l.shape[1] > 1:
            top2 = np.partition(l, -2, axis=1)[:, -2:]          # two largest, ascending
            lgap[r0:r0 + row_chunk] = top2[:, 1] - top2[:, 0]
            ptop2 = np.partition(p, -2, axis=1)[:, -2:]
            pmarg[r0:r0 + row_chunk] = ptop2[:, 1] - ptop2[:, 0]
        else:
            lgap[r0:r0 + row_chunk] = np.inf
            pmarg[r0:r0 + row_chunk] = np.inf
    return {"p_max": p_max, "argmax": argmax,
            "top2_prob_margin": pmarg, "top2_logit_gap": lgap}


# ---------------------------------------------------------------------------
# (3) Confidence-threshold commit              [RS] step 4; [HL] Fig. 1 states
# ---------------------------------------------------------------------------
def commit(tokens, p_max, argmax, threshold):
    """One commit decision per sequence.

    tokens [B, L'] int (MASK = -1 marks still-masked positions); p_max and
    argmax [B, L'] hold the step's confidence for the masked positions (other
    entries are ignored).  `threshold` is one number T, or a [B, L'] array of
    per-position thresholds T[b, i] (region thresholds: the summary's
    weaknesses paragraph proposes local thresholds that follow the region of
    the page; the scalar is the constant array).  For each sequence:
        S = { i masked : p_max[i] >= T[b, i] }                  (R1)
        if S is empty and some position is masked:
            S = { the masked i with the largest p_max, lowest i on ties }  (R2)
        tokens[i] = argmax[i] for i in S; other tokens unchanged   (R5)
    Returns (new tokens, committed mask [B, L'] bool).
    """
    tokens = np.array(tokens, dtype=np.int64, copy=True)
    B, L = tokens.shape
    T = np.broadcast_to(np.asarray(threshold, dtype=np.float64), (B, L))
    chosen = np.zeros((B, L), dtype=bool)
    for b in range(B):
        masked = [i for i in range(L) if tokens[b, i] == MASK]
        sel = [i for i in masked if p_max[b, i] >= T[b, i]]
        if not sel and masked:
            best = masked[0]
            for i in masked[1:]:
                if p_max[b, i] > p_max[b, best]:
                    best = i
            sel = [best]
        for i in sel:
            tokens[b, i] = argmax[b, i]
            chosen[b, i] = True
    return tokens, chosen


def denoise_step(tokens, h, W, threshold):
    """One full step: confidence for the masked rows, then commit.

    tokens [B, L'], h [B, L', H], W [V, H].  Returns (new tokens, p_max [B,L'],
    argmax [B,L'], committed mask [B,L'], confidence dict of the masked rows,
    masked (b, i) index arrays).  p_max / argmax are -1 at rows that were
    already committed before the step.
    """
    tokens = np.asarray(tokens)
    B, L = tokens.shape
    bi, ii = np.nonzero(tokens == MASK)
    p_max = np.full((B, L), -1.0)
    argmax = np.full((B, L), -1, dtype=np.int64)
    conf = None
    if len(bi):
        conf = confidence(np.asarray(h)[bi, ii], W)
        p_max[bi, ii] = conf["p_max"]
        argmax[bi, ii] = conf["argmax"]
    new, chosen = commit(tokens, p_max, argmax, threshold)
    return new, p_max, argmax, chosen, conf, (bi, ii)


def decode_block(h_steps, W, threshold, tokens0=None):
    """Denoise one block until no position is masked.

    h_steps [S, B, L', H] gives the hidden states at each step (step s uses
    h_steps[s]).  Returns (final tokens [B, L'], steps per sequence [B],
    list of per-step token arrays).  A sequence's step count is the number of
    steps it took until none of its positions was masked.
    """
    S, B, L, _ = np.asarray(h_steps).shape
    tokens = np.full((B, L), MASK, np.int64) if tokens0 is None else np.array(tokens0)
    steps = np.zeros(B, dtype=np.int64)
    trace = []
    s = 0
    while (tokens == MASK).any():
        if s >= S:
            raise RuntimeError("block not finished within the supplied steps")
        active = (tokens == MASK).any(axis=1)
        tokens, *_ = denoise_step(tokens, h_steps[s], W, threshold)
        steps += active
        trace.append(tokens.copy())
        s += 1
    return tokens, steps, trace


# ---------------------------------------------------------------------------
# (3b) Sampling reading of the inference settings           [RS] step 6
# ---------------------------------------------------------------------------
# The summary's settings "top-k=0, temperature=1.0, top-p=1.0" are read by
# default as greedy decoding (R4).  Read as sampling instead, they mean: draw
# the token from softmax(l / temperature) with no top-k and no nucleus
# truncation.  The draw uses the Gumbel-max identity: argmax_v (l_v / t + G_v)
# with G_v = -ln(-ln U_v) and U_v uniform on (0, 1) is distributed as
# softmax(l / t).  The confidence of the drawn token is its probability.
# U comes from a counter-based generator so that the GPU and this oracle draw
# the same numbers: Philox-4x64 with 10 rounds (Salmon, Moraes, Dror and Shaw,
# "Parallel random numbers: as easy as 1, 2, 3", SC'11) under the key
# (seed, 0), at counter (v, position // 8, offset, 0).  The block's four 64-bit
# words hold eight 23-bit fields: position p takes word (p // 2) % 4, bits
# 41..63 when p is even and bits 9..31 when p is odd, and U = (field + 1/2) /
# 2^23, exactly representable in fp32.  `offset` is the caller's step counter,
# so every denoise step draws afresh.

_M64 = (1 << 64) - 1
PHILOX_M = (0xD2E7470EE14C6C93, 0xCA5A826395121157)   # round multipliers
PHILOX_W = (0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B)   # Weyl key increments


def _mulhilo64(a, m):
    """High and low 64-bit halves of the 128-bit product a * m (a uint64 array)."""
    a = np.asarray(a, dtype=np.uint64)
    lo32 = np.uint64(0xFFFFFFFF)
    s32 = np.uint64(32)
    a0, a1 = a & lo32, a >> s32
    m0, m1 = np.uint64(m & 0xFFFFFFFF), np.uint64(m >> 32)
    p00, p01, p10, p11 = a0 * m0, a0 * m1, a1 * m0, a1 * m1
    mid = (p00 >> s32) + (p01 & lo32) + (p10 & lo32)
    hi = p11 + (p01 >> s32) + (p10 >> s32) + (mid >> s32)
    lo = (mid << s32) | (p00 & lo32)
    return hi, lo


def philox4x64_10(counter, key):
    """Philox-4x64-10 of a counter (4 uint64 arrays) under a key (2 ints).

    One round: (h0, l0) = M0 * c0, (h1, l1) = M1 * c2 (128-bit products);
    c <- (h1 ^ c1 ^ k0, l1, h0 ^ c3 ^ k1, l0); the key grows by (W0, W1)
    before every round but the first."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) for c in counter)
    k0, k1 = int(key[0]) & _M64, int(key[1]) & _M64
    for r in range(10):
        if r > 0:
            k0 = (k0 + PHILOX_W[0]) & _M64
            k1 = (k1 + PHILOX_W[1]) & _M64
        h0, l0 = _mulhilo64(c0, PHILOX_M[0])
        h1, l1 = _mulhilo64(c2, PHILOX_M[1])
        c0, c1, c2, c3 = h1 ^ c1 ^ np.uint64(k0), l1, h0 ^ c3 ^ np.uint64(k1), l0
    return c0, c1, c2, c3


def uniform01(v, pos, seed, offset=0):
    """U[v, pos] in (0, 1) for vocabulary entry v at position id pos."""
    v, pos = np.broadcast_arrays(np.asarray(v, dtype=np.int64), np.asarray(pos, dtype=np.int64))
    zero = np.zeros(v.shape, dtype=np.uint64)
    words = philox4x64_10((v, pos >> 3, zero + np.uint64(int(offset) & _M64), zero), (seed, 0))
    w = np.choose((pos >> 1) & 3, words)
    field = np.where((pos & 1) == 0, w >> np.uint64(41), (w >> np.uint64(9)) & np.uint64(0x7FFFFF))
    return (field.astype(np.float64) + 0.5) / float(1 << 23)


def sample_confidence(h, W, pos, seed, temperature, offset=0, row_chunk: int = 16):
    """Gumbel-max draw from softmax(h W^T / temperature) for each row of h.

    pos[m] is the position id of row m (b * L' + i).  Returns dict:
      token   = argmax_v (z_v + G_v), z = l / temperature (lowest v on ties)
      p_sel   = softmax(z)[token]
      key_gap = gap between the two largest z_v + G_v (exemption of near ties)
    """
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    pos = np.asarray(pos, dtype=np.int64)
    M, V = h.shape[0], W.shape[0]
    token = np.empty(M, dtype=np.int64)
    p_sel = np.empty(M)
    gap = np.empty(M)
    vs = np.arange(V)
    for r0 in range(0, M, row_chunk):
        z = (h[r0:r0 + row_chunk] @ W.T) / float(temperature)          # [m, V]
        g = -np.log(-np.log(uniform01(vs[None, :], pos[r0:r0 + row_chunk, None], seed, offset)))
        key = z + g
        t = np.argmax(key, axis=1)
        zmax = z.max(axis=1)
        lse = zmax + np.log(np.exp(z - zmax[:, None]).sum(axis=1))
        token[r0:r0 + row_chunk] = t
        p_sel[r0:r0 + row_chunk] = np.exp(z[np.arange(len(t)), t] - lse)
        if V > 1:
            top2 = np.partition(key, -2, axis=1)[:, -2:]
            gap[r0:r0 + row_chunk] = top2[:, 1] - top2[:, 0]
        else:
            gap[r0:r0 + row_chunk] = np.inf
    return {"token": token, "p_sel": p_sel, "key_gap": gap}


# Truncated sampling: the other settings of step 6, top-k and top-p, applied
# in the order samplers usually apply them (temperature, then top-k, then
# top-p on what top-k kept, renormalised).  Each leaves a value threshold:
#   top-k (k > 0, k < V): theta_k = the k-th largest z (entries equal to it
#       are all kept, so ties at the boundary never split);
#   top-p (0 < p < 1): over the kept entries sorted by z descending with
#       masses w = exp(z - max z), the first one at which the running mass
#       reaches p * (total kept mass); theta_p = its z (its ties kept).
# The kept set is {v : z_v >= max(theta_k, theta_p)}; the token is the
# Gumbel-max draw restricted to it (same noise G_v as above) and its
# confidence is its probability under the renormalised kept distribution.
# k = 0 and p = 1 keep everything, which is sample_confidence again.
def truncation_threshold(z, top_k=0, top_p=1.0):
    """Value threshold theta of one row z (fp64): entries with z >= theta are
    kept.  Also returns the top-p mass margin: min(target - mass before the
    boundary group, mass through it - target) / kept mass (inf without top-p)."""
    z = np.asarray(z, dtype=np.float64)
    zs = np.sort(z)[::-1]
    theta = -np.inf
    if 0 < top_k < len(z):
        theta = zs[top_k - 1]
    margin = np.inf
    if top_p < 1.0:
        kept = zs[zs >= theta]
        w = np.exp(kept - kept[0])
        cum = np.cumsum(w)
        target = top_p * cum[-1]
        j = int(np.searchsorted(cum, target, side="left"))
        j = min(j, len(kept) - 1)
        first = int(np.searchsorted(-kept, -kept[j], side="left"))   # start of j's tie group
        last = int(np.searchsorted(-kept, -kept[j], side="right")) - 1
        before = cum[first - 1] if first > 0 else 0.0
        margin = min(target - before, cum[last] - target) / cum[-1]
        theta = max(theta, kept[j])
    return theta, margin


def sample_confidence_truncated(h, W, pos, seed, temperature, top_k=0, top_p=1.0, offset=0,
                                row_chunk: int = 16):
    """Top-k / top-p truncated Gumbel-max draw for each row of h.

    Returns dict: token, p_sel (probability under the renormalised kept
    distribution), key_gap (gap between the two largest perturbed keys among
    the kept entries), theta, p_margin (truncation_threshold's margin) and
    band_mass (kept-mass share of the entries within 1e-3 of theta, the ones
    whose membership a small change of z could flip)."""
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    pos = np.asarray(pos, dtype=np.int64)
    M, V = h.shape[0], W.shape[0]
    out = {k: np.empty(M) for k in ("p_sel", "key_gap", "theta", "p_margin", "band_mass")}
    out["token"] = np.empty(M, dtype=np.int64)
    vs = np.arange(V)
    for r0 in range(0, M, row_chunk):
        z = (h[r0:r0 + row_chunk] @ W.T) / float(temperature)
        g = -np.log(-np.log(uniform01(vs[None, :], pos[r0:r0 + row_chunk, None], seed, offset)))
        for j in range(z.shape[0]):
            r = r0 + j
            theta, margin = truncation_threshold(z[j], top_k, top_p)
            keep = z[j] >= theta
            key = np.where(keep, z[j] + g[j], -np.inf)
            t = int(np.argmax(key))
            m = z[j][keep].max()
            w = np.where(keep, np.exp(z[j] - m), 0.0)
            out["token"][r] = t
            out["p_sel"][r] = w[t] / w.sum()
            kk = np.sort(key[keep])
            out["key_gap"][r] = kk[-1] - kk[-2] if len(kk) > 1 else np.inf
            out["theta"][r] = theta
            out["p_margin"][r] = margin
            band = np.abs(z[j] - theta) < 1e-3
            out["band_mass"][r] = (np.exp(z[j][band] - m).sum() / w.sum()
                                   if np.isfinite(theta) else 0.0)
    return out


def denoise_step_sampled(tokens, h, W, threshold, temperature, seed, offset=0, top_k=0,
                         top_p=1.0):
    """denoise_step with the sampling reading: each masked position draws its
    token (sample_confidence, or sample_confidence_truncated when top_k > 0 or
    top_p < 1; position id b * L' + i) and its confidence is the drawn token's
    probability; the commit rule is unchanged."""
    tokens = np.asarray(tokens)
    B, L = tokens.shape
    bi, ii = np.nonzero(tokens == MASK)
    conf = np.full((B, L), -1.0)
    tok = np.full((B, L), -1, dtype=np.int64)
    res = None
    if len(bi):
        if top_k > 0 or top_p < 1.0:
            res = sample_confidence_truncated(np.asarray(h)[bi, ii], W, bi * L + ii, seed,
                                              temperature, top_k, top_p, offset)
        else:
            res = sample_confidence(np.asarray(h)[bi, ii], W, bi * L + ii, seed, temperature,
                                    offset)
        conf[bi, ii] = res["p_sel"]
        tok[bi, ii] = res["token"]
    new, chosen = commit(tokens, conf, tok, threshold)
    return new, conf, tok, chosen, res, (bi, ii)


# ---------------------------------------------------------------------------
# (4) Paged KV cache: reading and appending          [RS] novelty (KV reuse)
# ---------------------------------------------------------------------------
def paged_read(pool, page_row, length, page_size):
    """Tokens [0, length) of one sequence from a paged pool.

    pool [num_pages, Hkv, page_size, D]; token p lives in physical page
    page_row[p // page_size] at slot p % page_size.  Returns [length, Hkv, D].
    """
    pool = np.asarray(pool)
    out = np.empty((length, pool.shape[1], pool.shape[3]), dtype=pool.dtype)
    for p in range(length):
        out[p] = pool[page_row[p // page_size], :, p % page_size, :]
    return out


def append_block(pool, page_table, ctx_len, blk, done, page_size):
    """Append a finished block's K (or V) to the cache of every done sequence.

    blk [B, L', Hkv, D]; done[b] says whether sequence b's block is fully
    committed.  For such b the block's token i goes to cache position
    ctx_len[b] + i, and ctx_len[b] grows by L'.  Returns (new pool, new ctx_len).
    """
    pool = np.array(pool, copy=True)
    ctx = np.array(ctx_len, dtype=np.int64, copy=True)
    B, L = blk.shape[0], blk.shape[1]
    for b in range(B):
        if not done[b]:
            continue
        for i in range(L):
            p = ctx[b] + i
            pool[page_table[b][p // page_size], :, p % page_size, :] = blk[b, i]
        ctx[b] += L
    return pool, ctx


# ---------------------------------------------------------------------------
# (5) Decoder layer stack                     [RS] reproduction paragraph
# ---------------------------------------------------------------------------
# The summary names the decoder (initialised from SDAR-1.7B-Chat-b32) but
# gives none of its internals.  The plainest reading that the rest supports
# (R10-R13 of the design notes):
#   x0      = E[token] for a confirmed position, e_mask for a masked one
#   layer l: xn = bf16(rms_norm(x));  [q | k | v] = bf16(xn Wqkv_l^T)
#            a  = bf16(block attention of q over layer l's cache and the
#                 block's own k, v)
#            x  = x + a Wo_l^T
# with rms_norm(x) = x / sqrt(mean(x^2) + eps), no learned gain, and no MLP.
# Activations are stored in bf16 between kernels (xn, q, k, v, a); the
# residual stream x is kept at full precision.  bf16() below rounds to the
# nearest bf16 value (ties to even), written out on the fp32 bit pattern.

def round_bf16(x):
    """Nearest bfloat16 value of x (via fp32, ties to even), returned as fp64."""
    f = np.asarray(x, dtype=np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    bits = (bits + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    out = bits.astype(np.uint32).view(np.float32).astype(np.float64)
    return np.where(np.isnan(f), np.nan, out)


def rms_norm(x, eps=1e-6):
    """x / sqrt(mean(x^2) + eps) along the last axis (no gain)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)


def embed(tokens, E, e_mask):
    """Input rows of the decoder: E[token] where confirmed, e_mask where masked.

    tokens [..., L'] int; E [V, H]; e_mask [H].  Returns [..., L', H] fp64."""
    tokens = np.asarray(tokens)
    E = np.asarray(E, dtype=np.float64)
    out = np.empty(tokens.shape + (E.shape[1],))
    masked = tokens == MASK
    out[masked] = np.asarray(e_mask, dtype=np.float64)
    out[~masked] = E[tokens[~masked]]
    return out


def silu(g):
    """g * sigmoid(g)."""
    return g / (1.0 + np.exp(-g))


def mlp_residual(x, w_gate_up, w_down, eps=1e-6):
    """Optional gated MLP after the attention residual (SwiGLU, the MLP of the
    Qwen3 family that SDAR derives from; the pages give no layer internals):
        xn = bf16(RMSNorm(x)); [g | u] = xn W_gu^T (gate rows first)
        a  = bf16(silu(g) * u);  x <- x + a W_down^T
    x [L', H] fp64; w_gate_up [2 I, H]; w_down [H, I]."""
    x = np.asarray(x, dtype=np.float64)
    Wgu = np.asarray(w_gate_up, dtype=np.float64)
    I = Wgu.shape[0] // 2
    xn = round_bf16(rms_norm(x, eps))
    gu = xn @ Wgu.T
    a = round_bf16(silu(gu[:, :I]) * gu[:, I:])
    return x + a @ np.asarray(w_down, dtype=np.float64).T


def decoder_layer(x, wqkv, wo, k_cache, v_cache, num_q_heads, num_kv_heads, eps=1e-6,
                  w_gate_up=None, w_down=None):
    """One layer for one sequence's block.

    x [L', H] (fp64 residual stream); wqkv [(Hq + 2 Hkv) D, H]; wo [H, Hq D];
    k_cache, v_cache [C, Hkv, D] (this layer's cached tokens); optionally the
    MLP weights (mlp_residual).  Returns (new x, k_blk, v_blk) where k_blk,
    v_blk [L', Hkv, D] are the block's keys and values of this layer (bf16
    values, what a finished block appends).
    """
    x = np.asarray(x, dtype=np.float64)
    L = x.shape[0]
    Hq, Hkv = num_q_heads, num_kv_heads
    D = np.asarray(wo).shape[1] // Hq
    xn = round_bf16(rms_norm(x, eps))
    qkv = round_bf16(xn @ np.asarray(wqkv, dtype=np.float64).T)
    q = qkv[:, :Hq * D].reshape(L, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(L, Hkv, D)
    v = qkv[:, (Hq + Hkv) * D:].reshape(L, Hkv, D)
    a = round_bf16(current_block_attention(q, k_cache, v_cache, k, v))
    x = x + a.reshape(L, Hq * D) @ np.asarray(wo, dtype=np.float64).T
    if w_gate_up is not None:
        x = mlp_residual(x, w_gate_up, w_down, eps)
    return x, k, v


def decoder_forward(tokens, E, e_mask, layers, caches, num_q_heads, num_kv_heads, eps=1e-6):
    """The layer stack over one sequence's current block.

    tokens [L']; layers = [(wqkv, wo), ...] or [(wqkv, wo, w_gate_up, w_down),
    ...] with the MLP; caches = [(k_cache, v_cache), ...] per layer.  Returns
    (x after the last layer [L', H], [k_blk per layer], [v_blk per layer])."""
    x = embed(tokens, E, e_mask)
    ks, vs = [], []
    for lw, (kc, vc) in zip(layers, caches):
        x, k, v = decoder_layer(x, lw[0], lw[1], kc, vc, num_q_heads, num_kv_heads, eps,
                                *lw[2:4])
        ks.append(k)
        vs.append(v)
    return x, ks, vs
