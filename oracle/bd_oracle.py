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
    entries are ignored).  For each sequence:
        S = { i masked : p_max[i] >= T }                        (R1)
        if S is empty and some position is masked:
            S = { the masked i with the largest p_max, lowest i on ties }  (R2)
        tokens[i] = argmax[i] for i in S; other tokens unchanged   (R5)
    Returns (new tokens, committed mask [B, L'] bool).
    """
    tokens = np.array(tokens, dtype=np.int64, copy=True)
    B, L = tokens.shape
    chosen = np.zeros((B, L), dtype=bool)
    for b in range(B):
        masked = [i for i in range(L) if tokens[b, i] == MASK]
        sel = [i for i in masked if p_max[b, i] >= threshold]
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
