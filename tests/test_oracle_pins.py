"""Pins of the CPU oracle to facts fixed outside it.

Each test ties one oracle function to something other than itself: a library
routine on a special case the block mask reduces to, a closed form, an
invariant the pages state, or a hand-worked example (tests/golden/).
Sources: "Rethinking Document OCR as Inverse Rendering via Diffusion Decoding"
(paper.rainbus.top summary), method steps 3-4 and the novelty paragraph;
"MinerU-Diffusion reads documents with diffusion decoding instead of left to
right", section "The idea: OCR as inverse rendering".
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _sdpa(q, k, v, mask=None, causal=False):
    """torch's fp64 CPU scaled_dot_product_attention on [S, H, D] inputs."""
    group = q.shape[1] // k.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).repeat_interleave(group, dim=1).permute(1, 0, 2)
    vt = torch.from_numpy(v).repeat_interleave(group, dim=1).permute(1, 0, 2)
    m = None if mask is None else torch.from_numpy(mask)
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, is_causal=causal)
    return o.permute(1, 0, 2).numpy()


def _qkv(rng, S, Hq, Hkv, D):
    return (rng.standard_normal((S, Hq, D)), rng.standard_normal((S, Hkv, D)),
            rng.standard_normal((S, Hkv, D)))


# --- attention ------------------------------------------------------------
def test_block_size_one_is_causal_attention():
    # one token per block: the mask is lower-triangular, i.e. AR decoding
    rng = np.random.default_rng(1)
    q, k, v = _qkv(rng, 13, 4, 2, 8)
    got = oracle.block_attention(q, k, v, np.arange(13), np.arange(13))
    np.testing.assert_allclose(got, _sdpa(q, k, v, causal=True), rtol=1e-12, atol=1e-12)


def test_single_block_is_full_bidirectional_attention():
    rng = np.random.default_rng(2)
    q, k, v = _qkv(rng, 11, 6, 3, 5)
    got = oracle.block_attention(q, k, v, np.zeros(11, int), np.arange(11))
    np.testing.assert_allclose(got, _sdpa(q, k, v), rtol=1e-12, atol=1e-12)


def test_prefix_and_blocks_match_boundary_mask():
    # mask built a second way: i sees j iff j < end of i's block
    rng = np.random.default_rng(3)
    P, L, nb = 5, 3, 3
    S = P + L * nb
    q, k, v = _qkv(rng, S, 4, 1, 6)
    block_id = np.array([0] * P + [1 + (j - P) // L for j in range(P, S)])
    end = np.array([P if i < P else P + L * ((i - P) // L + 1) for i in range(S)])
    mask = np.arange(S)[None, :] < end[:, None]
    got = oracle.block_attention(q, k, v, block_id, np.arange(S))
    np.testing.assert_allclose(got, _sdpa(q, k, v, mask=mask), rtol=1e-12, atol=1e-12)


def test_zero_query_averages_exactly_the_visible_values():
    # q = 0 makes the softmax uniform over the visible keys, so each output is
    # the mean of v over the visible set; v_j = 2^j identifies that set.
    P, L, nb = 3, 2, 3
    S = P + L * nb
    block_id = np.array([0] * P + [1 + (j - P) // L for j in range(P, S)])
    q = np.zeros((S, 1, 1))
    k = np.random.default_rng(4).standard_normal((S, 1, 1))
    v = (2.0 ** np.arange(S)).reshape(S, 1, 1)
    got = oracle.block_attention(q, k, v, block_id, np.arange(S))[:, 0, 0]
    for i in range(S):
        last = P - 1 if i < P else P + L * ((i - P) // L + 1) - 1
        visible = 2.0 ** np.arange(last + 1)
        assert got[i] == pytest.approx(visible.mean(), rel=1e-14)


def test_future_blocks_do_not_change_outputs():
    rng = np.random.default_rng(5)
    P, L, nb = 4, 4, 3
    S = P + L * nb
    q, k, v = _qkv(rng, S, 4, 2, 8)
    block_id = np.array([0] * P + [1 + (j - P) // L for j in range(P, S)])
    rows = np.arange(P + L, P + 2 * L)                      # block 2
    ref = oracle.block_attention(q, k, v, block_id, rows)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    fut = slice(P + 2 * L, S)                               # block 3
    q2[fut] = rng.standard_normal(q2[fut].shape) * 50
    k2[fut] = rng.standard_normal(k2[fut].shape) * 50
    v2[fut] = rng.standard_normal(v2[fut].shape) * 50
    got = oracle.block_attention(q2, k2, v2, block_id, rows)
    assert np.array_equal(got, ref)


def test_current_block_attention_is_block_attention_over_cache():
    rng = np.random.default_rng(6)
    C, L = 7, 4
    q, k, v = _qkv(rng, C + L, 4, 2, 8)
    got = oracle.current_block_attention(q[C:], k[:C], v[:C], k[C:], v[C:])
    block_id = np.array([0] * C + [1] * L)
    mask = block_id[None, :] <= block_id[:, None]
    ref = _sdpa(q, k, v, mask=mask)[C:]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


# --- confidence -----------------------------------------------------------
def test_two_word_vocab_closed_form():
    x = np.array([-7.0, -0.3, 0.0, 0.25, 4.0])
    h = x[:, None]
    W = np.array([[0.0], [1.0]])
    c = oracle.confidence(h, W)
    np.testing.assert_allclose(c["p_max"], 1.0 / (1.0 + np.exp(-np.abs(x))), rtol=1e-15)
    assert c["argmax"].tolist() == [0, 0, 0, 1, 1]      # x = 0 ties -> lowest id


def test_confidence_matches_logsumexp():
    rng = np.random.default_rng(7)
    h = rng.standard_normal((9, 16))
    W = rng.standard_normal((300, 16)) * 0.7
    c = oracle.confidence(h, W, row_chunk=4)
    l = h @ W.T
    np.testing.assert_allclose(c["p_max"], np.exp(l.max(1) - logsumexp(l, axis=1)), rtol=1e-12)
    assert np.array_equal(c["argmax"], l.argmax(1))
    srt = np.sort(l, axis=1)
    np.testing.assert_allclose(c["top2_logit_gap"], srt[:, -1] - srt[:, -2], rtol=1e-12)


def test_argmax_ties_take_lowest_id():
    rng = np.random.default_rng(8)
    W = rng.standard_normal((50, 8))
    W[31] = W[12]                                           # exact duplicate rows
    h = 20.0 * W[12][None, :]
    c = oracle.confidence(h, W)
    assert c["argmax"][0] == 12
    assert c["top2_logit_gap"][0] == 0.0


def test_uniform_logits_give_one_over_v():
    c = oracle.confidence(np.zeros((2, 4)), np.ones((37, 4)))
    np.testing.assert_allclose(c["p_max"], 1.0 / 37, rtol=1e-15)
    assert c["argmax"].tolist() == [0, 0]


def test_strong_planted_row_is_recovered():
    from block_diffusion_decoding_denoise_gb300 import workload as wl
    w = wl.WORKLOADS["tiny_fp32"]
    W = wl.lm_head(w)
    h, t = wl.planted_hidden(w, W, 0, steps=1, a_max=1e-9)   # noise only
    h_big, _ = wl.planted_hidden(w, W, 0, steps=1)
    # replace the amplitude by a large one: a * W[t]/|W[t]| + noise, a = 200
    dirs = W[t[0]].astype(np.float64)
    dirs /= np.linalg.norm(dirs, axis=1, keepdims=True)
    hp = h[0, 0].astype(np.float64) + 200.0 * dirs
    c = oracle.confidence(hp, W)
    assert np.array_equal(c["argmax"], t[0])
    assert (c["p_max"] > 0.99).all()


# --- commit ---------------------------------------------------------------
def test_golden_hand_worked_commit():
    with open(os.path.join(HERE, "golden", "tiny_commit_v2.json")) as f:
        g = json.load(f)
    W = np.array(g["W"])
    h = np.array(g["h_steps"])
    tokens, steps, trace = oracle.decode_block(h, W, g["threshold"])
    assert steps.tolist() == g["expected_steps"]
    assert [t.tolist() for t in trace] == g["expected_tokens_after_step"]
    _, p_max, *_ = oracle.denoise_step(np.full((1, 4), -1), h[0], W, g["threshold"])
    np.testing.assert_allclose(p_max[0], g["expected_p_max_step0"], rtol=1e-14)


def _random_step_inputs(rng, B=3, L=8, V=20, H=6, scale=3.0):
    return rng.standard_normal((L, B, L, H)) * scale, rng.standard_normal((V, H))


def test_threshold_zero_commits_everything_in_one_step():
    rng = np.random.default_rng(9)
    h, W = _random_step_inputs(rng)
    tokens, steps, trace = oracle.decode_block(h, W, 0.0)
    assert steps.tolist() == [1, 1, 1] and len(trace) == 1
    assert (tokens >= 0).all()


def test_threshold_above_one_commits_exactly_one_per_step():
    rng = np.random.default_rng(10)
    h, W = _random_step_inputs(rng)
    tokens, steps, trace = oracle.decode_block(h, W, 1.5)
    assert steps.tolist() == [8, 8, 8]
    prev = np.full((3, 8), -1)
    for t in trace:
        assert ((t != -1).sum(1) - (prev != -1).sum(1)).tolist() == [1, 1, 1]
        prev = t


def test_commit_rule_properties_random():
    # the rule is characterised by: commits only masked positions; commits
    # every masked position with p >= T; if none reaches T, commits exactly the
    # most confident one (lowest position on ties); leaves the rest unchanged.
    rng = np.random.default_rng(11)
    for _ in range(300):
        B, L = 2, int(rng.integers(1, 7))
        tokens = np.where(rng.random((B, L)) < 0.6, -1, rng.integers(0, 9, (B, L)))
        p = np.round(rng.random((B, L)), 1)                  # many exact ties
        a = rng.integers(0, 9, (B, L))
        T = float(rng.choice([0.0, 0.3, 0.5, 0.9, 1.01]))
        new, chosen = oracle.commit(tokens, p, a, T)
        for b in range(B):
            masked = tokens[b] == -1
            assert not chosen[b][~masked].any()
            assert np.array_equal(new[b][~masked], tokens[b][~masked])
            assert np.array_equal(new[b][chosen[b]], a[b][chosen[b]])
            assert np.array_equal(new[b][masked & ~chosen[b]], tokens[b][masked & ~chosen[b]])
            hi = masked & (p[b] >= T)
            if hi.any():
                assert np.array_equal(chosen[b], hi)
            elif masked.any():
                assert chosen[b].sum() == 1
                i = int(np.nonzero(chosen[b])[0][0])
                best = p[b][masked].max()
                assert p[b, i] == best
                assert i == int(np.nonzero(masked & (p[b] == best))[0][0])
            else:
                assert not chosen[b].any()


def test_region_thresholds_step_count_closed_form():
    # region A (T = 0): every masked position qualifies, so step 1 commits all
    # of A and nothing else; region B (T = 2 > any probability): its positions
    # only ever go through the fallback, one per step.  Steps = 1 + |B|.
    rng = np.random.default_rng(21)
    h, W = _random_step_inputs(rng)
    B, L = 3, 8
    regions = [np.arange(L) < 3, np.arange(L) % 2 == 0, np.arange(L) >= 7]
    T = np.stack([np.where(a, 0.0, 2.0) for a in regions])
    tokens, steps, trace = oracle.decode_block(h, W, T)
    assert steps.tolist() == [1 + int((~a).sum()) for a in regions]
    for b, a in enumerate(regions):
        assert np.array_equal(trace[0][b] != -1, a)
        for k in range(1, int(steps[b])):          # while the sequence is active
            assert (trace[k][b] != -1).sum() - (trace[k - 1][b] != -1).sum() == 1


def test_region_thresholds_match_scalar_per_region():
    # per-position thresholds: a position's decision uses only its own T.  A
    # sequence whose positions all share one value must decode exactly as the
    # scalar rule with that value, whatever the other sequences use.
    rng = np.random.default_rng(22)
    h, W = _random_step_inputs(rng, scale=1.5)
    T = np.array([[0.3] * 8, [0.6] * 8, [0.9] * 8])
    tok_r, steps_r, _ = oracle.decode_block(h, W, T)
    for b, t in enumerate((0.3, 0.6, 0.9)):
        tok_s, steps_s, _ = oracle.decode_block(h[:, b:b + 1], W, t)
        assert np.array_equal(tok_r[b], tok_s[0]) and steps_r[b] == steps_s[0]


def test_region_threshold_nan_never_qualifies():
    # NaN compares false: a NaN region commits only through the fallback,
    # exactly like T above one
    rng = np.random.default_rng(23)
    h, W = _random_step_inputs(rng)
    T_nan = np.where(np.arange(8) < 4, 0.0, np.nan)[None].repeat(3, 0)
    T_big = np.where(np.arange(8) < 4, 0.0, 1.5)[None].repeat(3, 0)
    a = oracle.decode_block(h, W, T_nan)
    b = oracle.decode_block(h, W, T_big)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert a[1].tolist() == [5, 5, 5]


def test_decode_invariants():
    rng = np.random.default_rng(12)
    h, W = _random_step_inputs(rng, scale=1.2)
    tokens, steps, trace = oracle.decode_block(h, W, 0.6)
    assert ((steps >= 1) & (steps <= 8)).all()
    for a, b in zip(trace[:-1], trace[1:]):
        done = a != -1
        assert np.array_equal(a[done], b[done])             # never revised
        assert (b != -1).sum() > (a != -1).sum()             # progress each step


def test_literal_planted_spec_never_reaches_half():
    # a ~ U(0,12), W ~ N(0,0.02): correct-token logit <= 12*0.02*sqrt(H) ~ 5.4
    # at H=512 against V-1 noise logits, so p_max stays far below 0.5 and
    # every step commits exactly one position through the fallback.
    from block_diffusion_decoding_denoise_gb300 import workload as wl
    w = wl.WORKLOADS["tiny_fp32"]
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0)
    tokens, steps, trace = oracle.decode_block(h, W, 0.5)
    assert steps.tolist() == [32]


# --- paged cache ----------------------------------------------------------
def test_paged_append_then_read_is_concatenation():
    rng = np.random.default_rng(13)
    B, L, Hkv, D, ps = 2, 5, 2, 3, 4
    ctx = np.array([6, 8])                                   # seq 0 straddles a page
    npg = 8
    table = rng.permutation(npg).reshape(B, npg // B)
    pool = rng.standard_normal((npg, Hkv, ps, D))
    before = [oracle.paged_read(pool, table[b], ctx[b], ps) for b in range(B)]
    blk = rng.standard_normal((B, L, Hkv, D))
    pool2, ctx2 = oracle.append_block(pool, table, ctx, blk, [True, True], ps)
    assert ctx2.tolist() == [11, 13]
    for b in range(B):
        got = oracle.paged_read(pool2, table[b], ctx2[b], ps)
        assert np.array_equal(got, np.concatenate([before[b], blk[b]]))
    pool3, ctx3 = oracle.append_block(pool, table, ctx, blk, [False, True], ps)
    assert ctx3.tolist() == [6, 13]
    assert np.array_equal(oracle.paged_read(pool3, table[0], 8, ps)[:6], before[0])


def test_paged_read_follows_page_table():
    ps = 2
    pool = np.arange(4 * 1 * ps * 1, dtype=float).reshape(4, 1, ps, 1)
    got = oracle.paged_read(pool, [3, 0], 4, ps)[:, 0, 0]
    assert got.tolist() == [6.0, 7.0, 0.0, 1.0]


# --- sampling reading (temperature sampling, no truncation) ---------------------
def test_philox_matches_numpy_bit_generator():
    # numpy's Philox bit generator is Philox-4x64-10; it advances its counter
    # by one before producing each block of four words.
    cases = [([0, 0, 0, 0], [0, 0]), ([5, 7, 11, 13], [123, 456]),
             ([2**64 - 2, 2**64 - 1, 3, 2**63], [2**64 - 1, 2**63 + 5])]
    for ctr, key in cases:
        bg = np.random.Philox(counter=np.array(ctr, dtype=np.uint64),
                              key=np.array(key, dtype=np.uint64))
        ref = bg.random_raw(4)
        got = oracle.philox4x64_10([np.uint64(ctr[0] + 1)] + [np.uint64(c) for c in ctr[1:]], key)
        assert [int(w) for w in got] == [int(w) for w in ref]


def test_philox_uniforms_are_uniform_and_decorrelated():
    from scipy import stats
    v = np.arange(200000)
    u0 = oracle.uniform01(v, 0, 12345)
    u1 = oracle.uniform01(v, 1, 12345)          # other half of the same 64-bit word
    u2 = oracle.uniform01(v, 0, 12345, offset=1)  # next step
    u4 = oracle.uniform01(v, 8, 12345)          # next counter along positions
    assert ((u0 > 0) & (u0 < 1)).all()
    u3 = oracle.uniform01(v, 3, 12345)          # another word of the same block
    for u in (u0, u1, u2, u3, u4):
        assert stats.kstest(u, "uniform").pvalue > 1e-3
    for u in (u1, u2, u3, u4):
        assert abs(np.corrcoef(u0, u)[0, 1]) < 0.01
    # the eight positions of one block use eight distinct fields of its words
    block = np.stack([oracle.uniform01(v[:1000], p, 12345) for p in range(8)])
    assert len({tuple(r) for r in block}) == 8
    assert abs(np.corrcoef(u0[:-1], u0[1:])[0, 1]) < 0.01   # neighbouring counters
    assert not np.array_equal(u0, oracle.uniform01(v, 0, 12346))
    assert np.array_equal(u0, oracle.uniform01(v, 0, 12345))
    # the 23-bit grid: U * 2^23 - 1/2 is an integer
    k = u0 * (1 << 23) - 0.5
    assert np.array_equal(k, np.floor(k))


@pytest.mark.parametrize("temperature", [1.0, 0.5, 2.0])
def test_gumbel_max_draws_follow_softmax(temperature):
    # one row per draw: same logits, different position ids -> independent draws
    from scipy import stats
    l = np.array([0.3, -1.2, 2.0, 0.0, 0.7])
    W = np.diag(l)                                  # h = ones -> logits = l
    n = 20000
    h = np.ones((n, 5))
    res = oracle.sample_confidence(h, W, np.arange(n), seed=7, temperature=temperature,
                                   row_chunk=4096)
    p = np.exp(l / temperature - logsumexp(l / temperature))
    counts = np.bincount(res["token"], minlength=5)
    chi = stats.chisquare(counts, n * p)
    assert chi.pvalue > 1e-4, (counts, n * p)
    np.testing.assert_allclose(res["p_sel"], p[res["token"]], rtol=1e-12)


def test_tiny_temperature_draw_is_the_argmax():
    rng = np.random.default_rng(21)
    h = rng.standard_normal((50, 8))
    W = rng.standard_normal((40, 8))
    res = oracle.sample_confidence(h, W, np.arange(50), seed=3, temperature=1e-4)
    assert np.array_equal(res["token"], (h @ W.T).argmax(axis=1))


def _logits_as_hw(z):
    # h = z, W = I: h W^T = z exactly
    z = np.atleast_2d(np.asarray(z, dtype=np.float64))
    return z, np.eye(z.shape[1])


def test_truncation_threshold_closed_forms():
    # ties at the top-k boundary are all kept
    th, _ = oracle.truncation_threshold([3.0, 1.0, 3.0, 3.0, 0.0], top_k=2)
    assert th == 3.0
    # top-p over probabilities (0.4, 0.25, 0.2, 0.1, 0.05): running mass 0.4,
    # 0.65, 0.85 -> p = 0.7 keeps the top three
    p = np.array([0.4, 0.25, 0.2, 0.1, 0.05])
    z = np.log(p)
    th, margin = oracle.truncation_threshold(z, top_p=0.7)
    assert np.isclose(th, np.log(0.2)) and np.isclose(margin, 0.05)
    # p exactly at a running-mass value keeps that entry and nothing below it
    th, _ = oracle.truncation_threshold(z, top_p=0.65 - 1e-12)
    assert np.isclose(th, np.log(0.25))
    # order: top-k first, then top-p on the renormalised remainder.  With
    # probabilities (0.5, 0.3, 0.15, 0.05), k = 2 leaves (0.625, 0.375), and
    # p = 0.6 then keeps only the first; top-p first would have kept two
    z = np.log([0.5, 0.3, 0.15, 0.05])
    th, _ = oracle.truncation_threshold(z, top_k=2, top_p=0.6)
    assert np.isclose(th, np.log(0.5))
    # no truncation
    assert oracle.truncation_threshold(z)[0] == -np.inf
    assert oracle.truncation_threshold(z, top_k=4)[0] == -np.inf


def test_truncated_draw_degenerate_cases():
    rng = np.random.default_rng(31)
    h = rng.standard_normal((6, 5))
    W = rng.standard_normal((40, 5))
    pos = np.arange(6)
    z = h @ W.T
    for kw in ({"top_k": 1}, {"top_p": 1e-12}):
        r = oracle.sample_confidence_truncated(h, W, pos, seed=5, temperature=1.0, **kw)
        assert np.array_equal(r["token"], z.argmax(1))       # only the argmax is kept
        assert np.allclose(r["p_sel"], 1.0)
    # no truncation is the untruncated sampler
    a = oracle.sample_confidence_truncated(h, W, pos, seed=5, temperature=0.8)
    b = oracle.sample_confidence(h, W, pos, seed=5, temperature=0.8)
    assert np.array_equal(a["token"], b["token"])
    np.testing.assert_allclose(a["p_sel"], b["p_sel"], rtol=1e-12)


@pytest.mark.parametrize("kw,kept", [({"top_k": 3}, [0, 1, 2]),
                                     ({"top_p": 0.7}, [0, 1, 2]),
                                     ({"top_k": 4, "top_p": 0.5}, [0, 1])])
def test_truncated_draws_follow_the_renormalised_distribution(kw, kept):
    # chi-square of 8000 draws (offsets 0..7999) against the kept entries'
    # renormalised probabilities; nothing outside the kept set is ever drawn
    p = np.array([0.4, 0.25, 0.2, 0.1, 0.05])
    h, W = _logits_as_hw(np.log(p))
    n = 8000
    toks, psel = [], []
    for off in range(n):
        r = oracle.sample_confidence_truncated(h, W, [3], seed=11, temperature=1.0,
                                               offset=off, **kw)
        toks.append(int(r["token"][0]))
        psel.append(float(r["p_sel"][0]))
    toks = np.array(toks)
    assert set(np.unique(toks)) <= set(kept)
    q = p[kept] / p[kept].sum()
    counts = np.array([(toks == k).sum() for k in kept])
    chi2 = float((((counts - n * q) ** 2) / (n * q)).sum())
    assert chi2 < 20.0, (chi2, counts)                        # df <= 2: p < 5e-5
    for k in kept:                                            # confidence = q of the token
        assert np.allclose(np.array(psel)[toks == k], q[kept.index(k)])


def test_sampled_step_uses_the_commit_rule():
    rng = np.random.default_rng(22)
    h = rng.standard_normal((2, 6, 4)) * 3
    W = rng.standard_normal((9, 4))
    tokens = np.full((2, 6), -1)
    tokens[0, 2] = 4
    new, conf, tok, chosen, res, (bi, ii) = oracle.denoise_step_sampled(tokens, h, W, 0.5, 1.0, 5)
    assert conf[0, 2] == -1 and tok[0, 2] == -1 and new[0, 2] == 4
    exp_new, _ = oracle.commit(tokens, conf, tok, 0.5)
    assert np.array_equal(new, exp_new)
    assert (new[chosen] == tok[chosen]).all()


# --- decoder layer stack (reading R10-R13) -------------------------------------
def test_round_bf16_matches_torch_conversion():
    rng = np.random.default_rng(31)
    x = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-6, 6, 5000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875, -3.0e38, 1e-40, np.inf,
                         -np.inf]])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(x)
    assert np.array_equal(got, ref)
    assert np.isnan(oracle.round_bf16([np.nan])).all()


def test_rms_norm_closed_forms():
    rng = np.random.default_rng(32)
    x = rng.standard_normal((7, 64)) * 3.0
    eps = 1e-6
    y = oracle.rms_norm(x, eps)
    ms = (x * x).mean(axis=1)
    np.testing.assert_allclose((y * y).mean(axis=1), ms / (ms + eps), rtol=1e-13)
    np.testing.assert_allclose(y / x, np.broadcast_to(1 / np.sqrt(ms + eps)[:, None], x.shape),
                               rtol=1e-13)
    c = np.full((1, 16), -0.5)
    np.testing.assert_allclose(oracle.rms_norm(c, eps), -1 / np.sqrt(1 + eps / 0.25), rtol=1e-14)
    if hasattr(F, "rms_norm"):
        ref = F.rms_norm(torch.from_numpy(x), (64,), eps=eps).numpy()
        np.testing.assert_allclose(y, ref, rtol=1e-12)


def test_embed_picks_rows_and_mask_row():
    E = np.arange(12.0).reshape(4, 3)
    e_mask = np.array([-1.0, -2.0, -3.0])
    got = oracle.embed(np.array([[2, -1, 0], [-1, -1, 3]]), E, e_mask)
    assert got.tolist() == [[[6, 7, 8], [-1, -2, -3], [0, 1, 2]],
                            [[-1, -2, -3], [-1, -2, -3], [9, 10, 11]]]


def _layer_inputs(rng, L=5, C=7, Hq=4, Hkv=2, D=8, H=24):
    x = rng.standard_normal((L, H))
    wqkv = rng.standard_normal(((Hq + 2 * Hkv) * D, H)) * 0.3
    wo = rng.standard_normal((H, Hq * D)) * 0.3
    kc = oracle.round_bf16(rng.standard_normal((C, Hkv, D)))
    vc = oracle.round_bf16(rng.standard_normal((C, Hkv, D)))
    return x, wqkv, wo, kc, vc


def test_decoder_layer_with_zero_output_projection_keeps_x():
    rng = np.random.default_rng(33)
    x, wqkv, wo, kc, vc = _layer_inputs(rng)
    x2, k, v = oracle.decoder_layer(x, wqkv, np.zeros_like(wo), kc, vc, 4, 2)
    assert np.array_equal(x2, x)
    xn = oracle.round_bf16(oracle.rms_norm(x))
    np.testing.assert_allclose(k.reshape(5, -1), oracle.round_bf16(xn @ wqkv[32:48].T), rtol=0)
    np.testing.assert_allclose(v.reshape(5, -1), oracle.round_bf16(xn @ wqkv[48:64].T), rtol=0)


def test_decoder_layer_uniform_attention_closed_form():
    # zero query weights make every softmax uniform: each query head h then
    # averages the values of KV head h // 2 over the cache and the block, and
    # Wo = [I | 0] copies head outputs into the first Hq*D features of x
    rng = np.random.default_rng(34)
    L, C, Hq, Hkv, D = 5, 7, 4, 2, 8
    H = Hq * D + 3
    x, wqkv, _, kc, vc = _layer_inputs(rng, L, C, Hq, Hkv, D, H)
    wqkv[:Hq * D] = 0.0
    wo = np.zeros((H, Hq * D))
    wo[:Hq * D] = np.eye(Hq * D)
    x2, k, v = oracle.decoder_layer(x, wqkv, wo, kc, vc, Hq, Hkv)
    vall = np.concatenate([vc, v])                          # [C + L, Hkv, D]
    mean = vall.mean(axis=0)                                # [Hkv, D]
    heads = oracle.round_bf16(np.stack([mean[h // 2] for h in range(Hq)]))  # [Hq, D]
    expect = x.copy()
    expect[:, :Hq * D] += heads.reshape(1, -1)
    np.testing.assert_allclose(x2, expect, rtol=1e-13, atol=1e-13)


def test_decoder_layer_matches_torch_composition():
    rng = np.random.default_rng(35)
    L, C, Hq, Hkv, D, H = 6, 9, 4, 2, 8, 40
    x, wqkv, wo, kc, vc = _layer_inputs(rng, L, C, Hq, Hkv, D, H)

    def bf(t):
        return t.to(torch.float32).to(torch.bfloat16).to(torch.float64)

    xt = torch.from_numpy(x)
    xn = bf(xt / torch.sqrt((xt * xt).mean(-1, keepdim=True) + 1e-6))
    qkv = bf(F.linear(xn, torch.from_numpy(wqkv)))
    q, k, v = qkv.split([Hq * D, Hkv * D, Hkv * D], dim=-1)
    kall = torch.cat([torch.from_numpy(kc).reshape(C, -1), k]).reshape(C + L, Hkv, D)
    vall = torch.cat([torch.from_numpy(vc).reshape(C, -1), v]).reshape(C + L, Hkv, D)
    qh = q.reshape(L, Hq, D).permute(1, 0, 2)
    kh = kall.repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)
    vh = vall.repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)
    a = F.scaled_dot_product_attention(qh, kh, vh).permute(1, 0, 2).reshape(L, Hq * D)
    ref = xt + F.linear(bf(a), torch.from_numpy(wo))
    x2, k2, v2 = oracle.decoder_layer(x, wqkv, wo, kc, vc, Hq, Hkv)
    np.testing.assert_allclose(x2, ref.numpy(), rtol=1e-9, atol=1e-9)
    assert np.array_equal(k2.reshape(L, -1), k.numpy())


def test_silu_closed_forms():
    g = np.array([0.0, 1.0, -1.0, 30.0, -30.0])
    s = oracle.silu(g)
    assert s[0] == 0.0
    np.testing.assert_allclose(s[1], 1.0 / (1.0 + np.exp(-1.0)), rtol=1e-15)
    np.testing.assert_allclose(s[1] - s[2], 1.0, rtol=1e-15)   # silu(g) - silu(-g) = g
    np.testing.assert_allclose(s[3], 30.0, rtol=1e-12)
    assert abs(s[4]) < 1e-11


def test_mlp_zero_gate_or_down_is_identity_and_torch_composition():
    rng = np.random.default_rng(37)
    L, H, I = 5, 24, 40
    x = rng.standard_normal((L, H))
    wgu = rng.standard_normal((2 * I, H)) * 0.3
    wd = rng.standard_normal((H, I)) * 0.3
    # silu(0) = 0: a zero gate makes the MLP add nothing, whatever the up rows
    z = wgu.copy()
    z[:I] = 0.0
    assert np.array_equal(oracle.mlp_residual(x, z, wd), x)
    assert np.array_equal(oracle.mlp_residual(x, wgu, np.zeros_like(wd)), x)
    # torch: F.silu, F.linear, with the bf16 roundings at the same points

    def bf(t):
        return t.to(torch.float32).to(torch.bfloat16).to(torch.float64)

    xt = torch.from_numpy(x)
    xn = bf(F.rms_norm(xt, (H,), eps=1e-6))
    g, u = F.linear(xn, torch.from_numpy(wgu)).split([I, I], dim=-1)
    ref = xt + F.linear(bf(F.silu(g) * u), torch.from_numpy(wd))
    np.testing.assert_allclose(oracle.mlp_residual(x, wgu, wd), ref.numpy(), rtol=1e-9,
                               atol=1e-9)
    # in the layer: after the attention residual
    _, wqkv, wo, kc, vc = _layer_inputs(rng, L, 7, 4, 2, 8, H)
    xa, k, v = oracle.decoder_layer(x, wqkv, wo, kc, vc, 4, 2)
    xm, k2, v2 = oracle.decoder_layer(x, wqkv, wo, kc, vc, 4, 2, 1e-6, wgu, wd)
    assert np.array_equal(xm, oracle.mlp_residual(xa, wgu, wd)) and np.array_equal(k, k2)


def test_decoder_forward_composes_layers():
    rng = np.random.default_rng(36)
    V, H, Hq, Hkv, D, L, C = 11, 16, 2, 1, 8, 4, 3
    E = rng.standard_normal((V, H))
    e_mask = rng.standard_normal(H)
    tokens = np.array([3, -1, 10, -1])
    layers = [(rng.standard_normal(((Hq + 2 * Hkv) * D, H)) * 0.2,
               rng.standard_normal((H, Hq * D)) * 0.2) for _ in range(3)]
    caches = [(rng.standard_normal((C, Hkv, D)), rng.standard_normal((C, Hkv, D)))
              for _ in range(3)]
    x, ks, vs = oracle.decoder_forward(tokens, E, e_mask, layers, caches, Hq, Hkv)
    y = oracle.embed(tokens, E, e_mask)
    for (wqkv, wo), (kc, vc), k, v in zip(layers, caches, ks, vs):
        y, k1, v1 = oracle.decoder_layer(y, wqkv, wo, kc, vc, Hq, Hkv)
        assert np.array_equal(k1, k) and np.array_equal(v1, v)
    assert np.array_equal(x, y)
