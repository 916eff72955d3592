"""GPU parity of the sampling reading (bd_sample_commit) against the oracle.

The oracle draws with the same counter-based generator (Philox-4x64-10 at
counter (v, position / 8, offset, 0)), so sampled tokens are compared token by
token; see tests/_parity.py for the exemption rule.  A chi-square test checks
the GPU's draws against softmax directly, independent of the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from block_diffusion_decoding_denoise_gb300 import bd
from block_diffusion_decoding_denoise_gb300 import workload as wl

from _parity import ConfRunner, SampleRunner, dev, lockstep_sampled_block, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_decoding_denoise_gb300 import build
    build.build()
    bd.load()


SMALL_BF16 = wl.WORKLOADS["sdar_b1"].with_(name="small_bf16", batch=3, hidden=256, vocab=1000,
                                           prefix=300, prefix_min=0)


def test_sampled_block_tiny_fp32():
    w = wl.WORKLOADS["tiny_fp32"]
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=40.0)
    st = lockstep_sampled_block(w, W, h, 0.95, 1.0, seed=11)
    assert st.steps_gpu[0] <= 32


@pytest.mark.parametrize("temperature", [1.0, 0.7])
def test_sampled_block_bf16_ragged_vocab(temperature):
    w = SMALL_BF16
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=30.0)
    lockstep_sampled_block(w, W, h, 0.9, temperature, seed=5)


def test_sampled_sparse_masked_positions():
    # masked positions scattered over position groups: the kernel's Philox
    # blocks are shared only by rows of one group of eight positions
    w = SMALL_BF16
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=30.0)
    tok0 = np.full((w.batch, w.block_len), 7)
    tok0[0, [1, 2, 5, 9, 10, 11, 12, 30]] = -1
    tok0[1, ::5] = -1
    tok0[2, 31] = -1
    lockstep_sampled_block(w, W, h, 0.95, 1.0, seed=123456789012345, tokens0=tok0)


def test_sampled_few_positions_read_in_place():
    # 64 positions: direct rows in the LM head, positions = row indices
    w = SMALL_BF16.with_(batch=2)
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=30.0)
    tok0 = np.full((w.batch, w.block_len), -1)
    tok0[1, 4:20] = 3
    lockstep_sampled_block(w, W, h, 0.9, 1.0, seed=21, tokens0=tok0)


def test_sampled_two_lmhead_passes():
    w = SMALL_BF16.with_(batch=9)                 # 288 rows: two passes of <= 256
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=30.0)
    lockstep_sampled_block(w, W, h, 0.9, 1.0, seed=3, max_steps=2)


def test_sampled_sdar_b1_full_size_first_step():
    w = wl.WORKLOADS["sdar_b1"]
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, steps=1, a_max=32.0)
    st = lockstep_sampled_block(w, W, h, w.threshold, 1.0, seed=2024, max_steps=1)
    assert st.rows_checked == 32


def test_sampled_draws_follow_softmax():
    # 2048 rows with the same logits, 10 draws each (offsets 0..9): the
    # histogram of drawn tokens against softmax in fp64 of the same bf16 inputs
    from scipy import stats
    w = SMALL_BF16.with_(batch=64, hidden=64, vocab=40)
    rng = np.random.default_rng(9)
    W = wl.round_bf16(rng.standard_normal((w.vocab, w.hidden)).astype(np.float32))
    x = wl.round_bf16((rng.standard_normal(w.hidden) * 0.25).astype(np.float32))
    h = np.broadcast_to(x, (w.batch, w.block_len, w.hidden)).copy()
    temp = 0.8
    run = SampleRunner(w, W, 2.0, temp, seed=77)
    hd = dev(h, w.dtype)
    counts = np.zeros(w.vocab, np.int64)
    l = W.astype(np.float64) @ x.astype(np.float64) / temp
    p = np.exp(l - l.max())
    p /= p.sum()
    for off in range(10):
        run.set_tokens(np.full((w.batch, w.block_len), -1))
        _, p_sel, s, _, _ = run.step(hd, off)
        counts += np.bincount(s.reshape(-1), minlength=w.vocab)
        np.testing.assert_allclose(p_sel.reshape(-1), p[s.reshape(-1)], atol=2e-3)
    n = counts.sum()
    keep = n * p >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(n * p[keep], n * p[~keep].sum())
    assert stats.chisquare(obs, exp).pvalue > 1e-4, (counts, n * p)


def test_low_temperature_draw_is_the_greedy_argmax():
    w = SMALL_BF16
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, steps=1, a_max=30.0)
    hd = dev(h[0], w.dtype)
    greedy = ConfRunner(w, W, 2.0)
    _, _, g_a, _, _ = greedy.step(hd)
    samp = SampleRunner(w, W, 2.0, 1e-4, seed=1)
    _, _, s, _, _ = samp.step(hd, 0)
    c = oracle.confidence(h[0].reshape(-1, w.hidden).astype(np.float64), W.astype(np.float64))
    # Gumbel noise spans less than 19.5 in units of z = l / 1e-4, so it cannot
    # reorder logits more than 1.95e-3 apart
    clear = (c["top2_logit_gap"] > 4e-3).reshape(w.batch, w.block_len)
    assert clear.mean() > 0.9
    assert np.array_equal(s[clear], g_a[clear])


def test_same_seed_and_offset_repeat_exactly():
    w = SMALL_BF16
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, steps=1, a_max=5.0)
    hd = dev(h[0], w.dtype)
    run = SampleRunner(w, W, 2.0, 1.0, seed=42)
    outs = []
    for off in (3, 3, 4):
        run.set_tokens(np.full((w.batch, w.block_len), -1))
        _, p, s, _, _ = run.step(hd, off)
        outs.append((p, s))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    assert (outs[0][1] != outs[2][1]).mean() > 0.3         # a new offset draws afresh


@pytest.mark.parametrize("temperature", [0.0, -1.0, float("nan"), float("inf"), 1e-9])
def test_bad_temperature_is_rejected(temperature):
    w = SMALL_BF16
    W = wl.lm_head(w)
    run = SampleRunner(w, W, 0.9, 1.0, seed=0)
    run.temp = temperature
    h = torch.zeros(w.batch, w.block_len, w.hidden, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bd.BDError) as e:
        run.step(h, 0)
    assert e.value.status == 1
    assert (run.tokens == -1).all()


def test_graph_replays_draw_fresh_noise():
    # the draw counter lives on the device: every replay of a captured step
    # reads it and advances it, so replay k draws exactly as offset n0 + k
    w = SMALL_BF16
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, steps=1, a_max=5.0)
    hd = dev(h[0], w.dtype)
    run = SampleRunner(w, W, 2.0, 1.0, seed=99)
    run.offset.fill_(40)
    run.set_tokens(np.full((w.batch, w.block_len), -1))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bd.bd_sample_commit(hd, run.W, run.T, run.temp, run.seed, run.offset, run.tokens,
                            run.p_sel, run.sampled, run.ncom, run.nmask, run.ws,
                            dev_status=run.status)
    torch.cuda.synchronize()
    assert int(run.offset.item()) == 40                     # capture runs nothing
    tokens0 = np.full((w.batch, w.block_len), -1)
    pos = np.arange(w.batch * w.block_len)
    seen = []
    for k in range(3):
        run.set_tokens(tokens0)
        g.replay()
        torch.cuda.synchronize()
        assert int(run.offset.item()) == 41 + k
        s = run.sampled.cpu().numpy().reshape(-1)
        ref = oracle.sample_confidence(h[0].reshape(-1, w.hidden).astype(np.float64),
                                       W.astype(np.float64), pos, 99, 1.0, offset=40 + k)
        ok = (s == ref["token"]) | (ref["key_gap"] < 1e-3)
        assert ok.all()
        seen.append(s)
    assert (seen[0] != seen[1]).mean() > 0.3
