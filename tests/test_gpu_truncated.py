"""GPU parity of top-k / top-p truncated sampling (bd_sample_commit_truncated).

The oracle computes every row's truncation threshold in fp64 over all V
logits and draws with the same counter-based noise; tokens and confidences
are compared row by row (exemptions in tests/_parity.py).  A chi-square test
checks the GPU's draws against the renormalised kept distribution directly.
"""
import numpy as np
import pytest
import torch

from block_diffusion_decoding_denoise_gb300 import bd
from block_diffusion_decoding_denoise_gb300 import workload as wl

from _parity import ConfRunner, SampleRunner, dev, lockstep_sampled_block

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


def test_truncated_block_tiny_fp32():
    # fp32: logits from the SIMT kernel
    w = wl.WORKLOADS["tiny_fp32"]
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=40.0)
    lockstep_sampled_block(w, W, h, 0.95, 1.0, seed=11, top_k=50, top_p=0.9)


@pytest.mark.parametrize("top_k,top_p", [(20, 1.0), (0, 0.9), (50, 0.8), (3, 0.5), (999, 1.0)])
def test_truncated_block_bf16_ragged_vocab(top_k, top_p):
    # V = 1000: the last 128-entry tile of the tensor-core logits is partial
    w = SMALL_BF16
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=30.0)
    lockstep_sampled_block(w, W, h, 0.9, 0.8, seed=5, top_k=top_k, top_p=top_p)


@pytest.mark.parametrize("vocab,top_k,top_p", [(997, 30, 0.9), (7, 2, 1.0), (7, 0, 0.6)])
def test_truncated_vocab_not_a_multiple_of_four(vocab, top_k, top_p):
    # rows that are not 16-byte aligned take the scalar load path of the
    # selection kernel; V = 7 also leaves most of the logits tile empty
    w = SMALL_BF16.with_(vocab=vocab)
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=30.0)
    lockstep_sampled_block(w, W, h, 0.9, 0.8, seed=9, top_k=top_k, top_p=top_p, max_steps=6)


def test_truncated_more_rows_than_one_pass():
    w = SMALL_BF16.with_(batch=9)                 # 288 rows: two passes of <= 256
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=30.0)
    lockstep_sampled_block(w, W, h, 0.9, 1.0, seed=3, max_steps=2, top_k=40, top_p=0.95)


def test_truncated_sdar_b1_full_size_first_steps():
    w = wl.WORKLOADS["sdar_b1"]
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, steps=2, a_max=32.0)
    st = lockstep_sampled_block(w, W, h, w.threshold, 1.0, seed=2024, max_steps=2, top_k=50,
                                top_p=0.9)
    assert st.rows_checked >= 32


def test_top_k_one_is_the_greedy_argmax():
    w = SMALL_BF16
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, steps=1, a_max=30.0)
    hd = dev(h[0], w.dtype)
    _, _, g_a, _, _ = ConfRunner(w, W, 2.0).step(hd)
    _, p, s, _, _ = SampleRunner(w, W, 2.0, 1.0, seed=1, top_k=1).step(hd, 0)
    assert np.array_equal(s, g_a)
    assert np.all(p == 1.0)


def test_no_truncation_is_the_sampled_call():
    w = SMALL_BF16
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, steps=1, a_max=5.0)
    hd = dev(h[0], w.dtype)
    a = SampleRunner(w, W, 2.0, 0.9, seed=8).step(hd, 4)
    run = SampleRunner(w, W, 2.0, 0.9, seed=8)
    run.truncated = True                          # call the truncated entry point with k=0, p=1
    b = run.step(hd, 4)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("top_k,top_p", [(5, 1.0), (0, 0.6), (8, 0.7)])
def test_truncated_draws_follow_the_kept_distribution(top_k, top_p):
    # 2048 rows with the same logits, 10 draws each: nothing outside the kept
    # set is drawn, and the histogram matches the renormalised kept softmax
    # (fp64 from the same bf16 inputs, the kept set from the same rule)
    from scipy import stats
    import oracle
    w = SMALL_BF16.with_(batch=64, hidden=64, vocab=40)
    rng = np.random.default_rng(19)
    W = wl.round_bf16(rng.standard_normal((w.vocab, w.hidden)).astype(np.float32))
    x = wl.round_bf16((rng.standard_normal(w.hidden) * 0.25).astype(np.float32))
    h = np.broadcast_to(x, (w.batch, w.block_len, w.hidden)).copy()
    temp = 0.8
    l = W.astype(np.float64) @ x.astype(np.float64) / temp
    theta, margin = oracle.truncation_threshold(l, top_k, top_p)
    assert margin > 1e-3
    keep = l >= theta
    p = np.where(keep, np.exp(l - l.max()), 0.0)
    p /= p.sum()
    run = SampleRunner(w, W, 2.0, temp, seed=77, top_k=top_k, top_p=top_p)
    hd = dev(h, w.dtype)
    counts = np.zeros(w.vocab, np.int64)
    for off in range(10):
        run.set_tokens(np.full((w.batch, w.block_len), -1))
        _, p_sel, s, _, _ = run.step(hd, off)
        counts += np.bincount(s.reshape(-1), minlength=w.vocab)
        np.testing.assert_allclose(p_sel.reshape(-1), p[s.reshape(-1)], atol=2e-3)
    assert counts[~keep].sum() == 0
    n = counts.sum()
    big = keep & (n * p >= 5)
    obs = np.append(counts[big], counts[keep & ~big].sum())
    exp = np.append(n * p[big], n * p[keep & ~big].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    assert stats.chisquare(obs, exp).pvalue > 1e-4, (counts, n * p)
