"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Inputs come from the seeded generators only; expected values come from the
oracle only.  See tests/_parity.py for the tolerances and exemption rule.
"""
import numpy as np
import pytest
import torch

import oracle
from block_diffusion_decoding_denoise_gb300 import bd
from block_diffusion_decoding_denoise_gb300 import workload as wl

from _parity import (ConfRunner, dev, gpu_attention, lockstep_block, make_cache,
                     oracle_attention, tol_for, torch_dtype)

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


def _attn_check(w, plen=None, seed=0, rows_of=None):
    s = make_cache(w, seed, plen)
    q, kb, vb = wl.block_qkv(w, 0, seed)
    got = gpu_attention(s, q, kb, vb)
    tol = tol_for(w.dtype)
    worst = 0.0
    for b in (range(w.batch) if rows_of is None else rows_of):
        ref = oracle_attention(s, b, q, kb, vb)
        err = float(np.abs(got[b] - ref).max())
        worst = max(worst, err)
        assert err <= tol, f"seq {b}: attention max-abs error {err} > {tol}"
    return worst


# --- attention --------------------------------------------------------------
def test_attention_tiny_fp32():
    _attn_check(wl.WORKLOADS["tiny_fp32"])


def test_attention_bf16_ragged_prefixes():
    # prefixes 0 (block only), 77 (ragged page), 300: several pages and a tail
    _attn_check(SMALL_BF16, plen=[0, 77, 300])


def test_attention_fp32_d128_gqa4():
    w = wl.WORKLOADS["tiny_fp32"].with_(name="f32_d128", batch=2, num_q_heads=8,
                                        num_kv_heads=2, head_dim=128, prefix=200, prefix_min=64)
    _attn_check(w, plen=[200, 64])


def test_attention_bf16_gqa4_128_rows():
    # 32 positions x 4 query heads per KV head = 128 rows: eight row groups per tile
    w = SMALL_BF16.with_(name="gqa4", num_q_heads=16, num_kv_heads=4, batch=2)
    _attn_check(w, plen=[333, 64])


def test_attention_bf16_head_dim_64():
    w = SMALL_BF16.with_(name="d64", head_dim=64, num_q_heads=8, num_kv_heads=2, batch=2)
    _attn_check(w, plen=[190, 0])


def test_attention_bf16_long_ragged_batch():
    # enough pages for the multi-item-per-CTA split (several items per SM)
    w = SMALL_BF16.with_(name="ragged", batch=6, prefix=3000, prefix_min=100)
    _attn_check(w, plen=[3000, 100, 2049, 64, 1, 2900], rows_of=[0, 1, 2, 3, 4, 5])


def test_attention_block_len_one_is_causal_step():
    # block size 1: the query sees the cache and itself, i.e. one AR step
    w = wl.WORKLOADS["tiny_fp32"].with_(name="ar", block_len=1, batch=2)
    _attn_check(w, plen=[130, 1])


def test_attention_sdar_b1_full():
    _attn_check(wl.WORKLOADS["sdar_b1"])


def test_attention_split_count_invariance():
    w = SMALL_BF16
    s = make_cache(w, 0, [300, 300, 300])
    q, kb, vb = wl.block_qkv(w, 0)
    a = gpu_attention(s, q, kb, vb)
    s.max_ctx = 4096                               # same data, another KV split
    b = gpu_attention(s, q, kb, vb)
    assert np.abs(a - b).max() <= 2e-2


def test_attention_paged_equals_contiguous_layout():
    w = SMALL_BF16
    s = make_cache(w, 0, [300, 77, 5])
    q, kb, vb = wl.block_qkv(w, 0)
    a = gpu_attention(s, q, kb, vb)
    # same cache, identity page table
    from block_diffusion_decoding_denoise_gb300.engine import PagedCache
    npg = s.cache.k.shape[0]
    table = np.full_like(s.cache.page_table_np, -1)
    off = 0
    for b in range(w.batch):
        n = int((s.cache.page_table_np[b] >= 0).sum())
        table[b, :n] = np.arange(off, off + n)
        off += n
    c2 = PagedCache(npg, w.num_kv_heads, w.head_dim, torch_dtype(w.dtype), table)
    for b in range(w.batch):
        c2.load_prefix(b, torch.from_numpy(s.k_pre[b]), torch.from_numpy(s.v_pre[b]))
    s.cache = c2
    assert np.array_equal(gpu_attention(s, q, kb, vb), a)


def test_attention_skips_finished_sequences():
    w = SMALL_BF16
    s = make_cache(w, 0, [10, 20, 30])
    q, kb, vb = wl.block_qkv(w, 0)
    tokens = torch.full((w.batch, w.block_len), -1, dtype=torch.int32, device="cuda")
    tokens[1] = 7                                   # sequence 1 fully committed
    got = gpu_attention(s, q, kb, vb, tokens=tokens)
    assert np.isnan(got[1]).all()
    assert not np.isnan(got[0]).any() and not np.isnan(got[2]).any()


def test_attention_corrupt_page_table_sets_status():
    w = SMALL_BF16
    s = make_cache(w, 0, [200, 200, 200])
    bad = s.cache.page_table_np.copy()
    bad[1, 1] = s.cache.k.shape[0] + 5             # outside the pool
    s.cache.page_table.copy_(torch.from_numpy(bad))
    q, kb, vb = wl.block_qkv(w, 0)
    out = torch.empty(w.batch, w.block_len, w.num_q_heads, w.head_dim, dtype=torch.bfloat16,
                      device="cuda")
    nws = bd.bd_block_attention_workspace(w.batch, w.block_len, w.num_q_heads, w.num_kv_heads,
                                          w.head_dim, s.max_ctx)
    ws = torch.zeros(max(nws, 1), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.bd_block_attention(s.cache.kv, s.ctx_len, None, dev(q, "bf16"), dev(kb, "bf16"),
                          dev(vb, "bf16"), out, ws, s.max_ctx, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 4                      # BD_ERR_DEVICE_CHECK


def test_bounded_wait_timeout_sets_status_and_context_survives():
    """A bounded device wait that runs out (the self-test kernel waits on a
    barrier nothing arrives at, with tensor memory allocated, nothing in
    flight) reports BD_ERR_TIMEOUT through the status word, and the context
    stays usable: an attention call right after it matches the oracle."""
    import time
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    bd.bd_debug_wait_timeout_selftest(st)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == 5                      # BD_ERR_TIMEOUT
    assert 0.9 <= dt < 10.0, f"the wait gave up after {dt:.2f} s"
    w = SMALL_BF16
    s = make_cache(w, 0, [200, 77, 0])
    q, kb, vb = wl.block_qkv(w, 0)
    got = gpu_attention(s, q, kb, vb)
    for b in range(w.batch):
        assert float(np.abs(got[b] - oracle_attention(s, b, q, kb, vb)).max()) <= 2e-2


# --- confidence + commit --------------------------------------------------------
def test_decode_tiny_fp32_literal_spec():
    w = wl.WORKLOADS["tiny_fp32"]
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0)
    st = lockstep_block(w, W, h, w.threshold)
    assert st.steps_gpu.tolist() == [32]           # fallback only under a ~ U(0,12)


def test_decode_tiny_fp32_strong_plant():
    # a ~ U(0,40): many positions clear 0.95, exercising the threshold path
    w = wl.WORKLOADS["tiny_fp32"]
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=40.0)
    st = lockstep_block(w, W, h, w.threshold)
    assert st.steps_gpu[0] < 32


def test_decode_small_bf16_ragged_vocab():
    w = SMALL_BF16
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=30.0)
    lockstep_block(w, W, h, 0.9)


@pytest.mark.parametrize("T,steps", [(0.0, 1), (1.5, 32)])
def test_decode_threshold_extremes(T, steps):
    w = SMALL_BF16
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0)
    st = lockstep_block(w, W, h, T)
    assert st.steps_gpu.tolist() == [steps] * w.batch


@pytest.mark.parametrize("batch", [1, 2])
def test_decode_few_positions_read_in_place(batch):
    # <= 64 positions per call: the LM head reads every row of h in place, no
    # compaction; the commit must still use only the masked rows
    w = SMALL_BF16.with_(batch=batch)
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=30.0)
    tok0 = np.full((w.batch, w.block_len), -1)
    tok0[0, ::3] = 5                              # some positions already committed
    st = lockstep_block(w, W, h, 0.9, tokens0=tok0)
    assert st.rows_checked > 0


def test_decode_region_thresholds():
    # per-position thresholds (bd_confidence_commit_regions): three regions per
    # sequence at different offsets, one sequence with a NaN region (never
    # qualifies), under a plant strong enough for every threshold to matter
    w = SMALL_BF16
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=30.0)
    B, L = w.batch, w.block_len
    T = np.empty((B, L))
    for b in range(B):
        i = (np.arange(L) + 7 * b) % L
        T[b] = np.where(i < 8, 0.99, np.where(i < 24, 0.7, 0.9))
    T[-1, :5] = np.nan
    st = lockstep_block(w, W, h, T)
    assert st.rows_checked > 0


def test_decode_region_thresholds_closed_form():
    # T = 0 on region A, T = 2 elsewhere: step 1 commits exactly A, then one
    # position per step through the fallback, so steps = 1 + (L' - |A|)
    w = SMALL_BF16
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0)
    B, L = w.batch, w.block_len
    sizes = [(5 * b + 3) % L for b in range(B)]
    T = np.stack([np.where(np.arange(L) < n, 0.0, 2.0) for n in sizes])
    st = lockstep_block(w, W, h, T)
    assert st.steps_gpu.tolist() == [1 + L - n if n else L for n in sizes]


def test_decode_more_rows_than_one_pass():
    # 5 x 32 = 160 masked rows: the LM head takes two passes of at most 128 rows
    w = SMALL_BF16.with_(batch=5)
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=30.0)
    lockstep_block(w, W, h, 0.9)


def test_decode_two_lmhead_passes():
    # 9 x 32 = 288 masked positions: two LM-head passes of up to 256 rows
    w = SMALL_BF16.with_(batch=9)
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=30.0)
    lockstep_block(w, W, h, 0.9, check_oracle_full=False)


def test_decode_partially_committed_entry_state():
    w = SMALL_BF16
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, a_max=30.0)
    tok0 = np.full((w.batch, w.block_len), -1)
    tok0[0, ::3] = 11
    tok0[2, :] = 5                                  # sequence 2 already finished
    tok0[2, 31] = -1
    st = lockstep_block(w, W, h, 0.95, tokens0=tok0)
    assert (st.final_gpu[0, ::3] == 11).all()


def test_decode_block_len_one():
    w = SMALL_BF16.with_(block_len=1)
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0)
    st = lockstep_block(w, W, h, 0.95)
    assert st.steps_gpu.tolist() == [1, 1, 1]


def test_argmax_tie_takes_lowest_id():
    w = SMALL_BF16.with_(batch=1)
    W = wl.lm_head(w)
    W[777] = W[5]                                   # exact duplicate rows
    W[999] = W[5]
    h = np.zeros((1, 1, w.block_len, w.hidden), np.float32)
    h[0, 0, :] = wl.round_bf16(W[5] * 40.0)
    run = ConfRunner(w, W, 0.0)
    tok, p, a, nc, nm = run.step(dev(h[0], w.dtype))
    assert (a[0] == 5).all() and (tok[0] == 5).all()
    c = oracle.confidence(h[0, 0].astype(np.float64), W.astype(np.float64))
    np.testing.assert_allclose(p[0], c["p_max"], atol=2e-2)


def test_vocab_of_one():
    w = SMALL_BF16.with_(batch=2, vocab=1)
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, steps=1)
    run = ConfRunner(w, W, 0.95)
    tok, p, a, nc, nm = run.step(dev(h[0], w.dtype))
    assert (p == 1.0).all() and (a == 0).all() and (tok == 0).all()
    assert nc.tolist() == [32, 32] and nm.tolist() == [0, 0]


def test_decode_sdar_b1_literal_spec():
    # full-size LM head (151936 x 2048); every step checked against fp64 logits
    w = wl.WORKLOADS["sdar_b1"]
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0)
    st = lockstep_block(w, W, h, w.threshold, check_oracle_full=False)
    assert st.steps_gpu.tolist() == [32]
    print(f"\nsdar_b1: rows={st.rows_checked} max|dp|={st.max_pmax_err:.2e} "
          f"max rel dp={st.max_rel_pmax_err:.2e} argmax compared={st.argmax_compared} "
          f"exempt={st.exempt_positions} adoptions={st.lockstep_adoptions}")
    # the 1e-3 margin exempts many rows at p_max near 1e-4; many are still decided
    assert st.argmax_compared >= st.rows_checked // 5


# --- append ---------------------------------------------------------------------
@pytest.mark.parametrize("name", ["tiny_fp32", "small_bf16"])
def test_append_matches_oracle(name):
    w = wl.WORKLOADS["tiny_fp32"].with_(batch=3) if name == "tiny_fp32" else SMALL_BF16
    s = make_cache(w, 0, [0, 77, 40], extra_blocks=2)
    _, kb, vb = wl.block_qkv(w, 0)
    nmask = torch.tensor([0, 3, 0], dtype=torch.int32, device="cuda")   # seq 1 not done
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k_before = s.cache.k.float().cpu().numpy()
    v_before = s.cache.v.float().cpu().numpy()
    bd.bd_append_block_kv(s.cache.kv, dev(kb, w.dtype), dev(vb, w.dtype), s.ctx_len, nmask,
                          dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    done = [True, False, True]
    k_exp, ctx_exp = oracle.append_block(k_before, s.cache.page_table_np, s.plen, kb, done, 64)
    v_exp, _ = oracle.append_block(v_before, s.cache.page_table_np, s.plen, vb, done, 64)
    assert s.ctx_len.cpu().numpy().tolist() == ctx_exp.tolist()
    assert np.array_equal(s.cache.k.float().cpu().numpy(), k_exp)
    assert np.array_equal(s.cache.v.float().cpu().numpy(), v_exp)


def test_attention_after_append_sees_block():
    # the appended block joins the cache: the next block attends to it
    w = SMALL_BF16
    s = make_cache(w, 0, [77, 0, 130], extra_blocks=2)
    _, kb, vb = wl.block_qkv(w, 0)
    bd.bd_append_block_kv(s.cache.kv, dev(kb, w.dtype), dev(vb, w.dtype), s.ctx_len)
    q1, kb1, vb1 = wl.block_qkv(w, 1)
    got = gpu_attention(s, q1, kb1, vb1)
    for b in range(w.batch):
        kc = np.concatenate([s.k_pre[b], kb[b]])
        vc = np.concatenate([s.v_pre[b], vb[b]])
        ref = oracle.current_block_attention(q1[b], kc, vc, kb1[b], vb1[b])
        assert np.abs(got[b] - ref).max() <= 2e-2


# --- host-side argument checks ------------------------------------------------
def test_host_validation_rejects_bad_arguments():
    w = SMALL_BF16
    W = torch.zeros(w.vocab, w.hidden, dtype=torch.bfloat16, device="cuda")
    h = torch.zeros(w.batch, w.block_len, w.hidden, dtype=torch.bfloat16, device="cuda")
    tok = torch.full((w.batch, w.block_len), -1, dtype=torch.int32, device="cuda")
    p = torch.empty(w.batch, w.block_len, device="cuda")
    a = torch.empty_like(tok)
    n1 = torch.empty(w.batch, dtype=torch.int32, device="cuda")
    n2 = torch.empty_like(n1)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(bd.BDError) as e:
        bd.bd_confidence_commit(h, W, 0.9, tok, p, a, n1, n2, ws)
    assert e.value.status == 6                        # workspace too small
    n = bd.bd_confidence_commit_workspace(bd.BD_BF16, w.batch, w.block_len, w.hidden, w.vocab)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    with pytest.raises(bd.BDError) as e:
        bd.bd_confidence_commit(h, W, float("nan"), tok, p, a, n1, n2, ws)
    assert e.value.status == 1
    assert bd.bd_block_attention_workspace(1, 32, 16, 8, 96, 100) == 0   # head_dim 96
    assert bd.bd_confidence_commit_workspace(bd.BD_BF16, 1, 33, 2048, 10) == 0
    assert (tok == -1).all()                          # nothing ran


# --- full-size batched serving workload, sampled against the oracle -------------
def test_serving_b64_full_size_sampled():
    """64 sequences with ragged prefixes (2048..12288) in a permuted paged cache and
    the 151936 x 2048 LM head: attention checked on sampled sequences, the first
    denoise step's confidence checked on two whole sequences, and the commit rule
    checked on every sequence."""
    w = wl.WORKLOADS["serving_b64"]
    s = make_cache(w, 0)
    q, kb, vb = wl.block_qkv(w, 0)
    got = gpu_attention(s, q, kb, vb)
    for b in (0, 17, 63):
        ref = oracle_attention(s, b, q, kb, vb)
        assert np.abs(got[b] - ref).max() <= 2e-2
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, steps=1)
    run = ConfRunner(w, W, w.threshold)
    tok, p, a, nc, nm = run.step(dev(h[0], w.dtype))
    # every sequence: exactly one commit (nothing reaches 0.95 under this recipe),
    # at a position whose GPU p_max is the largest, with the GPU argmax
    assert (nc == 1).all() and (nm == 31).all()
    for b in range(w.batch):
        i = int(np.nonzero(tok[b] != -1)[0][0])
        assert p[b, i] == p[b].max() and tok[b, i] == a[b, i]
    # two whole sequences against fp64 logits
    for b in (5, 40):
        c = oracle.confidence(h[0, b].astype(np.float64), W.astype(np.float64))
        assert np.abs(p[b] - c["p_max"]).max() <= 2e-2
        exempt = c["top2_prob_margin"] < 1e-3
        assert (a[b][~exempt] == c["argmax"][~exempt]).all()
        best = c["p_max"].max()
        i = int(np.nonzero(tok[b] != -1)[0][0])
        assert best - c["p_max"][i] < 1e-3        # same position up to the near-tie exemption
