"""Each attention kernel of the library against the oracle on the same cases.

bd_block_attention runs, for bf16, the cluster-per-segment kernel on small
problems and the tcgen05 head-pair kernel (SDAR shapes) or the mma.sync kernel
(other shapes) on large ones; the SIMT kernel for fp32.  The choice is by shape
alone.  The library's test hook bd_debug_force_attention_kernel forces one
kernel so that each is checked on small, ragged and full-size inputs (a kernel
that does not support a shape falls back to the one the shape picks).
- "pair" runs the head-pair kernel on every problem.  On small ones its tile
  ranges give more CTAs than tiles and many pieces per segment, all merged
  inside the launch.
- "cluster" and "pair_cluster" run the cluster forms of the mma.sync and
  head-pair kernels on every problem.  On sdar_b1 they run clusters of up to
  16 CTAs per segment.  On serving_b64 they run one CTA per segment, with up to
  193 tiles, so the page ids past the first 32 come from the page table one by
  one.
"""
import numpy as np
import pytest
import torch

from block_diffusion_decoding_denoise_gb300 import bd
from block_diffusion_decoding_denoise_gb300 import workload as wl

from _parity import gpu_attention, make_cache, oracle_attention

pytestmark = pytest.mark.gpu

SMALL = wl.WORKLOADS["sdar_b1"].with_(name="small_bf16", batch=3, hidden=256, vocab=1000,
                                      prefix=300, prefix_min=0)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_decoding_denoise_gb300 import build
    build.build()
    bd.load()


@pytest.fixture(params=["auto", "pair", "mma", "simt", "cluster", "pair_cluster"])
def impl(request):
    bd.bd_debug_force_attention_kernel(request.param)
    yield request.param
    bd.bd_debug_force_attention_kernel("auto")


def _check(w, plen, impl, blk=0):
    s = make_cache(w, 0, plen)
    q, kb, vb = wl.block_qkv(w, blk)
    got = gpu_attention(s, q, kb, vb)
    worst = 0.0
    for b in range(w.batch):
        err = float(np.abs(got[b] - oracle_attention(s, b, q, kb, vb)).max())
        worst = max(worst, err)
    assert worst <= 2e-2, f"{impl}: max-abs error {worst}"


def _poison_unused_rows(s):
    """NaN in every pool row that holds no cached token: the rest of each
    sequence's last page and every page no sequence uses."""
    cache = s.cache
    valid = torch.zeros(cache.k.shape[0], cache.k.shape[2], dtype=torch.bool)
    for b, n in enumerate(s.plen):
        pos = np.arange(int(n))
        pages = cache.page_table_np[b][pos // bd.BD_PAGE_SIZE]
        valid[torch.from_numpy(pages.astype(np.int64)),
              torch.from_numpy((pos % bd.BD_PAGE_SIZE).astype(np.int64))] = True
    bad = (~valid).to(cache.k.device)[:, None, :, None].expand_as(cache.k)
    cache.k.masked_fill_(bad, float("nan"))
    cache.v.masked_fill_(bad, float("nan"))


def test_nan_in_unused_pool_rows(impl):
    # A masked key has probability zero, and zero times NaN is NaN: no kernel
    # may let a pool row past a sequence's context reach its output (the
    # tails of partial last pages: 77, 130 and 1 tokens; the block tile of 32
    # keys in a 64-row stage)
    w = SMALL.with_(batch=4)
    s = make_cache(w, 0, [77, 300, 1, 130])
    _poison_unused_rows(s)
    q, kb, vb = wl.block_qkv(w, 0)
    got = gpu_attention(s, q, kb, vb)
    assert np.isfinite(got).all(), f"{impl}: non-finite output"
    worst = max(float(np.abs(got[b] - oracle_attention(s, b, q, kb, vb)).max())
                for b in range(w.batch))
    assert worst <= 2e-2, f"{impl}: max-abs error {worst}"


def test_ragged_prefixes(impl):
    # 0 (block only), 77 (odd page count, partial page), 300
    _check(SMALL, [0, 77, 300], impl)


def test_ragged_long_batch(impl):
    w = SMALL.with_(batch=6, prefix=3000, prefix_min=100)
    _check(w, [3000, 100, 2049, 64, 1, 2900], impl)


def test_sdar_b1(impl):
    _check(wl.WORKLOADS["sdar_b1"], None, impl)


def test_block_len_8(impl):
    # 8 positions x 2 heads = 16 query rows per KV head
    _check(SMALL.with_(block_len=8), [130, 5, 64], impl)


def test_serving_shapes_sampled(impl):
    # 64 ragged sequences (2048..12288 cached tokens): many pieces per segment
    # and segments inside one CTA's range; three sequences checked
    w = wl.WORKLOADS["serving_b64"]
    s = make_cache(w, 0)
    q, kb, vb = wl.block_qkv(w, 0)
    got = gpu_attention(s, q, kb, vb)
    for b in (0, 31, 63):
        err = float(np.abs(got[b] - oracle_attention(s, b, q, kb, vb)).max())
        assert err <= 2e-2, f"{impl}: sequence {b} max-abs error {err}"


def test_sequence_without_mask_is_skipped(impl):
    # sequence 1 has no masked position: its output rows stay untouched
    w = SMALL
    s = make_cache(w, 0, [300, 140, 65])
    q, kb, vb = wl.block_qkv(w, 0)
    tokens = np.full((w.batch, w.block_len), bd.BD_MASK, dtype=np.int32)
    tokens[1] = 7
    tokens[2, ::2] = 11                            # half committed: still attended
    got = gpu_attention(s, q, kb, vb, tokens=torch.from_numpy(tokens).cuda())
    assert np.isnan(got[1]).all()
    for b in (0, 2):
        err = float(np.abs(got[b] - oracle_attention(s, b, q, kb, vb)).max())
        assert err <= 2e-2, f"{impl}: sequence {b} max-abs error {err}"


def test_head_dim_64(impl):
    # D = 64: the head-pair kernel does not take it (it falls back by shape);
    # the mma.sync kernels run their 64-column instantiations
    w = SMALL.with_(head_dim=64)
    _check(w, [0, 77, 300], impl)
