"""Each attention kernel of the library against the oracle on the same cases.

bd_block_attention runs the tcgen05 head-pair kernel for large bf16 problems
at the SDAR shapes, the mma.sync kernel for the other bf16 cases and the SIMT
kernel for fp32, chosen by shape alone.  The library's test hook
bd_debug_force_attention_kernel forces one kernel so that each is checked on
small, ragged and full-size inputs (a kernel that does not support a shape
falls back to the one the shape picks).  "pair" runs the head-pair kernel
on every problem: on small ones its tile ranges give more CTAs than tiles and
many pieces per segment, all merged inside the launch.
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


@pytest.fixture(params=["auto", "pair", "mma", "simt"])
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
