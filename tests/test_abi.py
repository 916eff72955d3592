"""The C ABI: libbd.so builds, loads without a GPU and exports every symbol
that include/bd.h declares; host-side argument checks answer without
launching anything (so they run on a machine with no GPU)."""
import ctypes
import os
import re

import pytest

from block_diffusion_decoding_denoise_gb300 import bd, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return bd.load()


def _declared():
    with open(os.path.join(ROOT, "include", "bd.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bd_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("bd_block_attention", "bd_confidence_commit", "bd_append_block_kv",
              "bd_status_string"):
        assert n in names
    assert sorted(bd.EXPORTS) == names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert bd.bd_status_string(0) == "BD_OK"
    assert bd.bd_status_string(4) == "BD_ERR_DEVICE_CHECK"
    assert bd.bd_status_string(99) == "BD_ERR_UNKNOWN"
    assert bd.bd_version() >= 100


def test_workspace_queries_reject_bad_shapes(lib):
    assert bd.bd_confidence_commit_workspace(bd.BD_BF16, 1, 32, 2048, 151936) > 0
    assert bd.bd_confidence_commit_workspace(bd.BD_BF16, 1, 33, 2048, 151936) == 0
    assert bd.bd_confidence_commit_workspace(bd.BD_BF16, 1, 32, 100, 151936) == 0
    assert bd.bd_confidence_commit_workspace(7, 1, 32, 2048, 151936) == 0
    assert bd.bd_block_attention_workspace(1, 32, 16, 8, 96, 4096) == 0
    assert bd.bd_block_attention_workspace(1, 32, 16, 5, 128, 4096) == 0
    assert bd.bd_block_attention_workspace(1, 32, 16, 8, 128, -1) == 0


def test_null_arguments_are_rejected_before_any_launch(lib):
    f = lib.bd_confidence_commit
    st = f(1, 1, 32, 2048, 1000, None, None, 0.9, None, None, None, None, None, None, 0,
           None, None)
    assert st == 1
    st = lib.bd_block_attention(None, None, None, 1, 32, 16, 100, None, None, None, 0.1,
                                None, None, 0, None, None)
    assert st == 1
    kv = bd.PagedKV(1, 4, 64, 8, 128, 4, None, None, None)
    st = lib.bd_append_block_kv(ctypes.byref(kv), 1, 32, None, None, None, None, None, None)
    assert st == 1


def test_sample_commit_checks_arguments_on_the_host(lib):
    assert bd.bd_sample_commit_workspace(bd.BD_BF16, 1, 32, 2048, 151936) >= \
        bd.bd_confidence_commit_workspace(bd.BD_BF16, 1, 32, 2048, 151936)
    assert bd.bd_sample_commit_workspace(bd.BD_BF16, 1, 33, 2048, 151936) == 0
    f = lib.bd_sample_commit
    for temp in (0.0, -1.0, float("nan"), float("inf")):
        st = f(1, 1, 32, 2048, 1000, None, None, 0.9, temp, 1, None, None, None, None, None,
               None, None, 0, None, None)
        assert st == 1
    st = f(1, 1, 32, 2048, 1000, None, None, 0.9, 1.0, 1, None, None, None, None, None, None,
           None, 0, None, None)
    assert st == 1


def test_region_commit_checks_arguments_on_the_host(lib):
    f = lib.bd_confidence_commit_regions
    for thr in (None, 2, 4096 + 1):                      # missing or not 4-byte aligned
        st = f(1, 1, 32, 2048, 1000, None, None, thr, None, None, None, None, None, None, 0,
               None, None)
        assert st == 1
    st = f(1, 1, 33, 2048, 1000, None, None, 4096, None, None, None, None, None, None, 0,
           None, None)                                   # block_len above 32
    assert st == 1


def test_truncated_sample_commit_checks_arguments_on_the_host(lib):
    assert bd.bd_sample_commit_truncated_workspace(bd.BD_BF16, 1, 32, 2048, 151936) >= \
        bd.bd_sample_commit_workspace(bd.BD_BF16, 1, 32, 2048, 151936) + 32 * 151936 * 4
    assert bd.bd_sample_commit_truncated_workspace(bd.BD_BF16, 1, 33, 2048, 151936) == 0
    f = lib.bd_sample_commit_truncated
    for k, p in ((-1, 0.9), (5, 0.0), (5, 1.5), (5, float("nan")), (5, -0.5)):
        st = f(1, 1, 32, 2048, 1000, None, None, 0.9, 1.0, k, p, 1, 4096, None, None, None,
               None, None, None, 0, None, None)
        assert st == 1
    st = f(1, 1, 32, 2048, 1000, None, None, 0.9, 1.0, 5, 0.9, 1, None, None, None, None,
           None, None, None, 0, None, None)              # no draw counter
    assert st == 1


def test_mlp_call_checks_arguments_on_the_host(lib):
    assert bd.bd_mlp_workspace(32, 2048, 6144) > 32 * 6144 * 2
    for rows, H, inter in ((0, 2048, 6144), (32, 2000, 6144), (32, 2048, 100), (32, 8192, 64)):
        assert bd.bd_mlp_workspace(rows, H, inter) == 0
    st = lib.bd_mlp_residual(32, 2048, 6144, None, None, None, 1e-6, None, None, None, 0, None,
                             None)
    assert st == 1
    st = lib.bd_mlp_residual(32, 2048, 6144, 4096, 4096, 4096, -1.0, 4096, 4096, 4096, 1 << 30,
                             None, None)                 # negative eps
    assert st == 1


def test_decoder_calls_check_arguments_on_the_host(lib):
    # shapes the projection kernels cannot take return a zero workspace
    assert bd.bd_qkv_projection_workspace(256, 2048, 16, 8, 128) > 0
    assert bd.bd_qkv_projection_workspace(256, 2000, 16, 8, 128) == 0      # hidden % 64
    assert bd.bd_qkv_projection_workspace(256, 2048, 16, 8, 3) == 0        # features % 128
    assert bd.bd_out_projection_workspace(256, 2048, 2048) > 0
    assert bd.bd_out_projection_workspace(0, 2048, 2048) == 0
    # null pointers and bad sizes are rejected before any launch
    assert lib.bd_embed_rmsnorm(4, 2048, 100, None, None, None, 1e-6, None, None, None,
                                None) == 1
    assert lib.bd_embed_rmsnorm(4, 6000, 100, None, None, None, 1e-6, None, None, None,
                                None) == 1
    assert lib.bd_qkv_projection(256, 2048, 16, 8, 128, None, None, None, None, None, None, 0,
                                 None, None) == 1
    assert lib.bd_out_projection_residual(256, 2048, 2048, None, None, 1e-6, None, None, None,
                                          0, None, None) == 1
    kv = (bd.PagedKV * 2)(bd.PagedKV(1, 4, 64, 8, 128, 4, None, None, None),
                          bd.PagedKV(1, 4, 64, 8, 128, 4, None, None, None))
    assert lib.bd_append_block_kv_layers(kv, 2, 1, 32, None, None, None, None, None,
                                         None) == 1
    assert lib.bd_append_block_kv_layers(kv, 65, 1, 32, None, None, None, None, None,
                                         None) == 1
