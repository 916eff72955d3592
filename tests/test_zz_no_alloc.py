"""The allocation-free confidence/commit entry point.

bd_confidence_commit_noalloc serves callers that cannot allocate device
memory when they run a step (serving runtimes that forbid allocation
mid-request, plugins without access to their host's allocator, embedded
callers whose device memory is all handed out at start-up): it takes its
scratch space from a fixed array the library keeps on the device.  This test drives it through the C ABI for two consecutive
denoise steps and checks every output against bd_confidence_commit, which
uses a caller workspace.  It lives in a file of its own that pytest collects
last, and passes both alone and after the other tests.
"""
import numpy as np
import pytest
import torch

from block_diffusion_decoding_denoise_gb300 import bd
from block_diffusion_decoding_denoise_gb300 import workload as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_decoding_denoise_gb300 import build
    build.build()
    bd.load()


def _outputs(B, L):
    dev = "cuda"
    return (torch.empty(B, L, dtype=torch.float32, device=dev),
            torch.empty(B, L, dtype=torch.int32, device=dev),
            torch.empty(B, dtype=torch.int32, device=dev),
            torch.empty(B, dtype=torch.int32, device=dev))


@pytest.mark.parametrize("name,a_max", [("small", 30.0), ("sdar_b1", 12.0)])
def test_noalloc_matches_workspace_entry_point(name, a_max):
    base = wl.WORKLOADS["sdar_b1"]
    w = base.with_(batch=3, hidden=256, vocab=1000) if name == "small" else base
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, steps=2, a_max=a_max)
    Wd = torch.from_numpy(W).to("cuda", torch.bfloat16)
    hd = torch.from_numpy(h).to("cuda", torch.bfloat16)
    B, L = w.batch, w.block_len
    n = bd.bd_confidence_commit_workspace(bd.BD_BF16, B, L, w.hidden, w.vocab)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    tok_ref = torch.full((B, L), -1, dtype=torch.int32, device="cuda")
    tok_na = tok_ref.clone()
    ref, na = _outputs(B, L), _outputs(B, L)
    st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    st_na = torch.zeros(1, dtype=torch.int32, device="cuda")
    for step in range(2):                          # two calls in a row
        bd.bd_confidence_commit(hd[step], Wd, w.threshold, tok_ref, *ref, ws, dev_status=st_ref)
        bd.bd_confidence_commit_noalloc(hd[step], Wd, w.threshold, tok_na, *na, dev_status=st_na)
        torch.cuda.synchronize()
        assert int(st_ref.item()) == 0 and int(st_na.item()) == 0
        assert torch.equal(tok_ref, tok_na)
        assert torch.equal(ref[1], na[1])           # argmax
        assert torch.equal(ref[2], na[2]) and torch.equal(ref[3], na[3])
        np.testing.assert_allclose(na[0].cpu().numpy(), ref[0].cpu().numpy(), atol=2e-2, rtol=0)
        assert int((tok_na != -1).sum()) > 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # batch 64 x 32 positions at SDAR shapes needs far more than the 8 MiB array
    B, L, H, V = 64, 32, 2048, 151936
    assert bd.bd_confidence_commit_workspace(bd.BD_BF16, B, L, H, V) > (8 << 20)
    h = torch.zeros(B, L, H, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(V, H, dtype=torch.bfloat16, device="cuda")
    tok = torch.full((B, L), -1, dtype=torch.int32, device="cuda")
    p, a, n1, n2 = _outputs(B, L)
    with pytest.raises(bd.BDError) as e:
        bd.bd_confidence_commit_noalloc(h, W, 0.9, tok, p, a, n1, n2)
    assert e.value.status == 6                     # BD_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((tok == -1).all())                 # nothing ran
