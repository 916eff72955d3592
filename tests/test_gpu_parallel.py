"""The GPU side of a sequence split across GPUs, simulated on one GPU.

Vocabulary-parallel LM head: W is cut into slices; bd_confidence_shard
reduces each slice to 12-byte states per position, the states are stacked as
an all-gather would, and bd_commit_shards commits from them.  The result must
equal bd_confidence_commit over the whole W (and the oracle).  KV-split
attention: partials of several key slices, formed in numpy, merged by the
device merge against the oracle's attention over all keys.
"""
import numpy as np
import pytest
import torch

import oracle
from block_diffusion_decoding_denoise_gb300 import bd, parallel
from block_diffusion_decoding_denoise_gb300 import workload as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_decoding_denoise_gb300 import build
    build.build()
    bd.load()


@pytest.mark.parametrize("name,batch,shards", [("small", 3, 3), ("sdar_b1", 1, 4),
                                                ("sdar_b1", 8, 2)])
def test_vocab_parallel_commit_equals_whole_vocabulary(name, batch, shards):
    base = wl.WORKLOADS["sdar_b1"]
    w = base.with_(batch=batch, hidden=256, vocab=5000) if name == "small" else base.with_(batch=batch)
    W = wl.lm_head(w)
    h, _ = wl.planted_hidden(w, W, 0, steps=2, a_max=32.0)
    Wd = torch.from_numpy(W).to("cuda", torch.bfloat16)
    B, L = w.batch, w.block_len
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def outputs():
        return (torch.empty(B, L, device="cuda"), torch.empty(B, L, dtype=torch.int32, device="cuda"),
                torch.empty(B, dtype=torch.int32, device="cuda"),
                torch.empty(B, dtype=torch.int32, device="cuda"))
    tok_ref = torch.full((B, L), -1, dtype=torch.int32, device="cuda")
    tok_ref.view(-1)[::5] = 7                    # some positions already committed
    tok_sh = tok_ref.clone()
    ref, sh = outputs(), outputs()
    ws = torch.empty(bd.bd_confidence_commit_workspace(bd.BD_BF16, B, L, w.hidden, w.vocab),
                     dtype=torch.uint8, device="cuda")
    bounds = [parallel.vocab_shard_bounds(w.vocab, shards, r) for r in range(shards)]
    for step in range(2):
        hd = torch.from_numpy(h[step]).to("cuda", torch.bfloat16)
        bd.bd_confidence_commit(hd, Wd, w.threshold, tok_ref, *ref, ws, dev_status=st)
        recs = torch.empty(shards, B * L, 3, dtype=torch.int32, device="cuda")
        for r, (v0, v1) in enumerate(bounds):
            wsr = torch.empty(bd.bd_confidence_shard_workspace(B, L, w.hidden, v1 - v0),
                              dtype=torch.uint8, device="cuda")
            bd.bd_confidence_shard(hd, Wd[v0:v1], v0, tok_sh, recs[r], wsr, dev_status=st)
        bd.bd_commit_shards(recs, w.vocab, w.threshold, tok_sh, *sh, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        # same decisions and argmax; p_max equal up to the order of the fp32 sums
        assert torch.equal(tok_ref, tok_sh)
        assert torch.equal(ref[1], sh[1]) and torch.equal(ref[2], sh[2]) and torch.equal(ref[3], sh[3])
        pr, ps = ref[0].cpu().numpy(), sh[0].cpu().numpy()
        m = pr >= 0
        np.testing.assert_allclose(ps[m], pr[m], rtol=2e-5)
        assert (ps[~m] == -1).all()
        # and the oracle's confidence of the masked rows
        bi, ii = np.nonzero(sh[1].cpu().numpy() >= 0)
        c = oracle.confidence(h[step][bi, ii].astype(np.float64), W.astype(np.float64))
        np.testing.assert_allclose(ps[bi, ii], c["p_max"], atol=2e-2)
        ok = c["top2_prob_margin"] >= 1e-3
        assert np.array_equal(sh[1].cpu().numpy()[bi, ii][ok], c["argmax"][ok])


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_kv_split_merge_on_device(out_dtype):
    rng = np.random.default_rng(21)
    R, C, D, S = 64, 777, 128, 3
    q = rng.standard_normal((R, D))
    k = rng.standard_normal((C, D))
    v = rng.standard_normal((C, D))
    cuts = [0, 250, 251, 777]                   # one slice holds a single key
    m, l, o = [], [], []
    for s in range(S):
        sc = (q @ k[cuts[s]:cuts[s + 1]].T) / np.sqrt(D)
        mx = sc.max(axis=1)
        p = np.exp(sc - mx[:, None])
        m.append(mx)
        l.append(p.sum(axis=1))
        o.append(p @ v[cuts[s]:cuts[s + 1]])
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(np.stack(x), np.float32)).cuda()
    out = torch.empty(R, D, dtype=out_dtype, device="cuda")
    bd.bd_merge_attention_partials(dev(m), dev(l), dev(o), out)
    torch.cuda.synchronize()
    qq = np.zeros((C, 1, D))
    qq[C - R:, 0] = q
    ref = oracle.block_attention(qq, k[:, None, :], v[:, None, :], np.zeros(C, np.int64),
                                 np.arange(C - R, C))[:, 0, :]
    tol = 1e-5 if out_dtype == torch.float32 else 2e-2
    assert float(np.abs(out.float().cpu().numpy() - ref).max()) <= tol
    host = parallel.merge_attention_host(np.stack(m), np.stack(l), np.stack(o))
    assert float(np.abs(host - ref).max()) <= 1e-5
