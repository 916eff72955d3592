"""The combine logic of a sequence split across GPUs, with two CPU ranks
(torch.distributed, gloo).

Each rank computes its own part of the problem in plain numpy (a vocabulary
slice of the LM head, or a slice of the keys), the ranks exchange it with an
all-gather, and the library's host merge combines what was gathered; the
result must equal the oracle's single-rank answer ("Rethinking Document OCR
as Inverse Rendering via Diffusion Decoding", paper.rainbus.top summary,
method steps 3-4: the block's attention and each masked position's
confidence).  Ranks run as separate processes; nothing needs a GPU.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _vocab_rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from block_diffusion_decoding_denoise_gb300 import parallel
    rng = np.random.default_rng(11)            # the same inputs on every rank
    M, H, V = 24, 64, 1003
    h = rng.standard_normal((M, H))
    W = rng.standard_normal((V, H)) * 0.3
    h[:4] *= 6.0                                # a few confident rows
    masked = np.ones(M, bool)
    masked[5] = False                           # a committed position: empty state
    v0, v1 = parallel.vocab_shard_bounds(V, world, rank)
    logits = h @ W[v0:v1].T
    rec = np.zeros(M, parallel.RECORD)
    mx = logits.max(axis=1)
    rec["m"] = mx
    rec["s"] = np.exp(logits - mx[:, None]).sum(axis=1)
    rec["idx"] = logits.argmax(axis=1) + v0
    rec["m"][~masked] = -np.inf
    rec["s"][~masked] = 0.0
    rec["idx"][~masked] = np.iinfo(np.int32).max
    mine = torch.from_numpy(rec.view(np.int32).reshape(M, 3).copy())
    gathered = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(gathered, mine)
    g = np.stack([t.numpy() for t in gathered]).view(parallel.RECORD).reshape(world, M)
    merged = parallel.merge_records_host(g)
    out[rank] = (merged["s"].astype(np.float64), merged["idx"].astype(np.int64),
                 merged["m"].astype(np.float64))
    dist.destroy_process_group()


def _attention_rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from block_diffusion_decoding_denoise_gb300 import parallel
    rng = np.random.default_rng(12)
    R, C, D = 40, 301, 64                      # query rows, keys, head_dim
    q = rng.standard_normal((R, D))
    k = rng.standard_normal((C, D))
    v = rng.standard_normal((C, D))
    scale = 1.0 / np.sqrt(D)
    # keys split unevenly; rank 1's slice starts after every key row 0 may see
    lo, hi = (0, 170) if rank == 0 else (170, C)
    s = (q @ k[lo:hi].T) * scale
    m = s.max(axis=1)
    p = np.exp(s - m[:, None])
    l = p.sum(axis=1)
    o = p @ v[lo:hi]
    parts = torch.from_numpy(np.concatenate([m[:, None], l[:, None], o], axis=1).astype(np.float32))
    gathered = [torch.empty_like(parts) for _ in range(world)]
    dist.all_gather(gathered, parts)
    g = np.stack([t.numpy() for t in gathered])
    merged = parallel.merge_attention_host(g[:, :, 0], g[:, :, 1], g[:, :, 2:])
    out[rank] = merged.astype(np.float64)
    dist.destroy_process_group()


def _run(fn, world=2):
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=fn, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0, f"rank exited with {p.exitcode}"
        return dict(out)


def test_vocab_parallel_confidence_two_ranks_equals_single_rank():
    import oracle
    res = _run(_vocab_rank)
    rng = np.random.default_rng(11)
    M, H, V = 24, 64, 1003
    h = rng.standard_normal((M, H))
    W = rng.standard_normal((V, H)) * 0.3
    h[:4] *= 6.0
    ref = oracle.confidence(h, W)
    for rank in (0, 1):
        s, idx, m = res[rank]
        masked = np.arange(M) != 5
        np.testing.assert_allclose(1.0 / s[masked], ref["p_max"][masked], rtol=1e-5)
        assert np.array_equal(idx[masked], ref["argmax"][masked])
        assert np.isneginf(m[5]) and idx[5] == np.iinfo(np.int32).max
    assert np.array_equal(res[0][1], res[1][1])     # both ranks commit the same tokens


def test_kv_split_attention_two_ranks_equals_single_rank():
    import oracle
    res = _run(_attention_rank)
    rng = np.random.default_rng(12)
    R, C, D = 40, 301, 64
    q = rng.standard_normal((R, D))
    k = rng.standard_normal((C, D))
    v = rng.standard_normal((C, D))
    # the R query rows (one head) at the last R positions of a single block,
    # so each sees every key
    qq = np.zeros((C, 1, D))
    qq[C - R:, 0] = q
    ref = oracle.block_attention(qq, k[:, None, :], v[:, None, :], np.zeros(C, np.int64),
                                 np.arange(C - R, C))[:, 0, :]
    for rank in (0, 1):
        np.testing.assert_allclose(res[rank], ref, rtol=0, atol=2e-5)


def test_vocab_shard_bounds_cover_the_vocabulary():
    from block_diffusion_decoding_denoise_gb300 import parallel
    for V, world in [(151936, 8), (1003, 2), (7, 3), (5, 8)]:
        spans = [parallel.vocab_shard_bounds(V, world, r) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == V
        assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
        sizes = [b - a for a, b in spans]
        assert max(sizes) - min(sizes) <= 1
