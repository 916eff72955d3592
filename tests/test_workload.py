"""The seeded input generators: determinism and bf16 rounding."""
import numpy as np
import torch

from block_diffusion_decoding_denoise_gb300 import workload as wl


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1e-30, 3.0e38, 1.00390625, 1.01171875],
                                 dtype=np.float32)])
    ours = wl.round_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_generators_are_deterministic_and_chunk_independent():
    a = wl.normal_f32((3, 1 << 23), 0, 1, 99)
    b = wl.normal_f32((3, 1 << 23), 0, 1, 99)
    assert np.array_equal(a, b)
    assert abs(float(a.std()) - 1.0) < 1e-3


def test_page_tables_are_permutations():
    w = wl.WORKLOADS["serving_b64"]
    plen = wl.prefix_lengths(w)
    assert plen.min() >= 2048 and plen.max() <= 12288
    table, npg = wl.page_tables(w, plen + 32)
    used = table[table >= 0]
    assert sorted(used.tolist()) == list(range(npg))


def test_planted_hidden_shapes():
    w = wl.WORKLOADS["tiny_fp32"]
    W = wl.lm_head(w)
    h, t = wl.planted_hidden(w, W, 0, steps=3)
    assert h.shape == (3, 1, 32, 512) and t.shape == (1, 32)
    assert (t >= 0).all() and (t < w.vocab).all()
