"""Seeded input generators: known answers and distribution checks (CPU)."""
import numpy as np
import pytest
import torch

import workloads as W
from conftest import golden_rows


def test_philox_known_answers():
    rows = golden_rows("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for row in rows:
        v = [int(s, 16) for s in row.split()]
        out = W.philox4x32_10(v[0:4], v[4:6])
        assert list(out) == v[6:10]


def test_normal_moments_and_determinism():
    z = W.normal_f64(W.w_stream(9, 1, 2, 0), 400_000)
    assert abs(z.mean()) < 0.01
    assert abs(z.std() - 1.0) < 0.01
    # fourth moment of a Gaussian is 3
    assert abs((z ** 4).mean() - 3.0) < 0.08
    # counter-based: any slice regenerates identically
    part = W.normal_f64(W.w_stream(9, 1, 2, 0), 1000, first=12345)
    assert np.array_equal(part, z[12345:13345])


def test_normal_f32_is_one_rounding_of_f64():
    s = W.x_stream(9, 0, 0)
    a = W.normal_f32(s, 10_000, 0.02)
    b = W.normal_f64(s, 10_000, 0.02)
    assert np.array_equal(a, b.astype(np.float32))


def test_bf16_activations_round_to_nearest_even():
    s = W.x_stream(9, 3, 7)
    bits = W.normal_bf16(s, 50_000)
    f32 = W.normal_f32(s, 50_000)
    ref = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)


def test_zipf_popularity_and_gumbel_top_k():
    cfg = W.CONFIGS["prefill_35b"]
    p = W.zipf_popularity(cfg, 0)
    assert p.shape == (256,) and abs(p.sum() - 1) < 1e-12
    ranks = np.sort(p)[::-1]
    assert np.allclose(ranks[0] / ranks[9], 10 ** 1.1)
    logits = W.router_logits(cfg, 0, 0, T=512)
    top = np.argsort(-logits, axis=1, kind="stable")[:, :8]
    counts = np.bincount(top.ravel(), minlength=256)
    # the most popular expert is chosen far more often than the median one
    assert counts[np.argmax(p)] > 5 * np.median(counts)


def test_cache_stream_sets_share_and_logits():
    cfg = W.scaled(W.CONFIGS["cache_stream"], steps=200)
    sets = W.cache_stream_sets(cfg, 0, 200)
    assert all(len(s) == 8 and len(set(s)) == 8 for s in sets)
    shared = [len(set(a) & set(b)) for a, b in zip(sets, sets[1:])]
    assert 0.5 < np.mean(shared) / 8 < 0.7
    logits = W.cache_stream_logits(cfg, 0, 200)
    for s, chosen in enumerate(sets):
        top = sorted(np.argsort(-logits[s], kind="stable")[:8].tolist())
        assert top == chosen


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_config_shapes(name):
    cfg = W.CONFIGS[name]
    assert cfg.H % 256 == 0 and cfg.I % 128 == 0 and cfg.k <= cfg.E
    assert cfg.expert_bytes == 3 * cfg.H * cfg.I * 9 // 16
