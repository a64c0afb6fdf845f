"""Oracle pins: router top-k / softmax weights and the expert permutation (CPU).

Pins: brute-force sorting, the full softmax from an independent library
(scipy), invariance to a constant shift, crafted exact ties, and the
permutation's defining properties checked against Python's stable sort.
"""
import numpy as np
import pytest
import scipy.special

import oracle as O


def brute_topk(logits, k):
    T, E = logits.shape
    return np.array([[e for _, e in sorted((-float(logits[t, e]), e) for e in range(E))[:k]] for t in range(T)],
                    dtype=np.int32)


@pytest.mark.parametrize("T,E,k", [(5, 8, 2), (16, 256, 8), (3, 128, 8), (1, 7, 7)])
def test_route_matches_brute_force(T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    ids, w = O.route(logits, k)
    assert np.array_equal(ids, brute_topk(logits, k))
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)   # descending logits -> descending weights


def test_route_k_equals_e_is_the_full_softmax():
    rng = np.random.default_rng(11)
    logits = rng.normal(size=(4, 32)).astype(np.float32)
    ids, w = O.route(logits, 32)
    ref = scipy.special.softmax(logits.astype(np.float64), axis=1)
    got = np.zeros_like(ref)
    np.put_along_axis(got, ids.astype(np.int64), w, axis=1)
    assert np.allclose(got, ref, rtol=1e-13, atol=0)


def test_route_weights_are_renormalised_softmax():
    rng = np.random.default_rng(12)
    logits = rng.normal(size=(6, 64)).astype(np.float32)
    ids, w = O.route(logits, 4)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    assert np.allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13)


def test_route_shift_invariance():
    """Adding a constant to every logit (exactly, in fp32) leaves ids and weights unchanged."""
    rng = np.random.default_rng(13)
    logits = (rng.integers(-4096, 4096, size=(8, 256)) / 1024.0).astype(np.float32)  # exact multiples of 2^-10
    ids, w = O.route(logits, 8)
    ids2, w2 = O.route(logits + np.float32(64.0), 8)                             # still exact in fp32
    assert np.array_equal(ids, ids2)
    assert np.allclose(w, w2, rtol=1e-12)
    assert np.array_equal(ids, brute_topk(logits, 8))


def test_route_ties_go_to_lower_index():
    logits = np.zeros((3, 8), np.float32)
    logits[1, [6, 2, 4]] = 1.0
    logits[2, :] = [0.5, 0.5, -0.0, 0.0, 0.5, -1, 0.5, 0.0]
    ids, w = O.route(logits, 3)
    assert ids[0].tolist() == [0, 1, 2]
    assert ids[1].tolist() == [2, 4, 6]
    assert ids[2].tolist() == [0, 1, 4]
    assert np.allclose(w[0], 1 / 3) and np.allclose(w[1], 1 / 3)


def test_route_minus_inf_and_invalid():
    logits = np.array([[0.0, -np.inf, 1.0, -np.inf]], np.float32)
    ids, w = O.route(logits, 2)
    assert ids.tolist() == [[2, 0]]
    ids, w = O.route(logits, 3)
    assert ids.tolist() == [[2, 0, 1]] and w[0, 2] == 0.0
    all_ninf = np.full((1, 4), -np.inf, np.float32)
    ids, w = O.route(all_ninf, 2)
    assert ids.tolist() == [[0, 1]] and np.all(w == 0.5)
    for bad in (np.nan, np.inf):
        l2 = logits.copy()
        l2[0, 1] = bad
        with pytest.raises(O.OracleError):
            O.route(l2, 2)
    with pytest.raises(O.OracleError):
        O.route(logits, 5)


@pytest.mark.parametrize("T,E,k", [(4, 8, 2), (4096, 256, 8), (16, 256, 8), (1, 128, 8), (0, 8, 2)])
def test_permute_properties(T, E, k):
    rng = np.random.default_rng(T + E)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    ids, _ = O.route(logits, k) if T else (np.zeros((0, k), np.int32), None)
    offsets, perm, inv = O.permute(ids, E)
    flat = ids.reshape(-1)
    # stable sort by expert, i.e. by (expert, f)
    ref = sorted(range(T * k), key=lambda f: (int(flat[f]), f))
    assert perm.tolist() == ref
    assert np.array_equal(inv[perm], np.arange(T * k))
    assert np.array_equal(np.diff(offsets), np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


def test_permute_rejects_out_of_range():
    with pytest.raises(O.OracleError):
        O.permute(np.array([[0, 8]], np.int32), 8)
    with pytest.raises(O.OracleError):
        O.permute(np.array([[-1, 2]], np.int32), 8)
