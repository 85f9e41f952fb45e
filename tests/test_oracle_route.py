"""Pins of the oracle's routing and expert sort: brute force on small inputs
(Python sorting of tuples), closed forms of the softmax weights, and the
invariants of the per-expert offsets (a monotone prefix sum of the histogram
that leaves the sentinel bin out, so its last entry counts the live rows)."""
import numpy as np
import pytest
from scipy.special import softmax

from oracle import mark_sentinels, route_topk, sort_by_expert
from grouped_gemm_serving_gb300 import synth


def _brute_topk(lp, k):
    # order experts by (-value, id): ties go to the lower expert id
    return [sorted(range(len(row)), key=lambda e: (-row[e], e))[:k] for row in lp]


@pytest.mark.parametrize("T,E,k,ties", [(17, 8, 2, False), (33, 32, 4, False), (9, 128, 8, False),
                                        (40, 8, 3, True), (25, 16, 16, True), (5, 256, 8, False)])
def test_topk_ids_brute_force(T, E, k, ties):
    g = np.random.default_rng([T, E, k])
    if ties:
        logits = g.integers(-2, 3, size=(T, E)).astype(np.float32)   # many exact ties
    else:
        logits = g.standard_normal((T, E), dtype=np.float32)
    bias = g.standard_normal(E, dtype=np.float32) * np.float32(0.5)
    for b in (None, bias):
        ids, w = route_topk(logits, b, k)
        lp = logits if b is None else logits + b[None, :]
        assert ids.tolist() == _brute_topk(lp.tolist(), k)


def test_weights_closed_forms():
    g = np.random.default_rng(5)
    logits = g.standard_normal((64, 8), dtype=np.float32)
    # k = E with renormalisation is the full softmax, in pick order
    ids, w = route_topk(logits, None, 8)
    full = softmax(logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(full, ids, 1), rtol=1e-6)
    # renormalised top-k: weights sum to one and equal softmax over the picks
    ids, w = route_topk(logits, None, 2)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-6)
    picked = np.take_along_axis(logits.astype(np.float64), ids, 1)
    np.testing.assert_allclose(w, softmax(picked, axis=1), rtol=1e-6)
    assert np.all(w[:, 0] >= w[:, 1])
    # without renormalisation: the full softmax over all E at the picks
    ids0, w0 = route_topk(logits, None, 2, renormalize=False)
    assert np.array_equal(ids0, ids)
    np.testing.assert_allclose(w0, np.take_along_axis(full, ids, 1), rtol=1e-6)
    assert np.all(w0.sum(1) < 1.0)


def _brute_sort(ids, E):
    flat = ids.reshape(-1).tolist()
    order = [f for _, f in sorted((v, f) for f, v in enumerate(flat))]
    hist = [sum(1 for v in flat if v == e) for e in range(E)]
    offsets = [0]
    for h in hist:
        offsets.append(offsets[-1] + h)
    return order, offsets


@pytest.mark.parametrize("T,E,k,n_sent", [(64, 8, 2, 8), (50, 5, 3, 0), (31, 16, 4, 31 * 4),
                                          (128, 32, 4, 17), (1, 4, 4, 2)])
def test_sort_brute_force_and_invariants(T, E, k, n_sent):
    g = np.random.default_rng([T, E, k, n_sent])
    ids, _ = route_topk(g.standard_normal((T, E), dtype=np.float32), None, k)
    mask = np.zeros(T * k, np.uint8)
    mask[g.choice(T * k, n_sent, replace=False)] = 1
    ids = mark_sentinels(ids, mask, E)
    sr, rp, off = sort_by_expert(ids, E)
    order, offsets = _brute_sort(ids, E)
    assert sr.tolist() == order
    assert off.tolist() == offsets
    # invariants
    assert off[0] == 0 and np.all(np.diff(off) >= 0)
    assert off[E] == T * k - n_sent == int((ids != E).sum())
    assert np.array_equal(np.sort(sr), np.arange(T * k))
    assert np.array_equal(rp[sr], np.arange(T * k))
    flat = ids.reshape(-1)
    for e in range(E):
        seg = sr[off[e]:off[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)          # within an expert: token order
    assert np.all(flat[sr[off[E]:]] == E)       # sentinels last, in flat order
    assert np.all(np.diff(sr[off[E]:]) > 0)


def test_sentinels_not_clamped_onto_last_expert():
    # the replaced behaviour clamped the sentinel id to E-1; the last expert's
    # count must hold only its real rows
    wl = synth.WORKLOADS["tiny-8e-top2"]
    ids, _ = route_topk(synth.router_logits(wl), None, wl.k)
    real_last = int((ids == wl.E - 1).sum())
    ids_s = mark_sentinels(ids, synth.sentinel_mask(wl), wl.E)
    _, _, off = sort_by_expert(ids_s, wl.E)
    assert off[wl.E] == wl.R - wl.n_sentinel
    assert off[wl.E] - off[wl.E - 1] == int((ids_s == wl.E - 1).sum()) <= real_last
    clamped = np.minimum(ids_s, wl.E - 1)
    assert int((clamped == wl.E - 1).sum()) == off[wl.E] - off[wl.E - 1] + wl.n_sentinel
