"""GPU parity of routing + sort, FP8 quantisation, permute, SwiGLU and combine
against the CPU oracle, through the C ABI (the ctypes binding)."""
import numpy as np
import pytest
import torch

import oracle
from grouped_gemm_serving_gb300 import synth
from grouped_gemm_serving_gb300.synth import bf16_bits_to_f32
from tests.gpu_helpers import (assert_close_bf16, dev, dev_bf16, host, host_bf16_bits,
                               host_f32_from_bf16, require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    require_gpu()
    from grouped_gemm_serving_gb300 import moe as m
    return m


def _no_device_error(moe):
    assert moe.moe_get_device_error() == moe.MOE_DEVERR_NONE


# ---------------------------------------------------------------- routing + sort
ROUTE_CASES = [
    synth.WORKLOADS["tiny-8e-top2"],
    synth.WORKLOADS["32e-top4-h2880"],
    synth.WORKLOADS["128e-top8-h2048-zipf"],
    synth.WORKLOADS["256e-top8-h7168-fp8"],
    synth.Workload("odd", T=777, E=37, k=3, H=8, I=8, n_sentinel=50, bias="normal0.5"),
    synth.Workload("k1", T=300, E=5, k=1, H=8, I=8),
    synth.Workload("kE", T=33, E=16, k=16, H=8, I=8, n_sentinel=7),
    synth.Workload("norenorm", T=129, E=64, k=6, H=8, I=8, renormalize=False),
    synth.Workload("big-k", T=20, E=256, k=32, H=8, I=8),
]


def _check_route(moe, wl):
    logits, bias, mask = synth.router_logits(wl), synth.expert_bias(wl), synth.sentinel_mask(wl)
    ids, w = oracle.route_topk(logits, bias, wl.k, wl.renormalize)
    if mask is not None:
        ids = oracle.mark_sentinels(ids, mask, wl.E)
    sr, rp, off = oracle.sort_by_expert(ids, wl.E)
    r = moe.route_sort_t(wl.E, wl.k, logits=dev(logits), expert_bias=None if bias is None else dev(bias),
                         sentinel_mask=None if mask is None else dev(mask), renormalize=wl.renormalize)
    torch.cuda.synchronize()
    _no_device_error(moe)
    assert np.array_equal(host(r["ids"]), ids)
    assert np.array_equal(host(r["offsets"]), off)
    assert np.array_equal(host(r["sorted_rows"]), sr)
    assert np.array_equal(host(r["row_pos"]), rp)
    np.testing.assert_allclose(host(r["w"]), w, rtol=2e-6, atol=0)


@pytest.mark.parametrize("wl", ROUTE_CASES, ids=lambda w: w.name)
def test_route_sort_bit_exact(moe, wl):
    _check_route(moe, wl)


# Up to 1024 slots (T*k) form one sort block; one token more makes two.  Both
# sides of the one- and two-block boundaries, and a single token.
@pytest.mark.parametrize("T", [1, 3, 255, 256, 257, 511, 512, 513])
def test_route_sort_single_block_boundary(moe, T):
    _check_route(moe, synth.Workload(f"b{T}", T=T, E=16, k=4, H=8, I=8, n_sentinel=min(5, 4 * T - 1),
                                     bias="normal0.5"))


# A batch whose slots fit one sort block and whose routing work is small
# (tokens per warp x logits per lane <= 4) is routed and sorted by a single
# CTA: both sides of that limit for each logits-per-lane count.
@pytest.mark.parametrize("T,E,k", [(128, 32, 8), (129, 32, 4), (128, 8, 8), (64, 64, 8), (65, 64, 2),
                                   (32, 128, 8), (33, 128, 4), (1, 256, 8), (100, 200, 3)])
def test_route_sort_single_cta_boundary(moe, T, E, k):
    _check_route(moe, synth.Workload(f"c{T}-{E}-{k}", T=T, E=E, k=k, H=8, I=8, n_sentinel=min(7, T * k - 1),
                                     bias="normal0.5"))


@pytest.mark.parametrize("T", [500, 100])   # two-kernel and single-CTA paths
def test_route_ties_go_to_lower_expert(moe, T):
    g = np.random.default_rng(3)
    logits = g.integers(-1, 2, size=(T, 24)).astype(np.float32)   # heavy ties
    ids, w = oracle.route_topk(logits, None, 5)
    r = moe.route_sort_t(24, 5, logits=dev(logits))
    assert np.array_equal(host(r["ids"]), ids)
    np.testing.assert_allclose(host(r["w"]), w, rtol=2e-6)


def test_sort_of_given_ids_with_sentinels(moe):
    g = np.random.default_rng(4)
    T, E, k = 3000, 20, 4
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[g.random((T, k)) < 0.3] = E                          # many sentinels, some whole tokens
    ids[:10] = E
    sr, rp, off = oracle.sort_by_expert(ids, E)
    r = moe.route_sort_t(E, k, topk_ids=dev(ids))
    _no_device_error(moe)
    assert np.array_equal(host(r["sorted_rows"]), sr)
    assert np.array_equal(host(r["row_pos"]), rp)
    assert np.array_equal(host(r["offsets"]), off)
    assert host(r["offsets"])[-1] == (ids != E).sum()


@pytest.mark.parametrize("T,E,k", [(300, 20, 4), (64, 256, 8), (2, 3, 3)])
def test_sort_of_given_ids_with_sentinels_small(moe, T, E, k):
    g = np.random.default_rng(T + E)
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[g.random((T, k)) < 0.3] = E
    ids[0] = E                                               # a token with no live slot
    sr, rp, off = oracle.sort_by_expert(ids, E)
    r = moe.route_sort_t(E, k, topk_ids=dev(ids))
    _no_device_error(moe)
    assert np.array_equal(host(r["sorted_rows"]), sr)
    assert np.array_equal(host(r["row_pos"]), rp)
    assert np.array_equal(host(r["offsets"]), off)


def test_bad_expert_id_is_reported_not_placed(moe):
    ids = np.zeros((64, 2), np.int32)
    ids[:, 1] = 1
    ids[5, 0] = 99                                           # outside [0, E]
    r = moe.route_sort_t(8, 2, topk_ids=dev(ids))
    assert moe.moe_get_device_error() == moe.MOE_DEVERR_ROUTE
    sr = host(r["sorted_rows"])
    assert np.array_equal(np.sort(sr), np.arange(128))       # still a permutation
    assert host(r["offsets"])[-1] == 127                     # the bad slot sorts as a sentinel
    got = host(r["ids"])                                     # and reads as one in topk_ids
    assert got[5, 0] == 8 and np.array_equal(np.delete(got.reshape(-1), 10), np.delete(ids.reshape(-1), 10))


def test_route_never_picks_nan(moe):
    """A NaN logit is never picked; with at least k other values per token the
    picks and weights are those of the oracle with the NaNs at -inf."""
    g = np.random.default_rng(8)
    T, E, k = 300, 40, 4
    logits = g.standard_normal((T, E)).astype(np.float32)
    nan = g.random((T, E)) < 0.4
    nan[:, 5:5 + k] = False                                  # k finite values per token at least
    logits[nan] = np.nan
    ids, w = oracle.route_topk(np.where(nan, -np.inf, logits).astype(np.float32), None, k)
    r = moe.route_sort_t(E, k, logits=dev(logits))
    _no_device_error(moe)
    assert np.array_equal(host(r["ids"]), ids)
    np.testing.assert_allclose(host(r["w"]), w, rtol=2e-6)


def test_route_too_few_numbers_is_reported(moe):
    """A token with fewer than k non-NaN logits cannot be routed: the error is
    recorded and its unfilled slots sort as sentinels."""
    T, E, k = 64, 16, 4
    logits = np.random.default_rng(9).standard_normal((T, E)).astype(np.float32)
    logits[7, 2:] = np.nan                                   # two numbers for four picks
    r = moe.route_sort_t(E, k, logits=dev(logits))
    assert moe.moe_get_device_error() == moe.MOE_DEVERR_ROUTE
    assert np.array_equal(np.sort(host(r["sorted_rows"])), np.arange(T * k))
    assert host(r["offsets"])[-1] == T * k - 2
    assert set(host(r["ids"])[7, :2]) == {0, 1}
    assert np.all(host(r["ids"])[7, 2:] == E)               # unfilled picks read as sentinels


# ---------------------------------------------------------------- FP8 quantisation
def _act_inputs():
    g = np.random.default_rng(7)
    yield "normal", synth.dense_rows(333, 1024, 1)
    yield "odd-groups", synth.dense_rows(3, 384, 5)          # 9 groups: one half-warp idles
    yield "one-group", synth.dense_rows(1, 128, 6)
    heavy = g.standard_t(2, size=(64, 2048)).astype(np.float32) * 30
    heavy[3, :128] = 0                                       # an all-zero group
    heavy[4, 128:256] = 2.0 ** -100                          # subnormal codes only
    heavy[5, :] = g.normal(size=2048) * 1e-30
    yield "heavy", synth.to_bf16_bits(heavy)
    big = (g.normal(size=(8, 7168)) * 1e30).astype(np.float32)
    yield "huge", synth.to_bf16_bits(big)


@pytest.mark.parametrize("name,xb", list(_act_inputs()), ids=lambda v: v if isinstance(v, str) else "")
def test_act_quant_bit_exact(moe, name, xb):
    M, K = xb.shape
    q_ref, s_ref = oracle.quant_act_fp8(xb)
    q = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    s = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
    moe.moe_act_quant_fp8(dev_bf16(xb), M, K, q, s)
    assert np.array_equal(host(s).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(host(q), q_ref)


@pytest.mark.parametrize("E,N,K", [(2, 512, 256), (3, 200, 384), (1, 4096, 7168)])
def test_weight_quant_bit_exact(moe, E, N, K):
    wl = synth.Workload("wq", T=1, E=E, k=1, H=K, I=N // 2 if N % 2 == 0 else 1)
    w = np.stack([synth.to_bf16_bits(np.random.default_rng([e, N]).standard_normal((N, K), dtype=np.float32)
                                     * np.float32(0.02)) for e in range(E)])
    q_ref, s_ref = oracle.quant_weight_fp8(w)
    q = torch.empty((E, N, K), dtype=torch.uint8, device="cuda")
    s = torch.empty(s_ref.shape, dtype=torch.float32, device="cuda")
    moe.moe_weight_quant_fp8(dev_bf16(w), E, N, K, q, s)
    assert np.array_equal(host(s), s_ref)
    assert np.array_equal(host(q), q_ref)
    del wl


# ---------------------------------------------------------------- permute / combine
def _routing(T, E, k, n_sent, seed):
    wl = synth.Workload("p", T=T, E=E, k=k, H=8, I=8, n_sentinel=n_sent, seed=seed)
    ids, w = oracle.route_topk(synth.router_logits(wl), None, k)
    if n_sent:
        ids = oracle.mark_sentinels(ids, synth.sentinel_mask(wl), E)
    sr, rp, off = oracle.sort_by_expert(ids, E)
    return ids, w, sr, rp, off


@pytest.mark.parametrize("T,E,k,H,n_sent", [(64, 8, 2, 128, 8), (1000, 32, 4, 2880, 100), (257, 128, 8, 2048, 0)])
def test_permute_bf16_bit_exact(moe, T, E, k, H, n_sent):
    ids, w, sr, rp, off = _routing(T, E, k, n_sent, 1)
    x = synth.dense_rows(T, H, 2)
    R, L = T * k, int(off[-1])
    xp = torch.full((R, H), -7, dtype=torch.int16, device="cuda").view(torch.bfloat16)  # canary
    moe.moe_permute(moe.MOE_BF16, dev_bf16(x), None, T, H, k, dev(sr), dev(off), E, R, xp, None)
    _no_device_error(moe)
    got = host_bf16_bits(xp)
    assert np.array_equal(got[:L], oracle.permute(x, k, sr, L)[:L])
    assert np.all(got[L:].view(np.int16) == -7)              # rows >= L are not written


def test_permute_fp8_bytes_and_scales(moe):
    T, E, k, H = 500, 16, 4, 1024
    ids, w, sr, rp, off = _routing(T, E, k, 37, 2)
    q, s = oracle.quant_act_fp8(synth.dense_rows(T, H, 3))
    R, L = T * k, int(off[-1])
    xq_ref, xs_ref = oracle.permute(q, k, sr, L, x_scales=s)
    xp = torch.zeros((R, H), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((H // 128, R), dtype=torch.float32, device="cuda")   # group-major
    moe.moe_permute(moe.MOE_FP8_E4M3_B128, dev(q), dev(s), T, H, k, dev(sr), dev(off), E, R, xp, xs)
    _no_device_error(moe)
    assert np.array_equal(host(xp)[:L], xq_ref[:L])
    assert np.array_equal(host(xs).T[:L], xs_ref[:L])


# The first three take the row-split path (few tokens); the rest have a block
# of tokens per SM and take one warp per token, in both of its slot-group
# sizes (top-k up to 4, and above), with ragged row lengths.
@pytest.mark.parametrize("T,E,k,H,n_sent", [(64, 8, 2, 128, 8), (700, 32, 4, 2880, 90), (300, 128, 8, 2048, 0),
                                            (1300, 16, 1, 264, 50), (1300, 16, 3, 1032, 100),
                                            (1400, 64, 4, 2880, 200), (1300, 64, 5, 520, 0),
                                            (1250, 128, 8, 264, 300)])
def test_combine_matches_oracle(moe, T, E, k, H, n_sent):
    ids, w, sr, rp, off = _routing(T, E, k, n_sent, 5)
    R = T * k
    y2 = synth.dense_rows(R, H, 6)
    L = int(off[-1])
    y2[L:] = 0
    ref = oracle.combine(bf16_bits_to_f32(y2), ids, w, rp, E)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(dev_bf16(y2), dev(ids), dev(w), dev(rp), T, k, H, E, out)
    _no_device_error(moe)
    got = host_f32_from_bf16(out)
    assert_close_bf16(got, ref, rtol=2.0 ** -8, row_atol=1e-6)
    dead = (ids == E).all(axis=1)
    assert np.all(got[dead] == 0)


@pytest.mark.parametrize("T,k", [(400, 4), (1300, 1), (1300, 2), (1300, 4), (1300, 8)])
def test_permute_then_combine_is_identity(moe, T, k):
    E, H = 16, 512
    ids, _, sr, rp, off = _routing(T, E, k, 0, 9)
    x = synth.dense_rows(T, H, 10)
    xp = torch.empty((T * k, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(moe.MOE_BF16, dev_bf16(x), None, T, H, k, dev(sr), dev(off), E, T * k, xp, None)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    w = np.full((T, k), 1.0 / k, np.float32)
    moe.moe_combine(xp, dev(ids), dev(w), dev(rp), T, k, H, E, out)
    assert np.array_equal(host_bf16_bits(out), x)


def test_swiglu_matches_oracle(moe):
    M_cap, I, L = 1000, 768, 870
    E = 4
    off = np.array([0, 300, 300, 600, L], np.int32)
    y1 = synth.dense_rows(M_cap, 2 * I, 11, std=3.0)
    y1[L:] = synth.BF16_NAN
    ref = oracle.swiglu(bf16_bits_to_f32(y1), L)
    h = torch.full((M_cap, I), 5, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_swiglu(dev_bf16(y1), dev(off), E, M_cap, I, h)
    _no_device_error(moe)
    got = host_f32_from_bf16(h)
    assert_close_bf16(got[:L], ref[:L], rtol=2.0 ** -8, row_atol=1e-6)
    assert np.all(host_bf16_bits(h)[L:] == 0)


def test_invalid_offsets_are_rejected_on_device(moe):
    M_cap, I = 64, 64
    off = np.array([0, 10, 5, 70], np.int32)                 # decreasing and beyond M_cap
    y1 = torch.zeros((M_cap, 2 * I), dtype=torch.bfloat16, device="cuda")
    h = torch.full((M_cap, I), 3, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_swiglu(y1, dev(off), 3, M_cap, I, h)
    assert moe.moe_get_device_error() == moe.MOE_DEVERR_OFFSETS
    assert np.all(host_bf16_bits(h).view(np.int16) == 3)     # nothing written


def test_bounded_wait_times_out_and_context_survives(moe):
    # a wait on an mbarrier nothing arrives on gives up after 20 ms and
    # reports MOE_DEVERR_TIMEOUT; the next launches still work
    moe.moe_selftest_wait_timeout(20_000_000)
    assert moe.moe_get_device_error() == moe.MOE_DEVERR_TIMEOUT
    assert moe.moe_get_device_error() == moe.MOE_DEVERR_NONE     # read-and-clear
    r = moe.route_sort_t(8, 2, logits=torch.zeros((16, 8), device="cuda"))
    assert np.array_equal(host(r["offsets"])[[0, -1]], [0, 32])
