"""GPU parity of the tcgen05 grouped GEMM (bf16 and block-scaled FP8; store,
SwiGLU and SwiGLU+FP8-quantising epilogues) against the CPU oracle.

Shapes span several row and column tiles with ragged tails: experts with 0,
a few and more than 128 rows, N and K that are not multiples of the tile,
sentinel rows NaN-poisoned on input and checked to be exact zeros on output."""
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


def _weights(E, N, K, seed, std=0.05):
    return np.stack([synth.dense_rows(N, K, seed * 1000 + e, std=std, tensor_id=4) for e in range(E)])


BF16_CASES = [
    # E, M_cap, live, N, K, empty experts
    (4, 300, 260, 264, 200, 1),
    (8, 1100, 1000, 512, 136, 2),
    (3, 129, 129, 256, 64, 0),
    (16, 2048, 1500, 2880, 256, 3),
]


@pytest.mark.parametrize("E,M_cap,live,N,K,n_empty", BF16_CASES)
def test_bf16_store(moe, E, M_cap, live, N, K, n_empty):
    off = synth.grouped_offsets(E, live, seed=E + K, empty_experts=n_empty)
    A = synth.grouped_rows(M_cap, K, live, seed=N)
    B = _weights(E, N, K, 1)
    ref = oracle.grouped_gemm_bf16(A, B, off)
    C = torch.full((M_cap, N), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm(moe.MOE_BF16, dev_bf16(A), None, dev_bf16(B), None, dev(off), E, M_cap, N, K,
                         moe.MOE_EPI_STORE, C, None)
    assert moe.moe_get_device_error() == 0
    got = host_f32_from_bf16(C)
    assert_close_bf16(got[:live], ref[:live])
    assert np.all(host_bf16_bits(C)[live:] == 0)


@pytest.mark.parametrize("E,M_cap,live,I,K,n_empty", [
    (4, 300, 260, 200, 200, 1), (8, 1100, 1000, 256, 128, 2), (5, 700, 640, 2880, 192, 0),
    (2, 256, 256, 72, 64, 0)])
def test_bf16_swiglu(moe, E, M_cap, live, I, K, n_empty):
    off = synth.grouped_offsets(E, live, seed=E * 7 + K, empty_experts=n_empty)
    A = synth.grouped_rows(M_cap, K, live, seed=I)
    B = _weights(E, 2 * I, K, 2)
    ref = oracle.swiglu(oracle.grouped_gemm_bf16(A, B, off), live)
    h = torch.full((M_cap, I), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm(moe.MOE_BF16, dev_bf16(A), None, dev_bf16(B), None, dev(off), E, M_cap, 2 * I, K,
                         moe.MOE_EPI_SWIGLU, h, None)
    assert moe.moe_get_device_error() == 0
    got = host_f32_from_bf16(h)
    assert_close_bf16(got[:live], ref[:live])
    assert np.all(host_bf16_bits(h)[live:] == 0)


def _fp8_operands(E, M_cap, live, N, K, seed):
    off = synth.grouped_offsets(E, live, seed=seed, empty_experts=1 if E > 2 else 0)
    A = synth.grouped_rows(M_cap, K, live, seed=seed + 1)
    A[live:] = 0                                      # quantisation of NaN rows is undefined
    qa, sa = oracle.quant_act_fp8(A)
    qb, sb = oracle.quant_weight_fp8(_weights(E, N, K, seed + 2))
    return off, qa, sa, qb, sb


@pytest.mark.parametrize("E,M_cap,live,N,K", [(4, 300, 260, 512, 256), (8, 1000, 900, 384, 512),
                                             (3, 200, 200, 264, 128)])
def test_fp8_store(moe, E, M_cap, live, N, K):
    off, qa, sa, qb, sb = _fp8_operands(E, M_cap, live, N, K, 5)
    ref = oracle.grouped_gemm_fp8(qa, sa, qb, sb, off)
    C = torch.full((M_cap, N), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm(moe.MOE_FP8_E4M3_B128, dev(qa), dev(np.ascontiguousarray(sa.T)), dev(qb), dev(sb),
                         dev(off), E, M_cap, N, K, moe.MOE_EPI_STORE, C, None)
    assert moe.moe_get_device_error() == 0
    got = host_f32_from_bf16(C)
    assert_close_bf16(got[:live], ref[:live], rtol=2.0 ** -7, row_atol=2e-3)
    assert np.all(host_bf16_bits(C)[live:] == 0)


@pytest.mark.parametrize("E,M_cap,live,I,K", [(4, 300, 260, 256, 256), (6, 900, 800, 384, 384)])
def test_fp8_swiglu_and_quantising_epilogue(moe, E, M_cap, live, I, K):
    off, qa, sa, qb, sb = _fp8_operands(E, M_cap, live, 2 * I, K, 9)
    ref_h = oracle.swiglu(oracle.grouped_gemm_fp8(qa, sa, qb, sb, off), live)
    args = (dev(qa), dev(np.ascontiguousarray(sa.T)), dev(qb), dev(sb), dev(off), E, M_cap, 2 * I, K)
    h = torch.empty((M_cap, I), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_gemm(moe.MOE_FP8_E4M3_B128, *args, moe.MOE_EPI_SWIGLU, h, None)
    hq = torch.full((M_cap, I), 7, dtype=torch.uint8, device="cuda")
    hs = torch.full((I // 128, M_cap), -1.0, dtype=torch.float32, device="cuda")
    moe.moe_grouped_gemm(moe.MOE_FP8_E4M3_B128, *args, moe.MOE_EPI_SWIGLU_QUANT_FP8, hq, hs)
    assert moe.moe_get_device_error() == 0
    got_h = host_f32_from_bf16(h)
    assert_close_bf16(got_h[:live], ref_h[:live], rtol=2.0 ** -7, row_atol=2e-3)
    # the fused quantisation equals the standalone quantiser applied to the
    # bf16 h of the SwiGLU epilogue (same accumulators, same rounding)
    q2 = torch.empty((M_cap, I), dtype=torch.uint8, device="cuda")
    s2 = torch.empty((M_cap, I // 128), dtype=torch.float32, device="cuda")
    moe.moe_act_quant_fp8(h, M_cap, I, q2, s2)
    assert np.array_equal(host(hq)[:live], host(q2)[:live])
    assert np.array_equal(host(hs).T[:live], host(s2)[:live])
    # against the oracle: dequantised h within the e4m3 rounding of the oracle's h
    deq = oracle.e4m3_decode(host(hq)).reshape(M_cap, I // 128, 128) * host(hs).T[:, :, None]
    assert_close_bf16(deq.reshape(M_cap, I)[:live], ref_h[:live], rtol=2.0 ** -4 + 2.0 ** -7, row_atol=4e-3)
    # sentinel rows: code 0 and scale 1
    assert np.all(host(hq)[live:] == 0) and np.all(host(hs).T[live:] == 1.0)


def test_invalid_offsets_skip_the_gemm(moe):
    E, M_cap, N, K = 4, 256, 256, 64
    off = np.array([0, 100, 90, 200, 250], np.int32)
    A = torch.zeros((M_cap, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((E, N, K), dtype=torch.bfloat16, device="cuda")
    C = torch.full((M_cap, N), 9, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm(moe.MOE_BF16, A, None, B, None, dev(off), E, M_cap, N, K, moe.MOE_EPI_STORE, C, None)
    assert moe.moe_get_device_error() == moe.MOE_DEVERR_OFFSETS
    assert np.all(host_bf16_bits(C).view(np.int16) == 9)


def test_deterministic(moe):
    E, M_cap, live, N, K = 8, 1100, 1000, 512, 256
    off = synth.grouped_offsets(E, live, seed=3)
    A, B = dev_bf16(synth.grouped_rows(M_cap, K, live, seed=4)), dev_bf16(_weights(E, N, K, 3))
    outs = []
    for _ in range(2):
        C = torch.empty((M_cap, N), dtype=torch.bfloat16, device="cuda")
        moe.moe_grouped_gemm(moe.MOE_BF16, A, None, B, None, dev(off), E, M_cap, N, K, moe.MOE_EPI_STORE, C, None)
        outs.append(host_bf16_bits(C))
    assert np.array_equal(outs[0], outs[1])


# bf16 runs with swapped operands on CTA pairs: an expert's tokens form
# ceil(cnt/256) equal tiles rounded up to 16 rows, each CTA loading half of a
# tile (8 to 128 rows) as one box of that height.  Expert sizes around those
# boundaries (1, 15-17, 31-33, 255-257, 512-513 rows, several tiles) for both
# epilogues, with an N tail and K not a multiple of the 64-element k-block;
# and one expert per box height (tiles of 16, 32, .., 256 rows).
PAIR_COUNTS = [1, 15, 16, 17, 31, 32, 33, 255, 256, 257, 512, 513, 700, 0, 1500]
BOX_COUNTS = [9, 17, 40, 50, 70, 90, 100, 120, 130, 150, 170, 180, 200, 220, 240, 250]


@pytest.mark.parametrize("counts", ["boundaries", "box_heights"])
@pytest.mark.parametrize("epi", ["store", "swiglu"])
def test_bf16_token_tile_boundaries(moe, epi, counts):
    counts = PAIR_COUNTS if counts == "boundaries" else BOX_COUNTS
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    live = int(off[-1])
    M_cap, K = live + 40, 200
    N = 392 if epi == "store" else 2 * 200
    A = synth.grouped_rows(M_cap, K, live, seed=77)
    B = _weights(E, N, K, 8)
    ref = oracle.grouped_gemm_bf16(A, B, off)
    if epi == "swiglu":
        ref = oracle.swiglu(ref, live)
    ncol = N if epi == "store" else N // 2
    C = torch.full((M_cap, ncol), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm(moe.MOE_BF16, dev_bf16(A), None, dev_bf16(B), None, dev(off), E, M_cap, N, K,
                         moe.MOE_EPI_STORE if epi == "store" else moe.MOE_EPI_SWIGLU, C, None)
    assert moe.moe_get_device_error() == 0
    got = host_f32_from_bf16(C)
    assert_close_bf16(got[:live], ref[:live])
    assert np.all(host_bf16_bits(C)[live:] == 0)


@pytest.mark.parametrize("epi", ["store", "swiglu"])
def test_bf16_256_experts(moe, epi):
    # the most experts the library takes (the tile prefix holds 8 per lane),
    # counts from 0 to 300 rows
    E, K = 256, 64
    counts = np.array([(37 * e) % 301 if e % 7 else 0 for e in range(E)], np.int64)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    live = int(off[-1])
    M_cap = live + 8
    N = 136 if epi == "store" else 2 * 72
    A = synth.grouped_rows(M_cap, K, live, seed=256)
    B = _weights(E, N, K, 11)
    ref = oracle.grouped_gemm_bf16(A, B, off)
    if epi == "swiglu":
        ref = oracle.swiglu(ref, live)
    ncol = N if epi == "store" else N // 2
    C = torch.full((M_cap, ncol), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm(moe.MOE_BF16, dev_bf16(A), None, dev_bf16(B), None, dev(off), E, M_cap, N, K,
                         moe.MOE_EPI_STORE if epi == "store" else moe.MOE_EPI_SWIGLU, C, None)
    assert moe.moe_get_device_error() == 0
    assert_close_bf16(host_f32_from_bf16(C)[:live], ref[:live])
    assert np.all(host_bf16_bits(C)[live:] == 0)


# The last store feature tile of an expert holds N mod 256 features; when
# that is at most 128 it runs as an M = 128 pair MMA.  N = 8 .. 384 puts 8,
# 64, 128, 8, 64 and 128 features there; N = 392 (136 features) is the
# M = 256 control.
@pytest.mark.parametrize("counts", ["boundaries", "box_heights"])
@pytest.mark.parametrize("N", [8, 64, 128, 264, 320, 384, 392])
def test_bf16_store_half_used_last_tile(moe, N, counts):
    counts = PAIR_COUNTS if counts == "boundaries" else BOX_COUNTS
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    live = int(off[-1])
    M_cap, K = live + 24, 128
    A = synth.grouped_rows(M_cap, K, live, seed=N + 3)
    B = _weights(E, N, K, 10)
    ref = oracle.grouped_gemm_bf16(A, B, off)
    C = torch.full((M_cap, N), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm(moe.MOE_BF16, dev_bf16(A), None, dev_bf16(B), None, dev(off), E, M_cap, N, K,
                         moe.MOE_EPI_STORE, C, None)
    assert moe.moe_get_device_error() == 0
    assert_close_bf16(host_f32_from_bf16(C)[:live], ref[:live])
    assert np.all(host_bf16_bits(C)[live:] == 0)


# The last SwiGLU feature tile of an expert holds I mod 128 features; when
# that is at most 64 it runs as an M = 128 pair MMA (its own accumulator
# layout, N rounded up to 32).  I = 8 .. 192 puts 8, 40, 64, 8, 56 and 64
# features there; I = 200 (72 features) is the M = 256 control.  Token counts
# cross the 16- and 32-rounding of N.
@pytest.mark.parametrize("counts", ["boundaries", "box_heights"])
@pytest.mark.parametrize("I", [8, 40, 64, 136, 184, 192, 200])
def test_bf16_swiglu_half_used_last_tile(moe, I, counts):
    counts = PAIR_COUNTS if counts == "boundaries" else BOX_COUNTS
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    live = int(off[-1])
    M_cap, K = live + 24, 128
    A = synth.grouped_rows(M_cap, K, live, seed=I + 5)
    B = _weights(E, 2 * I, K, 9)
    ref = oracle.swiglu(oracle.grouped_gemm_bf16(A, B, off), live)
    h = torch.full((M_cap, I), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm(moe.MOE_BF16, dev_bf16(A), None, dev_bf16(B), None, dev(off), E, M_cap, 2 * I, K,
                         moe.MOE_EPI_SWIGLU, h, None)
    assert moe.moe_get_device_error() == 0
    assert_close_bf16(host_f32_from_bf16(h)[:live], ref[:live])
    assert np.all(host_bf16_bits(h)[live:] == 0)


# FP8 tiles an expert's rows 128 at a time.  Expert sizes around those
# boundaries (and 15-17, 31-33 rows: warps whose 32 rows are partly or wholly
# past the expert's end), for all three epilogues, with several column tiles.
FP8_COUNTS = [1, 15, 16, 17, 31, 33, 127, 128, 129, 255, 256, 257, 300, 0, 520]


@pytest.mark.parametrize("epi", ["store", "swiglu", "swiglu_q"])
def test_fp8_token_tile_boundaries(moe, epi):
    E = len(FP8_COUNTS)
    off = np.concatenate([[0], np.cumsum(FP8_COUNTS)]).astype(np.int32)
    live = int(off[-1])
    M_cap, K = live + 40, 256
    N = 384 if epi == "store" else 2 * 256
    A = synth.grouped_rows(M_cap, K, live, seed=78)
    A[live:] = 0
    qa, sa = oracle.quant_act_fp8(A)
    qb, sb = oracle.quant_weight_fp8(_weights(E, N, K, 9))
    ref = oracle.grouped_gemm_fp8(qa, sa, qb, sb, off)
    args = (dev(qa), dev(np.ascontiguousarray(sa.T)), dev(qb), dev(sb), dev(off), E, M_cap, N, K)
    if epi == "store":
        C = torch.full((M_cap, N), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        moe.moe_grouped_gemm(moe.MOE_FP8_E4M3_B128, *args, moe.MOE_EPI_STORE, C, None)
        assert moe.moe_get_device_error() == 0
        assert_close_bf16(host_f32_from_bf16(C)[:live], ref[:live], rtol=2.0 ** -7, row_atol=2e-3)
        assert np.all(host_bf16_bits(C)[live:] == 0)
        return
    I = N // 2
    ref_h = oracle.swiglu(ref, live)
    h = torch.full((M_cap, I), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm(moe.MOE_FP8_E4M3_B128, *args, moe.MOE_EPI_SWIGLU, h, None)
    assert moe.moe_get_device_error() == 0
    assert_close_bf16(host_f32_from_bf16(h)[:live], ref_h[:live], rtol=2.0 ** -7, row_atol=2e-3)
    assert np.all(host_bf16_bits(h)[live:] == 0)
    if epi == "swiglu_q":
        hq = torch.full((M_cap, I), 7, dtype=torch.uint8, device="cuda")
        hs = torch.full((I // 128, M_cap), -1.0, dtype=torch.float32, device="cuda")
        moe.moe_grouped_gemm(moe.MOE_FP8_E4M3_B128, *args, moe.MOE_EPI_SWIGLU_QUANT_FP8, hq, hs)
        assert moe.moe_get_device_error() == 0
        q2 = torch.empty((M_cap, I), dtype=torch.uint8, device="cuda")
        s2 = torch.empty((M_cap, I // 128), dtype=torch.float32, device="cuda")
        moe.moe_act_quant_fp8(h, M_cap, I, q2, s2)
        assert np.array_equal(host(hq)[:live], host(q2)[:live])
        assert np.array_equal(host(hs).T[:live], host(s2)[:live])
        assert np.all(host(hq)[live:] == 0) and np.all(host(hs).T[live:] == 1.0)


# FP8 with experts of several token tiles and a row buffer far larger than
# the live rows: expert sizes around multiples of 128 and 256 (up to eight
# row tiles), empty experts, all three epilogues; and the live rows'
# results must not depend on M_cap.
FP8_WIDE_COUNTS = [1, 127, 128, 129, 255, 256, 257, 383, 384, 385, 511, 512, 513, 0, 1000, 0, 0, 0, 0, 0]


def _fp8_wide_case(epi, seed):
    E = len(FP8_WIDE_COUNTS)
    off = np.concatenate([[0], np.cumsum(FP8_WIDE_COUNTS)]).astype(np.int32)
    live = int(off[-1])
    M_cap, K = 256 * E + 64, 384
    assert M_cap >= live
    N = 384 if epi == "store" else 2 * 256
    A = synth.grouped_rows(M_cap, K, live, seed=seed)
    A[live:] = 0
    qa, sa = oracle.quant_act_fp8(A)
    qb, sb = oracle.quant_weight_fp8(_weights(E, N, K, seed + 1))
    return E, off, live, M_cap, N, K, qa, sa, qb, sb


@pytest.mark.parametrize("epi", ["store", "swiglu", "swiglu_q"])
def test_fp8_many_row_tiles(moe, epi):
    E, off, live, M_cap, N, K, qa, sa, qb, sb = _fp8_wide_case(epi, 81)
    ref = oracle.grouped_gemm_fp8(qa, sa, qb, sb, off)
    args = (dev(qa), dev(np.ascontiguousarray(sa.T)), dev(qb), dev(sb), dev(off), E, M_cap, N, K)
    if epi == "store":
        C = torch.full((M_cap, N), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        moe.moe_grouped_gemm(moe.MOE_FP8_E4M3_B128, *args, moe.MOE_EPI_STORE, C, None)
        assert moe.moe_get_device_error() == 0
        assert_close_bf16(host_f32_from_bf16(C)[:live], ref[:live], rtol=2.0 ** -7, row_atol=2e-3)
        assert np.all(host_bf16_bits(C)[live:] == 0)
        return
    I = N // 2
    ref_h = oracle.swiglu(ref, live)
    h = torch.full((M_cap, I), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm(moe.MOE_FP8_E4M3_B128, *args, moe.MOE_EPI_SWIGLU, h, None)
    assert moe.moe_get_device_error() == 0
    assert_close_bf16(host_f32_from_bf16(h)[:live], ref_h[:live], rtol=2.0 ** -7, row_atol=2e-3)
    assert np.all(host_bf16_bits(h)[live:] == 0)
    if epi == "swiglu_q":
        hq = torch.full((M_cap, I), 7, dtype=torch.uint8, device="cuda")
        hs = torch.full((I // 128, M_cap), -1.0, dtype=torch.float32, device="cuda")
        moe.moe_grouped_gemm(moe.MOE_FP8_E4M3_B128, *args, moe.MOE_EPI_SWIGLU_QUANT_FP8, hq, hs)
        assert moe.moe_get_device_error() == 0
        q2 = torch.empty((M_cap, I), dtype=torch.uint8, device="cuda")
        s2 = torch.empty((M_cap, I // 128), dtype=torch.float32, device="cuda")
        moe.moe_act_quant_fp8(h, M_cap, I, q2, s2)
        assert np.array_equal(host(hq)[:live], host(q2)[:live])
        assert np.array_equal(host(hs).T[:live], host(s2)[:live])
        assert np.all(host(hq)[live:] == 0) and np.all(host(hs).T[live:] == 1.0)


def test_fp8_live_rows_do_not_depend_on_m_cap(moe):
    E, off, live, M_cap, N, K, qa, sa, qb, sb = _fp8_wide_case("store", 91)
    outs = []
    for m in (M_cap, live):
        C = torch.empty((m, N), dtype=torch.bfloat16, device="cuda")
        moe.moe_grouped_gemm(moe.MOE_FP8_E4M3_B128, dev(qa[:m]), dev(np.ascontiguousarray(sa[:m].T)), dev(qb),
                             dev(sb), dev(off), E, m, N, K, moe.MOE_EPI_STORE, C, None)
        assert moe.moe_get_device_error() == 0
        outs.append(host_bf16_bits(C)[:live])
    assert np.array_equal(outs[0], outs[1])
