"""Pins of the oracle's layer: a float64 per-token expert loop (the "eager"
backend of "Mixture of Experts in transformers": loop over each token's
chosen experts), a dense SwiGLU MLP through torch when E = 1 and k = 1,
scatter followed by gather being the identity, and the sentinel rules of the
transformers MoE/FP8 write-up (sentinel rows excluded, their outputs zero)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from grouped_gemm_serving_gb300 import synth
from grouped_gemm_serving_gb300.synth import bf16_bits_to_f32


def _eager(x, W1, W2, ids, w, E):
    """Per token, per picked expert: w * down(silu(gate(x)) * up(x)), float64."""
    T, k = ids.shape
    I = W2.shape[2]
    out = np.zeros((T, x.shape[1]))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            if e == E:
                continue
            y1 = W1[e] @ x[t]
            g, u = y1[:I], y1[I:]
            out[t] += w[t, j] * (W2[e] @ (g / (1 + np.exp(-g)) * u))
    return out


def _rel(a, b):
    return np.abs(a - b).max() / np.abs(b).max()


@pytest.mark.parametrize("name_or_shape", ["tiny-8e-top2", (40, 4, 4, 128, 128, 3), (30, 16, 3, 64, 96, 0)])
def test_layer_matches_eager_loop(name_or_shape):
    if isinstance(name_or_shape, str):
        wl = synth.WORKLOADS[name_or_shape]
    else:
        T, E, k, H, I, ns = name_or_shape
        wl = synth.Workload("t", T=T, E=E, k=k, H=H, I=I, n_sentinel=ns)
    x, W1, W2 = (synth.hidden_states(wl), synth.expert_weights(wl, "w1"),
                 synth.expert_weights(wl, "w2"))
    r = oracle.moe_forward(x, W1, W2, E=wl.E, k=wl.k, logits=synth.router_logits(wl),
                           bias=synth.expert_bias(wl), sentinel_mask=synth.sentinel_mask(wl))
    ref = _eager(bf16_bits_to_f32(x).astype(np.float64), bf16_bits_to_f32(W1).astype(np.float64),
                 bf16_bits_to_f32(W2).astype(np.float64), r["ids"], r["w"].astype(np.float64), wl.E)
    assert _rel(r["out"], ref) < 1e-6
    assert (r["ids"] == wl.E).sum() == wl.n_sentinel


def test_dense_mlp_special_case():
    # E = 1, k = 1: every token goes to the one expert with weight 1
    wl = synth.Workload("dense", T=48, E=1, k=1, H=64, I=160)
    x, W1, W2 = (synth.hidden_states(wl), synth.expert_weights(wl, "w1"),
                 synth.expert_weights(wl, "w2"))
    r = oracle.moe_forward(x, W1, W2, E=1, k=1, logits=synth.router_logits(wl))
    assert np.all(r["w"] == 1.0)
    xt = torch.from_numpy(bf16_bits_to_f32(x)).double()
    w1 = torch.from_numpy(bf16_bits_to_f32(W1[0])).double()
    w2 = torch.from_numpy(bf16_bits_to_f32(W2[0])).double()
    ref = (F.silu(xt @ w1[:160].T) * (xt @ w1[160:].T)) @ w2.T
    assert _rel(r["out"], ref.numpy()) < 1e-6


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_scatter_then_gather_is_identity(k):
    wl = synth.Workload("id", T=37, E=16, k=k, H=256, I=128, n_sentinel=0)
    x = synth.hidden_states(wl)
    ids, _ = oracle.route_topk(synth.router_logits(wl), None, k)
    sr, rp, off = oracle.sort_by_expert(ids, wl.E)
    xp = oracle.permute(x, k, sr, int(off[-1]))
    w = np.full((wl.T, k), 1.0 / k, np.float32)
    out = oracle.combine(bf16_bits_to_f32(xp), ids, w, rp, wl.E)
    assert np.array_equal(out, bf16_bits_to_f32(x))


def test_sentinel_rows_are_zero_and_do_not_disturb_live_tokens():
    wl = synth.Workload("s", T=24, E=4, k=2, H=128, I=128)
    x, W1, W2 = (synth.hidden_states(wl), synth.expert_weights(wl, "w1"),
                 synth.expert_weights(wl, "w2"))
    ids, w = oracle.route_topk(synth.router_logits(wl), None, wl.k)
    base = oracle.moe_forward(x, W1, W2, E=wl.E, k=wl.k, ids=ids, w=w)
    mask = np.zeros(wl.R, np.uint8)
    mask[[2 * 3, 2 * 3 + 1, 2 * 10]] = 1          # token 3 fully, token 10 partly unrouted
    ids_s = oracle.mark_sentinels(ids, mask, wl.E)
    r = oracle.moe_forward(x, W1, W2, E=wl.E, k=wl.k, ids=ids_s, w=w)
    assert np.all(r["out"][3] == 0.0)
    live = [t for t in range(wl.T) if t not in (3, 10)]
    assert np.array_equal(r["out"][live], base["out"][live])
    # token 10 keeps only its second slot
    _, rp, off = oracle.sort_by_expert(ids, wl.E)
    assert r["offsets"][-1] == wl.R - 3
    # grouped GEMM rows past the live ones are exactly zero even for NaN inputs
    A = synth.to_bf16_bits(np.random.default_rng(0).standard_normal((wl.R, wl.H)).astype(np.float32))
    L = int(r["offsets"][-1])
    A[L:] = synth.BF16_NAN
    Y = oracle.grouped_gemm_bf16(A, W1, r["offsets"])
    assert np.all(Y[L:] == 0.0) and np.all(np.isfinite(Y[:L]))


def test_fp8_gemm_equals_bf16_gemm_on_representable_values():
    # e4m3 values are exact in bf16: with unit scales both grouped GEMMs agree
    g = np.random.default_rng(4)
    E, M, N, K = 3, 50, 96, 256
    qa = g.integers(0, 256, size=(M, K), dtype=np.uint8)
    qb = g.integers(0, 256, size=(E, N, K), dtype=np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0
    qb[(qb & 0x7F) == 0x7F] = 0
    off = np.array([0, 20, 20, 45], np.int32)
    ones_a = np.ones((M, K // 128), np.float32)
    ones_b = np.ones((E, 1, K // 128), np.float32)
    y8 = oracle.grouped_gemm_fp8(qa, ones_a, qb, ones_b, off)
    a16 = synth.to_bf16_bits(oracle.e4m3_decode(qa))
    b16 = synth.to_bf16_bits(oracle.e4m3_decode(qb))
    y16 = oracle.grouped_gemm_bf16(a16, b16, off)
    np.testing.assert_allclose(y8, y16, rtol=1e-6, atol=1e-3)
    assert np.all(y8[45:] == 0.0)
    # scales multiply per (row, 128-column group) and per (128-row, 128-col) block
    sa = g.uniform(0.5, 2, size=(M, K // 128)).astype(np.float32)
    sb = g.uniform(0.5, 2, size=(E, 1, K // 128)).astype(np.float32)
    ys = oracle.grouped_gemm_fp8(qa, sa, qb, sb, off)
    da, db = oracle.e4m3_decode(qa).astype(np.float64), oracle.e4m3_decode(qb).astype(np.float64)
    for p in (0, 19, 20, 44):
        e = 0 if p < 20 else 2
        a = da[p] * np.repeat(sa[p], 128)
        b = db[e] * np.repeat(sb[e, 0], 128)[None, :]
        np.testing.assert_allclose(ys[p], b @ a, rtol=1e-5, atol=1e-2)


def test_fp8_layer_close_to_bf16_layer():
    wl = synth.WORKLOADS["tiny-8e-top2"]
    x, W1, W2 = (synth.hidden_states(wl), synth.expert_weights(wl, "w1"),
                 synth.expert_weights(wl, "w2"))
    kw = dict(E=wl.E, k=wl.k, logits=synth.router_logits(wl), sentinel_mask=synth.sentinel_mask(wl))
    ref = oracle.moe_forward(x, W1, W2, **kw)["out"]
    q1, s1 = oracle.quant_weight_fp8(W1)
    q2, s2 = oracle.quant_weight_fp8(W2)
    out8 = oracle.moe_forward(x, q1, q2, W1_scales=s1, W2_scales=s2, **kw)["out"]
    rel = np.abs(out8 - ref).max(1) / np.maximum(np.abs(ref).max(1), 1e-30)
    live = np.abs(ref).max(1) > 0
    # two e4m3 roundings (2^-4 relative each) on operands and on h
    assert rel[live].max() < 0.2 and np.median(rel[live]) < 0.1 and np.all(out8[~live] == 0)


@pytest.mark.parametrize("k", [1, 3, 8])
def test_permute_moves_fp8_rows_and_their_scales_by_token(k):
    # the scale rows follow the byte rows: xs[p] = s[sorted_rows[p] // k], and
    # rows at or past L (sentinels sort last) are not written
    wl = synth.Workload("ps", T=45, E=12, k=k, H=384, I=128, n_sentinel=min(9, 45 * k - 1))
    q, s = oracle.quant_act_fp8(synth.hidden_states(wl))
    ids, _ = oracle.route_topk(synth.router_logits(wl), None, k)
    ids = oracle.mark_sentinels(ids, synth.sentinel_mask(wl), wl.E)
    sr, _, off = oracle.sort_by_expert(ids, wl.E)
    L = int(off[-1])
    assert L == wl.R - wl.n_sentinel
    xp, xs = oracle.permute(q, k, sr, L, x_scales=s)
    tok = sr[:L] // k
    assert np.array_equal(xp[:L], q[tok]) and np.array_equal(xs[:L], s[tok])
    assert not np.any(xp[L:]) and not np.any(xs[L:])
    # the scale rows are those of the tokens, not of the slots
    if k > 1:
        assert not np.array_equal(xs[:L], s[np.minimum(sr[:L], wl.T - 1)])


def _torch_e4m3_bits(v):
    """e4m3 codes of fp32 values through PyTorch's float8_e4m3fn conversion
    (round to nearest even).  A quotient v / (amax / 448) can exceed 448 by an
    ulp or so when the scale rounded down; below 464, the midpoint to the next
    (NaN) code, PyTorch rounds it to 448 like a saturating conversion."""
    v = np.ascontiguousarray(v, np.float32)
    assert np.all(np.abs(v) < 464.0)
    return torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_e4m3_values(q):
    return torch.from_numpy(np.ascontiguousarray(q, np.uint8)).view(torch.float8_e4m3fn).float() \
        .numpy().astype(np.float64)


def _quant_rows(v32):
    """Per row and 128-column group: s = amax / 448 in fp32 (1 for a zero
    group), codes of v / s (fp32 division) through PyTorch's e4m3 codec."""
    M, K = v32.shape
    g = v32.reshape(M, K // 128, 128)
    amax = np.abs(g).max(axis=2)
    s = np.where(amax == 0, np.float32(1.0), amax / np.float32(448.0)).astype(np.float32)
    return _torch_e4m3_bits((g / s[..., None]).reshape(M, K)), s


def _block_scaled_matvec(a_codes, sa, w_codes, sw):
    """sum_kb (sa[kb] * sw[n // 128, kb]) * (exact e4m3 partial of block kb),
    blocks in ascending order, float64."""
    N, K = w_codes.shape
    a = _torch_e4m3_values(a_codes)
    w = _torch_e4m3_values(w_codes)
    out = np.zeros(N)
    for kb in range(K // 128):
        part = w[:, kb * 128:(kb + 1) * 128] @ a[kb * 128:(kb + 1) * 128]
        scale = np.float64(sa[kb]) * sw[np.arange(N) // 128, kb].astype(np.float64)
        out += scale * part
    return out


def _fp8_eager(x_bits, q1, s1, q2, s2, ids, w, E, round_h=True):
    """The FP8 layer token by token, written from the method's description:
    x quantised per token per 128 columns; for every picked expert a
    block-scaled gate_up product, silu(gate) * up, h rounded to bf16 and
    quantised the same way, a block-scaled down product, weighted sum over the
    picks.  Codecs through PyTorch, arithmetic in float64 (stored fp32 where
    the layer stores a tensor)."""
    T, k = ids.shape
    H = x_bits.shape[1]
    I = q2.shape[2]
    qx, sx = _quant_rows(bf16_bits_to_f32(x_bits))
    out = np.zeros((T, H), np.float32)
    for t in range(T):
        acc = np.zeros(H)
        for j in range(k):
            e = ids[t, j]
            if e == E:
                continue
            y1 = _block_scaled_matvec(qx[t], sx[t], q1[e], s1[e]).astype(np.float32)
            g, u = y1[:I].astype(np.float64), y1[I:].astype(np.float64)
            h = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
            if round_h:
                h = torch.from_numpy(h).to(torch.bfloat16).float().numpy()
            qh, sh = _quant_rows(h[None, :])
            y2 = _block_scaled_matvec(qh[0], sh[0], q2[e], s2[e]).astype(np.float32)
            acc += np.float64(w[t, j]) * y2.astype(np.float64)
        out[t] = acc.astype(np.float32)
    return out


@pytest.mark.parametrize("name_or_shape", ["tiny-8e-top2", (40, 6, 3, 256, 384, 7)])
def test_fp8_layer_matches_fp8_eager_loop(name_or_shape):
    if isinstance(name_or_shape, str):
        wl = synth.WORKLOADS[name_or_shape]
    else:
        T, E, k, H, I, ns = name_or_shape
        wl = synth.Workload("f8", T=T, E=E, k=k, H=H, I=I, n_sentinel=ns, dtype="fp8", bias="normal0.5")
    x, W1, W2 = (synth.hidden_states(wl), synth.expert_weights(wl, "w1"),
                 synth.expert_weights(wl, "w2"))
    q1, s1 = oracle.quant_weight_fp8(W1)
    q2, s2 = oracle.quant_weight_fp8(W2)
    r = oracle.moe_forward(x, q1, q2, W1_scales=s1, W2_scales=s2, E=wl.E, k=wl.k,
                           logits=synth.router_logits(wl), bias=synth.expert_bias(wl),
                           sentinel_mask=synth.sentinel_mask(wl))
    ref = _fp8_eager(x, q1, s1, q2, s2, r["ids"], r["w"], wl.E)
    live = np.abs(ref).max(1) > 0
    assert np.all(r["out"][~live] == 0.0)
    rel = np.abs(r["out"] - ref).max(1)[live] / np.abs(ref).max(1)[live]
    assert rel.max() < 1e-6, rel.max()
    # the loop tells the rounding of h apart: without it the layer moves by
    # far more than the tolerance above
    unrounded = _fp8_eager(x, q1, s1, q2, s2, r["ids"], r["w"], wl.E, round_h=False)
    drift = np.abs(unrounded - ref).max(1)[live] / np.abs(ref).max(1)[live]
    assert drift.max() > 1e-4
