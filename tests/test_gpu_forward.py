"""GPU parity of the whole layer (moe_forward) against the oracle on small
layers, in bf16 and FP8, with device and host buffers.

Error measure for layer outputs: per token row, max |y - y_ref| / max |y_ref|
against the fp32 oracle, at most 2e-2 (bf16) and 4e-2 (FP8); rows whose
reference is exactly zero (all slots sentinel) must be exactly zero."""
import numpy as np
import pytest
import torch

import oracle
from grouped_gemm_serving_gb300 import synth
from tests.gpu_helpers import dev, dev_bf16, host, host_f32_from_bf16, require_gpu, row_rel_err

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "fp8": 4e-2}


@pytest.fixture(scope="module")
def moe():
    require_gpu()
    from grouped_gemm_serving_gb300 import moe as m
    return m


def quantised_weights(moe, W):
    """bf16 bits [E, N, K] -> device e4m3 + scales through the library's quantiser."""
    E, N, K = W.shape
    q = torch.empty((E, N, K), dtype=torch.uint8, device="cuda")
    s = torch.empty((E, (N + 127) // 128, K // 128), dtype=torch.float32, device="cuda")
    moe.moe_weight_quant_fp8(dev_bf16(W), E, N, K, q, s)
    return q, s


def run_forward(moe, wl, x, W1, W2, W1s=None, W2s=None, host_io=False, logits=None, bias=None, mask=None):
    fp8 = W1s is not None
    T, H = wl.T, wl.H
    ids = torch.empty((T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, wl.k), dtype=torch.float32, device="cuda")
    if host_io:
        # a pinned output is written in place by the combine (or, with
        # MOE_FWD_STAGED_OUT, copied back like a pageable one); inputs are
        # copied in through the workspace
        pin = (lambda t: t.pin_memory()) if host_io != "pageable" else (lambda t: t.clone())
        xin = pin(torch.from_numpy(x.view(np.int16)))
        lin = pin(torch.from_numpy(logits))
        out = pin(torch.empty((T, H), dtype=torch.int16))
    else:
        xin, lin = dev_bf16(x), dev(logits)
        out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    a = moe.forward_args(dtype=moe.MOE_FP8_E4M3_B128 if fp8 else moe.MOE_BF16, T=T, E=wl.E, k=wl.k, H=H,
                         I=wl.I, x=xin, W1=W1, W2=W2, W1_scales=W1s, W2_scales=W2s, out=out, logits=lin,
                         expert_bias=None if bias is None else dev(bias),
                         sentinel_mask=None if mask is None else dev(mask), topk_ids=ids, topk_w=w,
                         renormalize=wl.renormalize, host_io=bool(host_io), staged_out=host_io == "pinned-staged")
    nbytes = moe.moe_forward_workspace_size(a)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    moe.moe_forward(a, ws, nbytes)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    y = out.view(torch.bfloat16).float().cpu().numpy() if host_io else host_f32_from_bf16(out.view(torch.bfloat16))
    return y, host(ids), host(w)


LAYERS = [
    synth.WORKLOADS["tiny-8e-top2"],
    synth.Workload("mid-16e-top4", T=300, E=16, k=4, H=256, I=384, n_sentinel=40, bias="normal0.5"),
    synth.Workload("ragged-12e-top3", T=97, E=12, k=3, H=136, I=200, n_sentinel=5),
    # a larger batch: several token tiles per expert, ragged rows (17
    # vectors), 400 sentinel slots
    synth.Workload("large-16e-top4", T=3000, E=16, k=4, H=136, I=200, n_sentinel=400, bias="normal0.5"),
]


@pytest.mark.parametrize("wl", LAYERS, ids=lambda w: w.name)
def test_forward_bf16(moe, wl):
    x, W1, W2 = synth.hidden_states(wl), synth.expert_weights(wl, "w1"), synth.expert_weights(wl, "w2")
    logits, bias, mask = synth.router_logits(wl), synth.expert_bias(wl), synth.sentinel_mask(wl)
    ref = oracle.moe_forward(x, W1, W2, E=wl.E, k=wl.k, logits=logits, bias=bias, sentinel_mask=mask)
    y, ids, w = run_forward(moe, wl, x, dev_bf16(W1), dev_bf16(W2), logits=logits, bias=bias, mask=mask)
    assert np.array_equal(ids, ref["ids"])
    err = row_rel_err(y, ref["out"])
    assert err.max() <= TOL["bf16"], err.max()
    dead = (ref["ids"] == wl.E).all(axis=1)
    assert np.all(y[dead] == 0)


@pytest.mark.parametrize("wl", [LAYERS[0], synth.Workload("fp8-16e-top4", T=200, E=16, k=4, H=256, I=384,
                                                          n_sentinel=30)], ids=lambda w: w.name)
def test_forward_fp8(moe, wl):
    x, W1, W2 = synth.hidden_states(wl), synth.expert_weights(wl, "w1"), synth.expert_weights(wl, "w2")
    logits, mask = synth.router_logits(wl), synth.sentinel_mask(wl)
    q1, s1 = oracle.quant_weight_fp8(W1)
    q2, s2 = oracle.quant_weight_fp8(W2)
    ref = oracle.moe_forward(x, q1, q2, W1_scales=s1, W2_scales=s2, E=wl.E, k=wl.k, logits=logits,
                             sentinel_mask=mask)
    dq1, ds1 = quantised_weights(moe, W1)
    dq2, ds2 = quantised_weights(moe, W2)
    assert np.array_equal(host(dq1), q1) and np.array_equal(host(ds2), s2)
    y, ids, _ = run_forward(moe, wl, x, dq1, dq2, ds1, ds2, logits=logits, mask=mask)
    assert np.array_equal(ids, ref["ids"])
    err = row_rel_err(y, ref["out"])
    assert err.max() <= TOL["fp8"], err.max()


@pytest.mark.parametrize("memory", ["pinned", "pinned-staged", "pageable"])
def test_forward_host_io_equals_device_path(moe, memory):
    wl = LAYERS[1]
    x, W1, W2 = synth.hidden_states(wl), synth.expert_weights(wl, "w1"), synth.expert_weights(wl, "w2")
    logits = synth.router_logits(wl)
    d1, d2 = dev_bf16(W1), dev_bf16(W2)
    y_dev, _, _ = run_forward(moe, wl, x, d1, d2, logits=logits)
    y_host, _, _ = run_forward(moe, wl, x, d1, d2, logits=logits, host_io=memory)
    assert np.array_equal(y_dev, y_host)
    y_again, _, _ = run_forward(moe, wl, x, d1, d2, logits=logits)
    assert np.array_equal(y_dev, y_again)                     # bit-reproducible


@pytest.mark.parametrize("memory", ["pinned", "pinned-staged", "pageable"])
def test_fp8_forward_host_io_equals_device_path(moe, memory):
    wl = synth.Workload("fp8-host-io", T=150, E=8, k=2, H=256, I=256, n_sentinel=9, dtype="fp8")
    x, W1, W2 = synth.hidden_states(wl), synth.expert_weights(wl, "w1"), synth.expert_weights(wl, "w2")
    logits, mask = synth.router_logits(wl), synth.sentinel_mask(wl)
    q1, s1 = oracle.quant_weight_fp8(W1)
    q2, s2 = oracle.quant_weight_fp8(W2)
    w = (dev(q1), dev(q2), dev(s1), dev(s2))
    y_dev, _, _ = run_forward(moe, wl, x, w[0], w[1], w[2], w[3], logits=logits, mask=mask)
    y_host, _, _ = run_forward(moe, wl, x, w[0], w[1], w[2], w[3], logits=logits, mask=mask, host_io=memory)
    assert np.array_equal(y_dev, y_host)


def test_expert_parallel_shards_on_one_gpu(moe):
    """Expert parallelism ("Mixture of Experts in transformers"): two shards of
    E/2 experts each, run one after the other through moe_forward with local
    ids (picks of the other shard's experts become sentinels); their partial
    outputs summed on the host equal the unsharded layer."""
    wl = synth.Workload("ep-16e-top4", T=256, E=16, k=4, H=256, I=384, n_sentinel=20)
    x, W1, W2 = synth.hidden_states(wl), synth.expert_weights(wl, "w1"), synth.expert_weights(wl, "w2")
    logits, mask = synth.router_logits(wl), synth.sentinel_mask(wl)
    ref = oracle.moe_forward(x, W1, W2, E=wl.E, k=wl.k, logits=logits, sentinel_mask=mask)
    ids, w = ref["ids"], ref["w"]
    total = np.zeros((wl.T, wl.H), np.float64)
    E_loc = wl.E // 2
    for r in range(2):
        lo = r * E_loc
        ids_loc = np.where((ids >= lo) & (ids < lo + E_loc), ids - lo, E_loc).astype(np.int32)
        out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
        ids_d, w_d = dev(ids_loc), dev(w)
        a = moe.forward_args(dtype=moe.MOE_BF16, T=wl.T, E=E_loc, k=wl.k, H=wl.H, I=wl.I, x=dev_bf16(x),
                             W1=dev_bf16(W1[lo:lo + E_loc]), W2=dev_bf16(W2[lo:lo + E_loc]), out=out,
                             topk_ids=ids_d, topk_w=w_d)
        n = moe.moe_forward_workspace_size(a)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        moe.moe_forward(a, ws, n)
        assert moe.moe_get_device_error() == 0
        total += host_f32_from_bf16(out)
    err = row_rel_err(total, ref["out"])
    assert err.max() <= TOL["bf16"], err.max()
    dead = (ids == wl.E).all(axis=1)
    assert np.all(total[dead] == 0)


@pytest.mark.parametrize("fp8", [False, True])
def test_forward_is_bit_reproducible(moe, fp8):
    """Every result is the same, bit for bit, from run to run: no floating-point
    atomics, fixed reduction orders.  Two runs of a layer with sentinels and a
    skewed routing (several token tiles per expert) compare byte for byte."""
    wl = synth.Workload("repro-16e-top4", T=1500, E=16, k=4, H=256, I=384, n_sentinel=60, bias="normal0.5")
    x, logits, bias, mask = (synth.hidden_states(wl), synth.router_logits(wl), synth.expert_bias(wl),
                             synth.sentinel_mask(wl))
    W1, W2 = synth.expert_weights(wl, "w1"), synth.expert_weights(wl, "w2")
    if fp8:
        (q1, s1), (q2, s2) = quantised_weights(moe, W1), quantised_weights(moe, W2)
        args = (q1, q2, s1, s2)
    else:
        args = (dev_bf16(W1), dev_bf16(W2))
    runs = [run_forward(moe, wl, x, *args, logits=logits, bias=bias, mask=mask) for _ in range(3)]
    for y, ids, w in runs[1:]:
        assert np.array_equal(y.view(np.uint32), runs[0][0].view(np.uint32))
        assert np.array_equal(ids, runs[0][1])
        assert np.array_equal(w.view(np.uint32), runs[0][2].view(np.uint32))


@pytest.mark.parametrize("staged_out", [False, True])
def test_host_io_calls_alternating_two_streams(moe, staged_out):
    """A serving loop through the host path: batches alternate over two streams
    (a workspace and pinned buffers each), which the library chains in call
    order.  Every batch's output equals the device-buffer call on its input."""
    wl = LAYERS[1]
    W1, W2 = dev_bf16(synth.expert_weights(wl, "w1")), dev_bf16(synth.expert_weights(wl, "w2"))
    logits = synth.router_logits(wl)
    xs = [synth.hidden_states(wl)]
    xs.append((xs[0].view(np.uint16) ^ np.uint16(0x8000)).view(xs[0].dtype))   # the same batch negated
    want = [run_forward(moe, wl, x, W1, W2, logits=logits)[0] for x in xs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs, args, wss = [], [], []
    for i in range(2):
        x_pin = torch.from_numpy(xs[i].view(np.int16)).pin_memory()
        l_pin = torch.from_numpy(logits).pin_memory()
        out = torch.empty((wl.T, wl.H), dtype=torch.int16).pin_memory()
        a = moe.forward_args(dtype=moe.MOE_BF16, T=wl.T, E=wl.E, k=wl.k, H=wl.H, I=wl.I, x=x_pin, W1=W1, W2=W2,
                             out=out, logits=l_pin, renormalize=wl.renormalize, host_io=True, staged_out=staged_out)
        n = moe.moe_forward_workspace_size(a)
        outs.append(out)
        args.append(a)
        wss.append((torch.empty(n, dtype=torch.uint8, device="cuda"), n))
    torch.cuda.synchronize()
    for b in range(6):
        i = b & 1
        outs[i].fill_(11)
        with torch.cuda.stream(streams[i]):
            moe.moe_forward(args[i], *wss[i])
        streams[i].synchronize()
        got = outs[i].view(torch.bfloat16).float().numpy()
        assert np.array_equal(got, want[i]), b
    # now back to back, without waiting in between
    for b in range(6):
        i = b & 1
        with torch.cuda.stream(streams[i]):
            moe.moe_forward(args[i], *wss[i])
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    for i in range(2):
        assert np.array_equal(outs[i].view(torch.bfloat16).float().numpy(), want[i])


@pytest.mark.parametrize("host_io", [False, True])
def test_forward_captured_in_a_cuda_graph(moe, host_io):
    """moe_forward enqueues no host synchronisation, so it can be captured
    into a CUDA graph (the host path takes the library's copy stream into the
    capture); replays give the eager call's output bit for bit."""
    wl = LAYERS[1]
    x = synth.hidden_states(wl)
    W1, W2 = dev_bf16(synth.expert_weights(wl, "w1")), dev_bf16(synth.expert_weights(wl, "w2"))
    logits = synth.router_logits(wl)
    want, _, _ = run_forward(moe, wl, x, W1, W2, logits=logits)
    if host_io:
        xin = torch.from_numpy(x.view(np.int16)).pin_memory()
        lin = torch.from_numpy(logits).pin_memory()
        out = torch.empty((wl.T, wl.H), dtype=torch.int16).pin_memory()
    else:
        xin, lin = dev_bf16(x), dev(logits)
        out = torch.empty((wl.T, wl.H), dtype=torch.int16, device="cuda")
    a = moe.forward_args(dtype=moe.MOE_BF16, T=wl.T, E=wl.E, k=wl.k, H=wl.H, I=wl.I, x=xin, W1=W1, W2=W2,
                         out=out, logits=lin, renormalize=wl.renormalize, host_io=host_io)
    n = moe.moe_forward_workspace_size(a)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        moe.moe_forward(a, ws, n)                     # warm-up outside the capture
        with torch.cuda.graph(g, stream=side):
            moe.moe_forward(a, ws, n)
    torch.cuda.synchronize()
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        got = out.view(torch.bfloat16).float().cpu().numpy()
        assert np.array_equal(got, want)
    assert moe.moe_get_device_error() == 0
