"""The allocation-free routing entry point, moe_route_sort_noalloc, for
callers that cannot allocate device memory themselves (a plug-in inside a
serving engine that owns the whole memory pool, or a hot path where an
allocation is not allowed).  It keeps its histogram in a static device array
inside the library; its results must equal moe_route_sort's on consecutive
calls, which also shows that every call clears the shared array it uses.
Kept in a late-sorting file so that it runs after every other test.  (Its
refusal of requests beyond the array is a host-side check, tested without a
GPU in test_abi.py.)"""
import numpy as np
import pytest
import torch

from grouped_gemm_serving_gb300 import synth
from tests.gpu_helpers import dev, host, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    require_gpu()
    from grouped_gemm_serving_gb300 import moe as m
    return m


def _outputs(wl):
    T, E, k = wl.T, wl.E, wl.k
    return dict(ids=torch.empty((T, k), dtype=torch.int32, device="cuda"),
                w=torch.empty((T, k), dtype=torch.float32, device="cuda"),
                sr=torch.empty(T * k, dtype=torch.int32, device="cuda"),
                rp=torch.empty(T * k, dtype=torch.int32, device="cuda"),
                off=torch.empty(E + 1, dtype=torch.int32, device="cuda"))


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(moe):
    cases = [synth.WORKLOADS["128e-top8-h2048-zipf"],
             synth.Workload("s", T=3000, E=37, k=3, H=8, I=8, n_sentinel=200, bias="normal0.5"),
             synth.WORKLOADS["tiny-8e-top2"]]
    for wl in cases:                      # consecutive calls reuse the one static array
        logits = dev(synth.router_logits(wl))
        bias = synth.expert_bias(wl)
        bias = None if bias is None else dev(bias)
        mask = synth.sentinel_mask(wl)
        mask = None if mask is None else dev(mask)
        ref, got = _outputs(wl), _outputs(wl)
        nws = moe.moe_route_sort_workspace_size(wl.T, wl.E, wl.k)
        ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
        moe.moe_route_sort(logits, bias, mask, ref["ids"], ref["w"], wl.T, wl.E, wl.k, 1, ref["sr"],
                           ref["rp"], ref["off"], ws, nws)
        for _ in range(2):
            moe.moe_route_sort_noalloc(logits, bias, mask, got["ids"], got["w"], wl.T, wl.E, wl.k, 1,
                                       got["sr"], got["rp"], got["off"])
            torch.cuda.synchronize()
            assert moe.moe_get_device_error() == 0
            for key in ref:
                assert np.array_equal(host(got[key]), host(ref[key])), (wl.name, key)

