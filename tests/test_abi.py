"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every entry point that include/moe.h declares, and rejects bad arguments on
the host before anything is launched."""
import os
import re

import pytest
import torch

from grouped_gemm_serving_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    gbuild.build()
    from grouped_gemm_serving_gb300 import moe as m
    return m


# The rejection tests below pass small integers as device pointers: they
# check that the host-side checks refuse the call before anything is
# launched.  They run only where no kernel can launch (no GPU), so that a
# regression in the order of those checks fails an assertion instead of
# launching a kernel on a bogus address.
host_only = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="fake-pointer rejection tests run only without a GPU")


def _declared():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(moe):
    names = _declared()
    assert {"moe_route_sort", "moe_permute", "moe_act_quant_fp8", "moe_grouped_gemm", "moe_swiglu",
            "moe_combine", "moe_forward"} <= set(names)
    lib = moe.lib()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # the binding wraps every declared entry point under the same name
    assert all(hasattr(moe, n) for n in names)


def test_abi_version_and_status_strings(moe):
    assert moe.moe_abi_version() == 1
    for st in range(7):
        assert moe.moe_status_string(st) not in ("", "unknown status")


def test_workspace_sizes(moe):
    assert moe.moe_route_sort_workspace_size(0, 8, 2) == 0
    assert moe.moe_route_sort_workspace_size(64, 300, 2) == 0
    assert moe.moe_route_sort_workspace_size(8192, 128, 8) >= 32 * 129 * 4
    a = moe.forward_args(dtype=moe.MOE_BF16, T=4096, E=32, k=4, H=2880, I=2880, x=1 << 20, W1=1 << 21,
                         W2=1 << 22, out=1 << 23, logits=1 << 24)
    R = 4096 * 4
    fused = moe.moe_forward_workspace_size(a)
    assert fused >= R * 2880 * 2 * 3                  # permuted x, h and the down output
    gat = moe.forward_args(dtype=moe.MOE_BF16, T=4096, E=32, k=4, H=2880, I=2880, x=1 << 20, W1=1 << 21,
                           W2=1 << 22, out=1 << 23, logits=1 << 24, gather=True)
    assert moe.moe_forward_workspace_size(gat) == fused - R * 2880 * 2   # no permuted copy of x
    bad = moe.forward_args(dtype=moe.MOE_FP8_E4M3_B128, T=64, E=8, k=2, H=2880, I=2880, x=1 << 20,
                           W1=1 << 21, W2=1 << 22, out=1 << 23, logits=1 << 24)
    assert moe.moe_forward_workspace_size(bad) == 0   # FP8 needs multiples of 128 and scales


@host_only
@pytest.mark.parametrize("call", [
    # (function, args) that must fail host-side with MOE_ERR_INVALID_ARG
    ("moe_route_sort", (None, None, None, None, None, 0, 8, 2, 1, None, None, None, None, 0, None)),
    ("moe_route_sort", (16, None, None, 16, 16, 4, 300, 2, 1, 16, 16, 16, 16, 1 << 20, None)),
    ("moe_route_sort", (16, None, None, 16, 16, 4, 8, 9, 1, 16, 16, 16, 16, 1 << 20, None)),
    ("moe_route_sort", (17, None, None, 16, 16, 4, 8, 2, 1, 16, 16, 16, 16, 1 << 20, None)),
    ("moe_act_quant_fp8", (16, 4, 100, 16, 16, None)),
    ("moe_act_quant_fp8", (18, 4, 128, 16, 16, None)),
    ("moe_weight_quant_fp8", (16, 2, 64, 96, 16, 16, None)),
    ("moe_permute", (0, 16, None, 4, 12, 2, 16, 16, 8, 8, 16, 16, None)),
    ("moe_permute", (1, 16, None, 4, 128, 2, 16, 16, 8, 8, 16, 16, None)),
    ("moe_permute", (0, 16, None, 4, 16, 2, 16, 16, 8, 7, 16, 16, None)),
    ("moe_grouped_gemm", (0, 16, None, 16, None, 16, 300, 64, 64, 64, 0, 16, None, None)),
    ("moe_grouped_gemm", (0, 16, None, 16, None, 16, 8, 64, 60, 64, 0, 16, None, None)),
    ("moe_grouped_gemm", (1, 16, None, 16, None, 16, 8, 64, 256, 128, 0, 16, None, None)),
    ("moe_grouped_gemm", (1, 16, 16, 16, 16, 16, 8, 64, 256, 100, 0, 16, None, None)),
    ("moe_grouped_gemm", (1, 16, 16, 16, 16, 16, 8, 64, 192, 128, 1, 16, None, None)),
    ("moe_grouped_gemm", (0, 16, None, 16, None, 16, 8, 64, 256, 64, 7, 16, None, None)),
    # gathered A: no sorted_rows, no tokens, k = 0, x misaligned, FP8 K not a multiple of 128
    ("moe_grouped_gemm_gather", (0, 16, None, 4, 2, None, 16, None, 16, 8, 64, 64, 64, 0, 16, None, None)),
    ("moe_grouped_gemm_gather", (0, 16, None, 0, 2, 16, 16, None, 16, 8, 64, 64, 64, 0, 16, None, None)),
    ("moe_grouped_gemm_gather", (0, 16, None, 4, 0, 16, 16, None, 16, 8, 64, 64, 64, 0, 16, None, None)),
    ("moe_grouped_gemm_gather", (0, 18, None, 4, 2, 16, 16, None, 16, 8, 64, 64, 64, 0, 16, None, None)),
    ("moe_grouped_gemm_gather", (1, 16, 16, 4, 2, 16, 16, 16, 16, 8, 64, 256, 100, 0, 16, None, None)),
    # batched products: FP8 N not a multiple of 128, k > E, misaligned out
    ("moe_batched_matmul", (1, 16, 16, 4, 256, 16, 2, 16, 16, 8, 200, 16, 16, 1 << 20, None)),
    ("moe_batched_matmul", (0, 16, None, 4, 64, 16, 9, 16, None, 8, 64, 16, 16, 1 << 20, None)),
    ("moe_batched_matmul", (0, 16, None, 4, 64, 16, 2, 16, None, 8, 64, 18, 16, 1 << 20, None)),
    ("moe_swiglu", (16, 16, 8, 64, 12, 16, None)),
    ("moe_combine", (16, 16, 16, 16, 4, 2, 12, 8, 16, None)),
    ("moe_combine", (16, 16, 16, 16, 4, 40, 16, 64, 16, None)),
])
def test_host_side_argument_checks(moe, call):
    name, args = call
    assert getattr(moe.lib(), name)(*args) == moe.MOE_ERR_INVALID_ARG


@host_only
def test_bf16_quantising_epilogue_is_unsupported(moe):
    st = moe.lib().moe_grouped_gemm(0, 16, None, 16, None, 16, 8, 64, 256, 64, 2, 16, None, None)
    assert st == moe.MOE_ERR_UNSUPPORTED


@host_only
def test_gather_needs_whole_128_byte_k_blocks(moe):
    # bf16 K = 200 is 400 bytes per row: not a whole number of k-blocks
    st = moe.lib().moe_grouped_gemm_gather(0, 16, None, 4, 2, 16, 16, None, 16, 8, 64, 64, 200, 0, 16, None, None)
    assert st == moe.MOE_ERR_UNSUPPORTED


def test_forward_gathers_only_whole_k_blocks(moe):
    # H = 200 (bf16) cannot be gathered: the separate scatter's buffer is in the workspace
    kw = dict(dtype=moe.MOE_BF16, T=64, E=8, k=2, I=256, x=1 << 20, W1=1 << 21, W2=1 << 22, out=1 << 23,
              logits=1 << 24)
    odd = moe.moe_forward_workspace_size(moe.forward_args(H=200, gather=True, **kw))
    odd_sep = moe.moe_forward_workspace_size(moe.forward_args(H=200, **kw))
    assert odd == odd_sep
    gat = moe.moe_forward_workspace_size(moe.forward_args(H=256, gather=True, **kw))
    sep = moe.moe_forward_workspace_size(moe.forward_args(H=256, **kw))
    assert sep == gat + 64 * 2 * 256 * 2


@host_only
def test_workspace_too_small_is_reported(moe):
    st = moe.lib().moe_route_sort(16, None, None, 16, 16, 64, 8, 2, 1, 16, 16, 16, 16, 4, None)
    assert st == moe.MOE_ERR_WORKSPACE
    st = moe.lib().moe_batched_matmul(0, 16, None, 4, 64, 16, 2, 16, None, 8, 64, 16, 16, 4, None)
    assert st == moe.MOE_ERR_WORKSPACE


@host_only
def test_selftest_limit_is_checked_on_host(moe):
    assert moe.lib().moe_selftest_wait_timeout(0, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.lib().moe_selftest_wait_timeout(3_000_000_000, None) == moe.MOE_ERR_INVALID_ARG


@host_only
def test_noalloc_rejects_requests_beyond_its_scratch(moe):
    # E = 256, k = 8: 128 tokens per sort block, 257 counters each; 256 KiB of
    # counters hold 255 blocks, so 32768 tokens (256 blocks) are refused
    lib = moe.lib()
    st = lib.moe_route_sort_noalloc(16, None, None, 16, 16, 32768, 256, 8, 1, 16, 16, 16, None)
    assert st == moe.MOE_ERR_WORKSPACE
    st = lib.moe_route_sort_noalloc(16, None, None, 16, 16, 600000, 256, 8, 1, 16, 16, 16, None)
    assert st == moe.MOE_ERR_WORKSPACE
