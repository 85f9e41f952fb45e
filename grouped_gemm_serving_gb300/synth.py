"""Seeded synthetic inputs for the MoE expert layer.

This module draws random numbers and nothing else: router logits, per-expert
routing biases, hidden states, stacked expert weights, sentinel slot masks and
the pre-permuted rows of the live-row sweep.  It holds none of the layer's
arithmetic (no routing, sorting, quantisation or GEMM), so that the CUDA path
and the CPU oracle can both be fed from it without sharing any of the method.

Every tensor comes from its own numpy ``default_rng`` stream keyed by
``(seed, tensor_id, expert)``, so large weight stacks can be drawn expert by
expert, in parallel, and a subset of experts can be regenerated on its own.

Floating point inputs are drawn in fp32 and stored as bf16 bit patterns
(``uint16``, round to nearest even), which is how the layer receives them.

Workload shapes follow the MoE layers described in "Mixture of Experts in
transformers" (sections on the basic MoE concept and on expert backends: a
router picks k of E experts per token; 32-expert top-4 as in gpt-oss-20b) and
the sentinel sweep of "Hugging Face Transformers: MoE and FP8 kernel
optimisation" (section 2, MoE sentinel handling: 16384 permuted rows with
100 % / 50 % / 12.5 % of them live).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import numpy as np

# stream ids: one per kind of tensor
_LOGITS, _BIAS, _X, _W1, _W2, _SENT, _SWEEP_A = 1, 2, 3, 4, 5, 6, 7

BF16_NAN = np.uint16(0x7FC0)


@dataclass(frozen=True)
class Workload:
    """One synthetic MoE layer.

    T tokens, E experts, top-k routing, hidden size H, expert intermediate I
    (gate_up weight ``[E, 2I, H]``, down weight ``[E, H, I]``).
    ``bias`` selects the per-expert routing bias: ``"none"``, ``"normal0.5"``
    (N(0, 0.5) per expert, skewed load) or ``"zipf1.1"`` (log of a Zipf(1.1)
    popularity over a random ranking of the experts).
    """

    name: str
    T: int
    E: int
    k: int
    H: int
    I: int
    dtype: str = "bf16"           # "bf16" or "fp8" (e4m3, 128-blocked scales)
    bias: str = "none"
    n_sentinel: int = 0           # slots marked unrouted (expert id = E)
    renormalize: bool = True      # top-k weights renormalised over the k picks
    x_std: float = 1.0
    w_std: float = 0.02
    seed: int = 0

    @property
    def R(self) -> int:
        """Number of routed slots, T*k (rows of the permuted buffers)."""
        return self.T * self.k

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # tiny layer: 64 tokens, 8 experts top-2, H=128, I=256, 8 sentinel slots
    "tiny-8e-top2": Workload("tiny-8e-top2", T=64, E=8, k=2, H=128, I=256, n_sentinel=8),
    # gpt-oss-like 32-expert top-4 layer, H = I = 2880, biased (skewed) routing
    "32e-top4-h2880": Workload("32e-top4-h2880", T=4096, E=32, k=4, H=2880, I=2880,
                               bias="normal0.5"),
    # 128-expert top-8, H=2048, I=768, Zipf(1.1) expert popularity
    "128e-top8-h2048-zipf": Workload("128e-top8-h2048-zipf", T=8192, E=128, k=8, H=2048,
                                     I=768, bias="zipf1.1"),
    # decode-sized batch of the same 32-expert layer: 64 tokens
    "32e-top4-h2880-t64": Workload("32e-top4-h2880-t64", T=64, E=32, k=4, H=2880, I=2880,
                                   bias="normal0.5"),
    # 256-expert top-8 fine-grained FP8 layer, H=7168, I=2048
    "256e-top8-h7168-fp8": Workload("256e-top8-h7168-fp8", T=4096, E=256, k=8, H=7168,
                                    I=2048, dtype="fp8"),
    # decode-sized batch of the FP8 layer: 64 tokens
    "256e-top8-h7168-fp8-t64": Workload("256e-top8-h7168-fp8-t64", T=64, E=256, k=8, H=7168,
                                        I=2048, dtype="fp8"),
}


def _rng(seed: int, tensor_id: int, index: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, tensor_id, index])


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), round to nearest even."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    out = ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)
    out[np.isnan(a)] = BF16_NAN
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact widening)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def router_logits(wl: Workload) -> np.ndarray:
    """Router logits, fp32 ``[T, E]``, N(0, 1)."""
    return _rng(wl.seed, _LOGITS).standard_normal((wl.T, wl.E), dtype=np.float32)


def expert_bias(wl: Workload):
    """Per-expert routing bias, fp32 ``[E]``, or None."""
    if wl.bias == "none":
        return None
    g = _rng(wl.seed, _BIAS)
    if wl.bias == "normal0.5":
        return (0.5 * g.standard_normal(wl.E)).astype(np.float32)
    if wl.bias == "zipf1.1":
        rank = g.permutation(wl.E) + 1          # expert e has popularity rank rank[e]
        return (-1.1 * np.log(rank.astype(np.float64))).astype(np.float32)
    raise ValueError(f"unknown bias kind {wl.bias!r}")


def hidden_states(wl: Workload) -> np.ndarray:
    """Token hidden states as bf16 bits ``[T, H]``, N(0, x_std)."""
    x = _rng(wl.seed, _X).standard_normal((wl.T, wl.H), dtype=np.float32)
    if wl.x_std != 1.0:
        x *= np.float32(wl.x_std)
    return to_bf16_bits(x)


def _weight_shape(wl: Workload, which: str):
    if which == "w1":
        return 2 * wl.I, wl.H
    if which == "w2":
        return wl.H, wl.I
    raise ValueError(which)


def expert_weight(wl: Workload, which: str, e: int) -> np.ndarray:
    """One expert's weight as bf16 bits: w1 ``[2I, H]`` (gate rows then up
    rows) or w2 ``[H, I]``; N(0, w_std)."""
    n, kdim = _weight_shape(wl, which)
    tid = _W1 if which == "w1" else _W2
    w = _rng(wl.seed, tid, e).standard_normal((n, kdim), dtype=np.float32)
    w *= np.float32(wl.w_std)
    return to_bf16_bits(w)


def expert_weights(wl: Workload, which: str, experts=None, threads: int | None = None,
                   out: np.ndarray | None = None) -> np.ndarray:
    """Stacked expert weights as bf16 bits ``[len(experts), N, K]``.

    ``experts`` defaults to all E; each expert's slice is drawn from its own
    stream, so any subset reproduces the same values as the full stack.
    """
    experts = list(range(wl.E)) if experts is None else list(experts)
    n, kdim = _weight_shape(wl, which)
    if out is None:
        out = np.empty((len(experts), n, kdim), dtype=np.uint16)
    threads = threads or min(16, os.cpu_count() or 1)

    def fill(i):
        out[i] = expert_weight(wl, which, experts[i])

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(fill, range(len(experts))))
    return out


def sentinel_mask(wl: Workload) -> np.ndarray | None:
    """uint8 ``[T*k]``: 1 marks a routed slot as a sentinel (unrouted/padded).

    ``n_sentinel`` distinct flat slots drawn without replacement."""
    if wl.n_sentinel == 0:
        return None
    m = np.zeros(wl.R, dtype=np.uint8)
    m[_rng(wl.seed, _SENT).choice(wl.R, wl.n_sentinel, replace=False)] = 1
    return m


# ---------------------------------------------------------------------------
# live-row sweep of the grouped GEMM: rows already in expert order


@dataclass(frozen=True)
class Sweep:
    """Grouped-GEMM sweep: ``M_cap`` permuted rows over E experts, of which
    the first ``live`` are routed, split equally over the experts; the rest are
    sentinel rows (NaN-poisoned on input, zero on output)."""

    M_cap: int = 16384
    E: int = 128
    H: int = 2048
    I: int = 768
    live: int = 16384
    seed: int = 0

    @property
    def workload(self) -> Workload:
        return Workload(f"sweep-{self.E}e-h{self.H}-m{self.M_cap}-live{self.live}",
                        T=self.M_cap, E=self.E, k=1, H=self.H, I=self.I, seed=self.seed)


def sweep_rows(sw: Sweep) -> np.ndarray:
    """Permuted activations, bf16 bits ``[M_cap, H]``: N(0,1) for live rows,
    bf16 NaN for every row at or beyond ``live``."""
    a = to_bf16_bits(_rng(sw.seed, _SWEEP_A).standard_normal((sw.M_cap, sw.H),
                                                              dtype=np.float32))
    a[sw.live:] = BF16_NAN
    return a


def sweep_offsets(sw: Sweep) -> np.ndarray:
    """int32 ``[E+1]`` expert boundaries with ``live // E`` rows per expert."""
    if sw.live % sw.E:
        raise ValueError("live rows must split equally over the experts")
    return (np.arange(sw.E + 1, dtype=np.int64) * (sw.live // sw.E)).astype(np.int32)


def grouped_offsets(E: int, live: int, seed: int = 0, empty_experts: int = 0) -> np.ndarray:
    """int32 ``[E+1]`` boundaries of ``live`` rows split at random over E
    experts (multinomial), with ``empty_experts`` of them forced to zero rows."""
    g = _rng(seed, _SWEEP_A, 1)
    p = g.random(E) + 0.05
    if empty_experts:
        p[g.choice(E, empty_experts, replace=False)] = 0.0
    counts = g.multinomial(live, p / p.sum())
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def grouped_rows(M_cap: int, K: int, live: int, seed: int = 0, std: float = 1.0) -> np.ndarray:
    """bf16 bits ``[M_cap, K]``: N(0, std) for the first ``live`` rows, NaN after."""
    a = _rng(seed, _SWEEP_A, 2).standard_normal((M_cap, K), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    a = to_bf16_bits(a)
    a[live:] = BF16_NAN
    return a


def dense_rows(M: int, K: int, seed: int, std: float = 1.0, tensor_id: int = 3) -> np.ndarray:
    """bf16 bits ``[M, K]`` N(0, std) -- generic activations for kernel tests."""
    a = _rng(seed, tensor_id, 17).standard_normal((M, K), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return to_bf16_bits(a)
