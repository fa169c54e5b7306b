"""Seeded synthetic inputs for the Gated DeltaNet tail-replay workloads.

This module only draws random numbers. It holds none of the recurrence's
arithmetic, so both the CUDA path and the fp64 CPU oracle can take their
inputs from it without sharing any of the method.

The distributions stand in for the hidden states that a trained hybrid
model's linear-attention projections would produce on LongBench / RULER
prompts (the workloads of "Tail-Replay: Escaping the Curse of Linear
Attention in Prefix Caching for Hybrid LLMs", section 4). No item of those
suites is used or needed:

* q, k: standard normal per element, then each (token, head) vector is
  divided by its Euclidean length (a uniform draw on the unit sphere), then
  rounded to the storage dtype.
* v: standard normal, rounded to the storage dtype.
* beta: sigmoid of a standard normal (always in (0, 1)).
* g = log(alpha): -softplus(N(0,1) + 2) * gate_scale, so alpha is in (0, 1]
  as the GDN gate requires.  gate_scale = 0.1 is the default; a "weak decay"
  variant uses 1e-3 so that chunk transitions do not underflow.

All arrays are numpy; values that the GPU stores in bf16 are returned as
float32 arrays holding exactly bf16-representable numbers, so the oracle can
widen them to fp64 without any rounding of its own.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

DTYPES = ("f32", "bf16")


def config_seed(config: int, layer: int = 0) -> int:
    """Seed of one (config, layer) pair: 1234 + 1000 * layer + config."""
    return 1234 + 1000 * layer + config


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even).

    Returns float32 values whose low 16 bits are zero. NaN/Inf never occur in
    the generated inputs.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).reshape(x.shape)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return round_to_bf16(x)
    raise ValueError(f"unknown dtype {dtype!r}")


def _unit_rows(rng: np.random.Generator, shape) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    n = np.sqrt(np.sum(x.astype(np.float64) ** 2, axis=-1, keepdims=True))
    return (x / n).astype(np.float32)


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, x)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


@dataclass
class ReplayInputs:
    """One batch of replay tails, packed along the token axis."""

    q: np.ndarray  # [T, h_k, d_k] float32 (dtype-representable)
    k: np.ndarray  # [T, h_k, d_k]
    v: np.ndarray  # [T, h_v, d_v]
    g: np.ndarray  # [T, h_v] float32, log of the gate alpha
    beta: np.ndarray  # [T, h_v] float32
    cu_seqlens: np.ndarray  # [n_seqs + 1] int32
    dtype: str
    S0: np.ndarray | None = None  # [n_seqs, h_v, d_v, d_k] float32 or None

    @property
    def n_seqs(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def h_k(self) -> int:
        return int(self.q.shape[1])

    @property
    def h_v(self) -> int:
        return int(self.v.shape[1])

    @property
    def d_k(self) -> int:
        return int(self.q.shape[2])

    @property
    def d_v(self) -> int:
        return int(self.v.shape[2])


def make_replay_inputs(
    lengths,
    h_k: int,
    h_v: int,
    d_k: int,
    d_v: int,
    dtype: str = "bf16",
    seed: int = 1234,
    gate_scale: float = 0.1,
    unit_qk: bool = True,
    with_S0: bool = False,
    S0_scale: float = 1.0,
) -> ReplayInputs:
    """Draw q, k, v, g, beta for len(lengths) packed sequences.

    ``unit_qk=False`` leaves q and k as raw normals (to exercise the in-kernel
    L2 normalisation).  ``with_S0`` adds a random fp32 initial state.
    """
    lengths = [int(n) for n in lengths]
    if any(n < 0 for n in lengths):
        raise ValueError("negative sequence length")
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    rng = np.random.Generator(np.random.PCG64(seed))
    if unit_qk:
        q = _unit_rows(rng, (T, h_k, d_k))
        k = _unit_rows(rng, (T, h_k, d_k))
    else:
        q = rng.standard_normal((T, h_k, d_k), dtype=np.float32)
        k = rng.standard_normal((T, h_k, d_k), dtype=np.float32)
    v = rng.standard_normal((T, h_v, d_v), dtype=np.float32)
    beta = _sigmoid(rng.standard_normal((T, h_v), dtype=np.float32)).astype(np.float32)
    g = (-_softplus(rng.standard_normal((T, h_v), dtype=np.float32) + 2.0) * gate_scale).astype(np.float32)
    S0 = None
    if with_S0:
        S0 = (rng.standard_normal((len(lengths), h_v, d_v, d_k), dtype=np.float32) * S0_scale).astype(np.float32)
    return ReplayInputs(
        q=_store(q, dtype), k=_store(k, dtype), v=_store(v, dtype), g=g, beta=beta,
        cu_seqlens=cu, dtype=dtype, S0=S0,
    )


def tail_length(prefix_len: int, ratio: float) -> int:
    """Replay tail of a matched prefix: the last ceil(ratio * prefix_len) tokens."""
    return int(math.ceil(ratio * prefix_len))


def varlen_tail_lengths(n_tails: int, seed: int, prefixes=(8192, 16384, 32768), lo=0.05, hi=0.10):
    """Tail lengths of concurrent cache hits: prefix L uniform over ``prefixes``,
    replay ratio uniform in [lo, hi], tail = ceil(ratio * L)."""
    rng = np.random.Generator(np.random.PCG64(seed ^ 0x5EED))
    Ls = rng.choice(np.asarray(prefixes), size=n_tails)
    rho = rng.uniform(lo, hi, size=n_tails)
    return [tail_length(int(L), float(r)) for L, r in zip(Ls, rho)]


# The five workloads, by name.  Sizes follow the method's own model shapes
# (Qwen-style GDN layers: 16 q/k heads shared by 32 v heads, head dim 128).
WORKLOADS = {
    "tiny": dict(lengths=[256], h_k=2, h_v=2, d_k=64, d_v=64, dtype="f32", config=0),
    "layer_r1638": dict(lengths=[1638], h_k=16, h_v=32, d_k=128, d_v=128, dtype="bf16", config=1),
    "layer_r3277": dict(lengths=[3277], h_k=16, h_v=32, d_k=128, d_v=128, dtype="bf16", config=1),
    "full_32k": dict(lengths=[32768], h_k=16, h_v=32, d_k=128, d_v=128, dtype="bf16", config=4),
}


def workload_inputs(name: str, layer: int = 0, **over) -> ReplayInputs:
    w = dict(WORKLOADS[name])
    w.update(over)
    cfg = w.pop("config")
    return make_replay_inputs(seed=config_seed(cfg, layer), **w)


def varlen_workload_inputs(layer: int, n_tails: int = 64, h_k: int = 16, h_v: int = 32, d: int = 128,
                           dtype: str = "bf16") -> ReplayInputs:
    """64 concurrent replay tails of one GDN layer (each layer its own seed)."""
    seed = config_seed(2, layer)
    lengths = varlen_tail_lengths(n_tails, seed)
    return make_replay_inputs(lengths, h_k, h_v, d, d, dtype=dtype, seed=seed)


def chunk_workload_inputs(layer: int = 0, n_chunks: int = 16, chunk_len: int = 2048, h_k: int = 16, h_v: int = 32,
                          d: int = 128, weak_decay: bool = False) -> ReplayInputs:
    """Isolated chunks of one layer for the chunk-operator / composition workload: ``n_chunks``
    chunks of ``chunk_len`` tokens in fp32, each chunk its own sequence of cu_seqlens.
    ``weak_decay`` scales the gates by 1e-3 instead of 0.1, so that the chunk transitions T_C do
    not underflow to zero in fp32."""
    return make_replay_inputs([chunk_len] * n_chunks, h_k, h_v, d, d, dtype="f32", seed=config_seed(3, layer),
                              gate_scale=1e-3 if weak_decay else 0.1)
