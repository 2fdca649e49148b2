"""Seeded synthetic workloads for the Kimi-K3 shared-expert SwiGLU MLP.

This module only *draws inputs*: it holds the five workload shapes and a
counter-based Gaussian generator.  It contains none of the MLP arithmetic, so
both the CPU oracle side (tests, ``bench.py --impl reference``) and the CUDA
side draw identical bytes from it without sharing any of the method's code.

Generator (written from the published definitions, not from any library):
  * SplitMix64 (Vigna): value ``i`` of stream ``(seed, tensor_id)`` is the
    SplitMix64 output function applied to ``base + (i + 1) * 0x9E3779B97F4A7C15``
    where ``base`` is itself one SplitMix64 output of ``seed * 2**20 + tensor_id``.
  * Box-Muller: each pair of 64-bit outputs (a, b) gives two normals
    ``r*cos(2*pi*v)``, ``r*sin(2*pi*v)`` with ``r = sqrt(-2 ln u)``,
    ``u = ((a >> 11) + 1) / 2**53`` in (0, 1], ``v = (b >> 11) / 2**53``.
  * scale by sigma in fp64, round fp64 -> fp32 -> bf16 (both round-to-nearest-even).
    The double rounding only defines which bf16 inputs are drawn; it is not a
    step of the method.

Shapes follow the pages' workloads: hidden 7168 and shared intermediate 6144
("[Kimi-K3] Add option to shard the shared expert instead of replicating",
section "Problem"), the merged MLA q_a/kv_a projection of 2,112 x 7,168 at
TP16 ("[II] TP-shard Kimi MLA latent projections", section "Behavior"), and the
tiny tp=4 / hidden 16 / intermediate 12 / 3-tokens-per-rank equivalence case
(prhub analysis of vllm PR #50656, section "关键源码片段").
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids inside one seed's family of streams
TID_X, TID_GATE, TID_UP, TID_DOWN, TID_MERGED = 0, 1, 2, 3, 4


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, tensor_id: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([(seed * (1 << 20) + tensor_id) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix(s + _GAMMA)[0]


def splitmix64(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the stream ``(seed, tensor_id)``."""
    base = _stream_base(seed, tensor_id)
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix(base + idx * _GAMMA)


def _normal_pairs(seed: int, tensor_id: int, p0: int, p1: int) -> np.ndarray:
    two53 = float(1 << 53)
    raw = splitmix64(seed, tensor_id, 2 * p0, 2 * (p1 - p0))
    a = raw[0::2]
    b = raw[1::2]
    u = ((a >> np.uint64(11)).astype(np.float64) + 1.0) / two53
    v = (b >> np.uint64(11)).astype(np.float64) / two53
    r = np.sqrt(-2.0 * np.log(u))
    th = 2.0 * math.pi * v
    pair = np.empty((p1 - p0, 2), dtype=np.float64)
    pair[:, 0] = r * np.cos(th)
    pair[:, 1] = r * np.sin(th)
    return pair.reshape(-1)


def normal_f64(seed: int, tensor_id: int, n: int, chunk: int = 1 << 20) -> np.ndarray:
    """``n`` standard normals (fp64) from the Box-Muller pairs of the stream.

    Chunks are independent (the generator is counter based), so they are drawn
    on a thread pool; the result does not depend on the chunking.
    """
    out = np.empty(n, dtype=np.float64)
    npairs = (n + 1) // 2

    def work(p0: int) -> None:
        p1 = min(npairs, p0 + chunk)
        flat = _normal_pairs(seed, tensor_id, p0, p1)
        lo = 2 * p0
        hi = min(n, 2 * p1)
        out[lo:hi] = flat[: hi - lo]

    starts = list(range(0, npairs, chunk))
    if len(starts) <= 1:
        for s in starts:
            work(s)
    else:
        with ThreadPoolExecutor(max_workers=min(len(starts), os.cpu_count() or 1)) as ex:
            list(ex.map(work, starts))
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round-to-nearest-even (NaN kept quiet)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def gaussian_bf16(seed: int, tensor_id: int, shape, sigma: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0, sigma^2) draws, row-major ``shape``."""
    n = int(np.prod(shape))
    z = normal_f64(seed, tensor_id, n)
    if sigma != 1.0:
        z *= sigma
    return f32_to_bf16_bits(z.astype(np.float32)).reshape(shape)


# --------------------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "mlp" | "sharded" | "merged" (which entry points it drives)
    T: int                    # tokens (gathered)
    H: int                    # hidden
    I: int = 0                # intermediate (MLP kinds)
    tp: int = 1               # emulated tensor-parallel shards
    weight_seed: int = 0
    x_seed: int = 0
    unit_sigma_weights: bool = False   # N(0,1) weights instead of N(0, 1/fan_in)
    partial_dtype: str = "bf16"        # "bf16" | "f32" (sharded kinds)
    q_dim: int = 0            # merged projection: q_a rows
    kv_dim: int = 0           # merged projection: kv_a rows
    notes: str = field(default="", compare=False)

    @property
    def sigma_gate_up(self) -> float:
        return 1.0 if self.unit_sigma_weights else 1.0 / math.sqrt(self.H)

    @property
    def sigma_down(self) -> float:
        return 1.0 if self.unit_sigma_weights else 1.0 / math.sqrt(self.I)


TINY_SHARDED = Workload(
    "tiny_sharded_tp4", "sharded", T=12, H=16, I=12, tp=4, weight_seed=0, x_seed=0,
    unit_sigma_weights=True, partial_dtype="f32",
    notes="tp=4, hidden 16, intermediate 12 (3 per shard), 12 tokens (3 per shard); N(0,1)")
DECODE_T64 = Workload(
    "decode_t64", "mlp", T=64, H=7168, I=6144, weight_seed=1, x_seed=1,
    notes="shared-expert layer at decode, T=64")
TP8_EMULATED = Workload(
    "tp8_emulated_t128", "sharded", T=128, H=7168, I=6144, tp=8, weight_seed=1, x_seed=3,
    partial_dtype="bf16",
    notes="decode weights split into 8 intermediate slices of 768; 16 tokens per shard")
MLA_MERGED = Workload(
    "mla_merged_tp16_t128", "merged", T=128, H=7168, tp=16, weight_seed=4, x_seed=4,
    q_dim=1536, kv_dim=576,
    notes="merged q_a/kv_a projection 2112x7168, TP16 column shards of 96+36")
PREFILL_T8192 = Workload(
    "prefill_t8192", "mlp", T=8192, H=7168, I=6144, weight_seed=2, x_seed=2,
    notes="shared-expert layer at prefill, T=8192")

WORKLOADS = [TINY_SHARDED, DECODE_T64, TP8_EMULATED, MLA_MERGED, PREFILL_T8192]
BY_NAME = {w.name: w for w in WORKLOADS}


def make_mlp_weights(w: Workload):
    """(w_gate_up [2I x H], w_down [H x I]) as bf16 bit patterns.

    The gate and up weights are drawn as two tensors and stacked gate-first, the
    layout a merged gate_up projection holds.
    """
    gate = gaussian_bf16(w.weight_seed, TID_GATE, (w.I, w.H), w.sigma_gate_up)
    up = gaussian_bf16(w.weight_seed, TID_UP, (w.I, w.H), w.sigma_gate_up)
    down = gaussian_bf16(w.weight_seed, TID_DOWN, (w.H, w.I), w.sigma_down)
    return np.concatenate([gate, up], axis=0), down


def make_x(w: Workload, T: int | None = None) -> np.ndarray:
    T = w.T if T is None else T
    return gaussian_bf16(w.x_seed, TID_X, (T, w.H), 1.0)


def make_merged_weight(w: Workload) -> np.ndarray:
    rows = w.q_dim + w.kv_dim
    sigma = 1.0 if w.unit_sigma_weights else 1.0 / math.sqrt(w.H)
    return gaussian_bf16(w.weight_seed, TID_MERGED, (rows, w.H), sigma)


def make_custom(seed: int, tensor_id: int, shape, sigma: float = 1.0) -> np.ndarray:
    """Free-form draw for edge-case tests (ragged shapes)."""
    return gaussian_bf16(seed, tensor_id, shape, sigma)
