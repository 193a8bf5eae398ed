"""Seeded synthetic inputs for the Gated DeltaNet recurrence.

This module is shared by the CPU oracle tests and by the GPU tests and benchmark,
so that both sides see the same input bytes.  It holds no arithmetic of the
recurrence itself: only a counter-based random number generator, the input
distributions, the shapes of the workloads, and the rounding of values to the
storage dtype.

Generator
---------
SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; the 64-bit finaliser as published by S. Vigna).  Output
number ``i`` (0-based) of a generator seeded with ``s`` is ``mix(s + (i+1)*G)``
with ``G = 0x9E3779B97F4A7C15``, so any index can be drawn directly.  Every tensor
of a workload draws from its own stream: stream ``j`` uses indices
``j * 2**40 + i``.

Uniforms are ``((x >> 11) + 0.5) * 2**-53`` (never 0 or 1).  Normals come from
the Box-Muller transform (Box and Muller, 1958) on the pair of uniforms with
indices ``2p`` and ``2p+1``: ``r = sqrt(-2 ln u1)``, ``z[2p] = r cos(2 pi u2)``,
``z[2p+1] = r sin(2 pi u2)``.

Distributions (the workloads' recipe)
-------------------------------------
* q, k: N(0, 1), then each (token, head) vector is divided by its exact fp64
  Euclidean norm;
* v: N(0, 1);
* g = log(sigmoid(a)) = -softplus(-a) with a ~ N(3, 1), so the per-token decay
  exp(g) = sigmoid(a) lies in (0, 1);
* beta = sigmoid(b), b ~ N(0, 1);
* initial state: zeros, or N(0, sigma^2) with sigma = 0.1.

Draw order (stream index): q 0, k 1, v 2, a 3, b 4, S0 5.

Raw gate projections (for kernels that form the gates themselves): a_raw, b_raw ~ N(0, 1) in the
storage dtype (streams 6, 7); per value head A_log ~ N(-0.5, 0.5) and dt_bias ~ N(0, 0.5) in fp32
(streams 8, 9), which puts exp(A_log) and the decay in the ranges the handbook reports on real
input.  Output gate: z ~ N(0, 1) like the outputs (stream 10), norm weight ~ N(1, 0.1) fp32 per
value feature (stream 11).

Rounding to the storage dtype: fp64 -> fp32 round-to-nearest-even; for bf16 the
fp32 value is rounded again to bf16 (round-to-nearest-even on the fp32 bits).
Arrays are returned as float32 holding exactly the stored values, so a caller can
widen them to fp64 for the oracle or narrow them to bf16 for the GPU without any
further rounding.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os
from typing import Optional, Sequence

import numpy as np

__all__ = [
    "GOLDEN_GAMMA",
    "splitmix64",
    "uniforms",
    "normals",
    "round_to_dtype",
    "Workload",
    "WORKLOADS",
    "make_prefill_inputs",
    "make_decode_inputs",
    "unit_rows",
]

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_STRIDE = 1 << 40
_CHUNK = 1 << 22  # values generated per numpy batch (bounds temporary memory)

STREAM_Q, STREAM_K, STREAM_V, STREAM_A, STREAM_B, STREAM_S0 = range(6)
STREAM_RAW_A, STREAM_RAW_B, STREAM_A_LOG, STREAM_DT_BIAS = range(6, 10)
STREAM_Z, STREAM_NORM_W = range(10, 12)
STREAM_DOUT, STREAM_DSF = range(12, 14)


def splitmix64(seed: int, idx: np.ndarray) -> np.ndarray:
    """Outputs number ``idx`` (uint64 array) of SplitMix64 seeded with ``seed``."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (idx.astype(np.uint64) + np.uint64(1)) * GOLDEN_GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniforms(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """``count`` uniforms in (0, 1) from stream ``stream`` starting at index ``start``."""
    idx = np.arange(start, start + count, dtype=np.uint64) + np.uint64(stream * _STREAM_STRIDE)
    x = splitmix64(seed, idx)
    return ((x >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normals(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    """``count`` standard normals (fp64) of stream ``stream``, element ``start`` onwards."""
    out = np.empty(count, dtype=np.float64)
    done = 0
    while done < count:
        n = min(_CHUNK, count - done)
        e0 = start + done            # first normal index of this batch
        p0 = e0 // 2                 # first Box-Muller pair
        p1 = (e0 + n + 1) // 2       # one past the last pair
        u = uniforms(seed, stream, 2 * p0, 2 * (p1 - p0))
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        th = 2.0 * math.pi * u2
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(th)
        z[1::2] = r * np.sin(th)
        off = e0 - 2 * p0
        out[done:done + n] = z[off:off + n]
        done += n
    return out


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp64 values to ``dtype`` ('f32' or 'bf16'); returns float32 holding them."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == "f32":
        return f
    if dtype != "bf16":
        raise ValueError(f"unknown dtype {dtype!r}")
    bits = f.view(np.uint32)
    lsb = (bits >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        rounded = (bits + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return rounded.view(np.float32)


def unit_rows(x: np.ndarray) -> np.ndarray:
    """Divide each vector along the last axis by its exact fp64 Euclidean norm."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True))


def _parallel_slabs(total: int, slab: int, fn) -> None:
    """Run ``fn(start, stop)`` over ``[0, total)`` in slabs on a thread pool (numpy releases the GIL)."""
    starts = list(range(0, total, slab))
    if len(starts) <= 1:
        for s0 in starts:
            fn(s0, min(total, s0 + slab))
        return
    workers = min(len(starts), os.cpu_count() or 1, 32)
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(lambda s0: fn(s0, min(total, s0 + slab)), starts))


def _normal_tensor(seed, stream, shape, mean=0.0, std=1.0):
    n = int(np.prod(shape))
    return (mean + std * normals(seed, stream, n)).reshape(shape)


def _unit_tensor(seed, stream, shape, dtype):
    """Unit-norm rows generated and rounded in slabs to bound fp64 temporaries."""
    d = shape[-1]
    rows = int(np.prod(shape[:-1]))
    out = np.empty((rows, d), dtype=np.float32)
    slab = max(1, (_CHUNK // 4) // d)

    def fill(r0, r1):
        z = normals(seed, stream, (r1 - r0) * d, start=r0 * d).reshape(r1 - r0, d)
        out[r0:r1] = round_to_dtype(unit_rows(z), dtype)

    _parallel_slabs(rows, slab, fill)
    return out.reshape(shape)


def _rounded_normal(seed, stream, shape, dtype, mean=0.0, std=1.0):
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)

    def fill(s0, s1):
        out[s0:s1] = round_to_dtype(mean + std * normals(seed, stream, s1 - s0, start=s0), dtype)

    _parallel_slabs(n, _CHUNK // 4, fill)
    return out.reshape(shape)


def _log_sigmoid(a):
    # log(sigmoid(a)) = -softplus(-a), written to stay finite for large |a|
    return -(np.maximum(-a, 0.0) + np.log1p(np.exp(-np.abs(a))))


def _sigmoid(b):
    return 1.0 / (1.0 + np.exp(-b))


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shapes and distributions of one synthetic workload."""
    name: str
    kind: str                      # "prefill" or "decode"
    dtype: str                     # "f32" or "bf16": storage type of q, k, v, g, beta, out
    B: int                         # batch (prefill) or sequences (decode)
    T: int                         # tokens per sequence (prefill, total when packed) or steps (decode)
    Hqk: int
    Hv: int
    dk: int
    dv: int
    chunk: int = 64
    s0_std: float = 0.0            # 0 -> zero initial state
    seqlens: Optional[Sequence[int]] = None   # packed variable-length sequences (B must be 1)
    seed: int = 0

    @property
    def num_seqs(self) -> int:
        return len(self.seqlens) if self.seqlens is not None else self.B

    @property
    def cu_seqlens(self) -> Optional[np.ndarray]:
        if self.seqlens is None:
            return None
        return np.concatenate([[0], np.cumsum(self.seqlens)]).astype(np.int32)


WORKLOADS = {
    # small fp32 case: every parity check runs it in full
    "tiny_f32": Workload("tiny_f32", "prefill", "f32", B=1, T=64, Hqk=2, Hv=2, dk=32, dv=32, chunk=16),
    # 4-layer character-LM-sized heads (4 heads of 32), bf16 in / fp32 state
    "charlm_bf16": Workload("charlm_bf16", "prefill", "bf16", B=4, T=512, Hqk=4, Hv=4, dk=32, dv=32, chunk=64),
    # chunked prefill, 16 QK heads shared by 32 V heads of dim 128, random initial state
    "prefill_gqa_8k": Workload("prefill_gqa_8k", "prefill", "bf16", B=2, T=8192, Hqk=16, Hv=32, dk=128, dv=128,
                               chunk=64, s0_std=0.1),
    # long-context prefill: 4 packed sequences with state reset at each boundary
    "prefill_varlen_128k": Workload("prefill_varlen_128k", "prefill", "bf16", B=1, T=131072, Hqk=16, Hv=32,
                                    dk=128, dv=128, chunk=64, seqlens=(65536, 32768, 24576, 8192)),
    # recurrent decode: 256 sequences x 32 V heads, 512 consecutive steps, fp32 state resident on the device
    "decode_256x512": Workload("decode_256x512", "decode", "bf16", B=256, T=512, Hqk=16, Hv=32, dk=128, dv=128,
                               s0_std=0.1),
}


def make_prefill_inputs(w: Workload, with_s0: bool = True):
    """Inputs of a prefill workload, as float32 arrays holding the stored values.

    Returns dict with q, k [B, T, Hqk, dk]; v [B, T, Hv, dv]; g, beta [B, T, Hv];
    S0 [num_seqs, Hv, dk, dv] (fp32 state, or None when zero); cu_seqlens (int32 or None).
    """
    B, T = w.B, w.T
    q = _unit_tensor(w.seed, STREAM_Q, (B, T, w.Hqk, w.dk), w.dtype)
    k = _unit_tensor(w.seed, STREAM_K, (B, T, w.Hqk, w.dk), w.dtype)
    v = _rounded_normal(w.seed, STREAM_V, (B, T, w.Hv, w.dv), w.dtype)
    a = _normal_tensor(w.seed, STREAM_A, (B, T, w.Hv), mean=3.0)
    b = _normal_tensor(w.seed, STREAM_B, (B, T, w.Hv))
    g = round_to_dtype(_log_sigmoid(a), w.dtype)
    beta = round_to_dtype(_sigmoid(b), w.dtype)
    S0 = None
    if with_s0 and w.s0_std > 0:
        S0 = _rounded_normal(w.seed, STREAM_S0, (w.num_seqs, w.Hv, w.dk, w.dv), "f32", std=w.s0_std)
    return dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0, cu_seqlens=w.cu_seqlens)


def make_decode_inputs(w: Workload, steps: Optional[int] = None):
    """Inputs of a decode workload: per-step q, k [steps, N, Hqk, dk], v [steps, N, Hv, dv],
    g, beta [steps, N, Hv], and the initial fp32 state S0 [N, Hv, dk, dv]."""
    steps = w.T if steps is None else steps
    N = w.B
    q = _unit_tensor(w.seed, STREAM_Q, (steps, N, w.Hqk, w.dk), w.dtype)
    k = _unit_tensor(w.seed, STREAM_K, (steps, N, w.Hqk, w.dk), w.dtype)
    v = _rounded_normal(w.seed, STREAM_V, (steps, N, w.Hv, w.dv), w.dtype)
    a = _normal_tensor(w.seed, STREAM_A, (steps, N, w.Hv), mean=3.0)
    b = _normal_tensor(w.seed, STREAM_B, (steps, N, w.Hv))
    g = round_to_dtype(_log_sigmoid(a), w.dtype)
    beta = round_to_dtype(_sigmoid(b), w.dtype)
    if w.s0_std > 0:
        S0 = _rounded_normal(w.seed, STREAM_S0, (N, w.Hv, w.dk, w.dv), "f32", std=w.s0_std)
    else:
        S0 = np.zeros((N, w.Hv, w.dk, w.dv), dtype=np.float32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0)


def scaled(w: Workload, **changes) -> Workload:
    """A copy of ``w`` with some fields changed (smaller shapes for quick checks)."""
    return dataclasses.replace(w, **changes)


def make_raw_gates(w: Workload, lead_shape=None):
    """Raw gate projections a, b [*lead_shape, Hv] (rounded to the workload dtype) and per-head
    A_log, dt_bias [Hv] fp32.  lead_shape defaults to (B, T)."""
    lead = (w.B, w.T) if lead_shape is None else tuple(lead_shape)
    a = _rounded_normal(w.seed, STREAM_RAW_A, (*lead, w.Hv), w.dtype)
    b = _rounded_normal(w.seed, STREAM_RAW_B, (*lead, w.Hv), w.dtype)
    A_log = round_to_dtype(_normal_tensor(w.seed, STREAM_A_LOG, (w.Hv,), mean=-0.5, std=0.5), "f32")
    dt_bias = round_to_dtype(_normal_tensor(w.seed, STREAM_DT_BIAS, (w.Hv,), std=0.5), "f32")
    return dict(a=a, b=b, A_log=A_log, dt_bias=dt_bias)


def make_output_gate(w: Workload, out_shape):
    """Output-gate inputs: z shaped like the outputs (workload dtype) and norm_weight [dv] fp32."""
    z = _rounded_normal(w.seed, STREAM_Z, tuple(out_shape), w.dtype)
    norm_w = round_to_dtype(_normal_tensor(w.seed, STREAM_NORM_W, (w.dv,), mean=1.0, std=0.1), "f32")
    return dict(z=z, norm_weight=norm_w)


def make_backward_inputs(w: Workload):
    """Upstream gradients for the backward pass: dout like the outputs (workload dtype), N(0,1), and
    dS_final like the final states (fp32), N(0, 0.1^2)."""
    dout = _rounded_normal(w.seed, STREAM_DOUT, (w.B, w.T, w.Hv, w.dv), w.dtype)
    dSf = _rounded_normal(w.seed, STREAM_DSF, (w.num_seqs, w.Hv, w.dk, w.dv), "f32", std=0.1)
    return dict(dout=dout, dSf=dSf)
