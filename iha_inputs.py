"""Seeded synthetic inputs for the Interleaved Head Attention forward pass.

This module only draws random numbers and arranges them into arrays of the
shapes the method consumes.  It holds none of the method's arithmetic, so both
the CUDA path (through its Python binding) and the fp64 oracle can be fed from
it without sharing any computation.

Generator: a counter-based SplitMix64 stream (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014), one stream per
(seed, tensor tag), element i taking counter i.  Uniforms on (0, 1) are the top
53 bits plus half an ulp; normals are Box-Muller pairs (element i uses uniforms
2i and 2i+1).  The draw is done in float64, scaled by the standard deviation,
rounded to float32 and, for bf16 workloads, rounded to bfloat16 (round to
nearest even).  Identical on every machine and NumPy version.

Value distributions (unit-variance mixed projections, O(1) attention scores):
  X ~ N(0, 1)          [B, N, D]
  W_Q, W_K, W_V ~ N(0, 1/D)          [D, H*d], column block m = W^(m)
  alpha_Q/K/V ~ N(0, 1/H)            [H(m), H(h), P(j)]
  R ~ N(0, 1/(H*P))                  [H, H*P], column h'*P + j
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TAG_MUL = np.uint64(0xD1B54A32D192ED03)

TAGS = {"X": 1, "W_Q": 2, "W_K": 3, "W_V": 4,
        "alpha_Q": 5, "alpha_K": 6, "alpha_V": 7, "R": 8}

MASK_NONE, MASK_CAUSAL, MASK_WINDOW = 0, 1, 2


def _splitmix64(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = x + _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, tag: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([np.uint64(seed) ^ (np.uint64(tag) * _TAG_MUL)], dtype=np.uint64)
        return _splitmix64(s)[0]


def uniform01(seed: int, tag: int, n: int, offset: int = 0) -> np.ndarray:
    """n uniforms on (0, 1) from stream (seed, tag), counters offset..offset+n-1."""
    base = _stream_base(seed, tag)
    ctr = np.arange(offset, offset + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        u = _splitmix64(base + ctr * _GOLDEN)
    return (u >> np.uint64(11)).astype(np.float64) * (2.0 ** -53) + 2.0 ** -54


def normal(seed: int, tag: int, n: int, std: float = 1.0, chunk: int = 1 << 22) -> np.ndarray:
    """n float32 draws from N(0, std^2) (Box-Muller on the stream's uniform pairs)."""
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        u = uniform01(seed, tag, 2 * m, offset=2 * s)
        z = np.sqrt(-2.0 * np.log(u[0::2])) * np.cos(2.0 * math.pi * u[1::2])
        out[s:s + m] = (z * std).astype(np.float32)
    return out


@dataclass(frozen=True)
class Workload:
    """One IHA forward problem: shapes, mask and arithmetic type of X/W/out."""
    name: str
    B: int
    N: int
    H: int
    d: int
    P: int
    mask_mode: int
    window: int
    dtype: str          # "f32" or "bf16" (X, W, out); alpha and R are always fp32
    seed: int

    @property
    def D(self) -> int:
        return self.H * self.d

    @property
    def PN(self) -> int:
        return self.P * self.N

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five problems the method is measured on, named by what they are.
WORKLOADS = {
    "tiny_f32_nomask": Workload("tiny_f32_nomask", B=1, N=64, H=4, d=32, P=2,
                                mask_mode=MASK_NONE, window=0, dtype="f32", seed=0),
    "bf16_causal_n1024": Workload("bf16_causal_n1024", B=2, N=1024, H=16, d=64, P=2,
                                  mask_mode=MASK_CAUSAL, window=0, dtype="bf16", seed=1),
    "bf16_window1024_n4096": Workload("bf16_window1024_n4096", B=4, N=4096, H=16, d=128, P=2,
                                      mask_mode=MASK_WINDOW, window=1024, dtype="bf16", seed=2),
    "bf16_causal_p4_n8192": Workload("bf16_causal_p4_n8192", B=1, N=8192, H=16, d=128, P=4,
                                     mask_mode=MASK_CAUSAL, window=0, dtype="bf16", seed=3),
    "bf16_window4096_n16384": Workload("bf16_window4096_n16384", B=1, N=16384, H=16, d=128, P=2,
                                       mask_mode=MASK_WINDOW, window=4096, dtype="bf16", seed=4),
}
WORKLOAD_ORDER = list(WORKLOADS)


def _cast(a: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(a)
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def make_inputs(w: Workload) -> dict:
    """CPU tensors for workload w. X/W are fp32 or bf16 (per w.dtype); alpha, R fp32."""
    D, Hd, H, P = w.D, w.H * w.d, w.H, w.P
    s = w.seed
    inp = {
        "X": _cast(normal(s, TAGS["X"], w.B * w.N * D).reshape(w.B, w.N, D), w.dtype),
        "W_Q": _cast(normal(s, TAGS["W_Q"], D * Hd, 1.0 / math.sqrt(D)).reshape(D, Hd), w.dtype),
        "W_K": _cast(normal(s, TAGS["W_K"], D * Hd, 1.0 / math.sqrt(D)).reshape(D, Hd), w.dtype),
        "W_V": _cast(normal(s, TAGS["W_V"], D * Hd, 1.0 / math.sqrt(D)).reshape(D, Hd), w.dtype),
    }
    for k in ("alpha_Q", "alpha_K", "alpha_V"):
        inp[k] = torch.from_numpy(normal(s, TAGS[k], H * H * P, 1.0 / math.sqrt(H)).reshape(H, H, P))
    inp["R"] = torch.from_numpy(normal(s, TAGS["R"], H * H * P, 1.0 / math.sqrt(H * P)).reshape(H, H * P))
    return inp


def local_global_schedule(N: int, P_local: int, n_local: int = 4):
    """Per-layer (P, mask_mode, window) of the hybrid local/global schedule of the pages'
    appendix C: n_local sliding-window IHA layers with window N / (2 P^2) tokens, then one
    global layer, taken as one pseudo-head per head (P = 1) over the causal mask -- the
    layer the appendix's FLOP balance counts at plain-attention cost."""
    w = max(1, N // (2 * P_local * P_local))
    return [(P_local, MASK_WINDOW, w)] * n_local + [(1, MASK_CAUSAL, 0)]


def make_stack_inputs(B: int, N: int, H: int, d: int, dtype: str, seed: int, schedule) -> list:
    """CPU inputs of a layer stack: one dict per layer (the make_inputs tensors for that
    layer's P, seeds seed, seed+1, ...) with its P, mask_mode and window; only layer 0's X
    is the stack input."""
    layers = []
    for l, (P, mode, window) in enumerate(schedule):
        w = Workload(f"stack_layer{l}", B=B, N=N, H=H, d=d, P=P, mask_mode=mode, window=window, dtype=dtype,
                     seed=seed + l)
        inp = make_inputs(w)
        inp.update(P=P, mask_mode=mode, window=window, workload=w)
        layers.append(inp)
    return layers


def identity_mixing(H: int, P: int) -> torch.Tensor:
    """alpha[m, h, j] = 1 if m == h else 0, for every j (each pseudo-head copies its own head)."""
    a = torch.zeros(H, H, P, dtype=torch.float32)
    for h in range(H):
        a[h, h, :] = 1.0
    return a


def first_block_contraction(H: int, P: int) -> torch.Tensor:
    """R[h, h*P + 0] = 1, else 0: head h keeps its own first pseudo-block."""
    r = torch.zeros(H, H * P, dtype=torch.float32)
    for h in range(H):
        r[h, h * P] = 1.0
    return r


def as_f64(inp: dict) -> dict:
    """Exact float64 copies (numpy) of the values a device would receive."""
    return {k: v.to(torch.float64).numpy() for k, v in inp.items()}
