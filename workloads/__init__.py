"""Seeded synthetic workloads for the MoE route / dispatch / combine path.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark. It draws random numbers and shapes them into inputs; it holds none of
the method's arithmetic (no top-k, no softmax, no quantisation, no combine).
Rounding a normal sample to bf16 is done by PyTorch's CPU cast, so this module
carries no codec of its own either.

Generator: SplitMix64 over a 64-bit counter (Steele, Lea & Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014), two draws per sample,
Box-Muller transform in float64. Every array is a pure function of
(seed, stream, index), so a sub-range can be regenerated without the rest.

Workloads (shapes of the models the pages name; no weights or datasets):

  tiny          T=64,   H=256,  E=8,   k=2, R=2, C=64,   bf16
  v2lite        T=256,  H=2048, E=64,  k=6, R=4, C=256,  bf16   (DeepSeek-V2-Lite decode)
  mixtral_skew  T=4096, H=4096, E=8,   k=2, R=8, C=4096, bf16   (Mixtral prefill,
                logits + b_e, b_e = 1.5*ln(1/(e+1)), Zipf-like hot experts)
  dsv3_fp8      T=1024, H=7168, E=256, k=8, R=8, C=128,  fp8 e4m3 block-128
                (DeepSeek-V3 decode; 8 virtual DP source ranks x 128 tokens)
  dbo           T=8192, H=7168, E=256, k=8, R=8, C=1024, bf16, two micro-batches
                of 4096 tokens (Dual Batch Overlap prefill)

x ~ bf16(float32(N(0,1))), logits ~ float32(N(0,1)) (+ float32(b_e), added in
float32), expert scale s_e = 1 + e/E evaluated in float32.

Expert weights of the grouped GEMM (random; the pages ship none) are drawn as
storage directly, not quantised from real values: e4m3 codes with a uniform
sign and a magnitude code uniform in 0x30..0x77 (|w| in [0.5, 240]), and one
fp32 scale per 128 x 128 block, 2^-8 * (1 + u) with u uniform in [0, 1).
make_weights draws them with SplitMix64 (small cases, checked by the oracle);
make_weights_device draws the same distribution with PyTorch's seeded device
generator (full-size runs, where a host draw of gigabytes would take minutes).
bf16 weights (for bf16 rows): bf16(float32(N(0,1) * 2^-5)), host (make_weights_bf16)
or device (make_weights_bf16_device, PyTorch's generator).
"""
from __future__ import annotations

from dataclasses import dataclass, replace
import math

import numpy as np

MASK64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB

STREAM_X = 1
STREAM_LOGITS = 2
STREAM_W = 3
STREAM_W_SCALE = 4
STREAM_W_BF16 = 5
W_MAG_LO, W_MAG_N = 0x30, 72          # magnitude codes 0x30..0x77

DTYPE_BF16 = 0
DTYPE_FP8_E4M3_B128 = 1


@dataclass(frozen=True)
class Workload:
    name: str
    T: int          # tokens
    H: int          # hidden size (elements per token row)
    E: int          # routed experts
    k: int          # experts per token
    R: int          # virtual expert-parallel ranks
    C: int          # capacity: rows reserved per expert
    dtype: int = DTYPE_BF16
    bias: str = "none"             # "none" | "zipf15": b_e = 1.5*ln(1/(e+1))
    src_ranks: int = 1             # virtual DP source ranks (token t comes from rank t // (T // src_ranks))
    micro_batches: int = 1         # 2 for the dual-batch-overlap workload
    seed: int = 1000

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", T=64, H=256, E=8, k=2, R=2, C=64, seed=1000),
    "v2lite": Workload("v2lite", T=256, H=2048, E=64, k=6, R=4, C=256, seed=1001),
    "mixtral_skew": Workload("mixtral_skew", T=4096, H=4096, E=8, k=2, R=8, C=4096,
                             bias="zipf15", seed=1002),
    "dsv3_fp8": Workload("dsv3_fp8", T=1024, H=7168, E=256, k=8, R=8, C=128,
                         dtype=DTYPE_FP8_E4M3_B128, src_ranks=8, seed=1003),
    "dbo": Workload("dbo", T=8192, H=7168, E=256, k=8, R=8, C=1024,
                    micro_batches=2, seed=1004),
}


def _stream_key(seed: int, stream: int) -> int:
    """A 64-bit key per (seed, stream): one SplitMix64 step of seed*2^16 + stream."""
    return int(splitmix64((seed * 65536 + stream) & MASK64, 0, 1)[0])


def splitmix64(key: int, start: int, n: int) -> np.ndarray:
    """Outputs start..start+n-1 of the SplitMix64 sequence seeded with `key`."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    z = np.uint64(key & MASK64) + i * np.uint64(_GOLDEN)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_MIX1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_MIX2)
    return z ^ (z >> np.uint64(31))


def normals(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    """float64 N(0,1) samples start..start+n-1 of (seed, stream)."""
    key = _stream_key(seed, stream)
    z = splitmix64(key, 2 * start, 2 * n)
    a = z[0::2] >> np.uint64(11)
    b = z[1::2] >> np.uint64(11)
    u1 = (a.astype(np.float64) + 1.0) * (2.0 ** -53)      # (0, 1]
    u2 = b.astype(np.float64) * (2.0 ** -53)              # [0, 1)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def _to_bf16_bits(f32: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def make_x(w: Workload, t0: int = 0, nt: int | None = None, chunk: int = 1 << 22) -> np.ndarray:
    """Token rows x[t0:t0+nt] as bf16 bit patterns, shape [nt, H], dtype uint16."""
    nt = w.T - t0 if nt is None else nt
    out = np.empty(nt * w.H, dtype=np.uint16)
    base = t0 * w.H
    for s in range(0, nt * w.H, chunk):
        n = min(chunk, nt * w.H - s)
        out[s:s + n] = _to_bf16_bits(normals(w.seed, STREAM_X, base + s, n).astype(np.float32))
    return out.reshape(nt, w.H)


def expert_bias(w: Workload) -> np.ndarray:
    """Per-expert float32 logit bias b_e (zeros unless the workload is skewed)."""
    if w.bias == "none":
        return np.zeros(w.E, dtype=np.float32)
    if w.bias == "zipf15":
        return np.array([1.5 * math.log(1.0 / (e + 1)) for e in range(w.E)], dtype=np.float64).astype(np.float32)
    raise ValueError(w.bias)


def make_logits(w: Workload, t0: int = 0, nt: int | None = None) -> np.ndarray:
    """Router logits[t0:t0+nt], float32 [nt, E]: float32(N(0,1)) + float32(b_e)."""
    nt = w.T - t0 if nt is None else nt
    z = normals(w.seed, STREAM_LOGITS, t0 * w.E, nt * w.E).astype(np.float32).reshape(nt, w.E)
    b = expert_bias(w)
    if w.bias != "none":
        z = (z + b[None, :]).astype(np.float32)
    return np.ascontiguousarray(z)


def expert_scale(w: Workload) -> np.ndarray:
    """Synthetic expert scale s_e = 1 + e/E, evaluated in float32."""
    e = np.arange(w.E, dtype=np.float32)
    return (np.float32(1.0) + e / np.float32(w.E)).astype(np.float32)


def make_inputs(w: Workload) -> dict:
    """All host inputs of one workload: x (uint16 bf16 bits), logits, s."""
    return {"x": make_x(w), "logits": make_logits(w), "s": expert_scale(w)}



def make_weights(w: Workload, e0: int = 0, ne: int | None = None, N: int | None = None):
    """Experts e0..e0+ne-1 of the grouped GEMM's weights: e4m3 codes
    w_q[ne][N][H] (uint8) and fp32 block scales w_scale[ne][N/128][H/128].
    N defaults to H (an H -> H map per expert)."""
    ne = w.E - e0 if ne is None else ne
    N = w.H if N is None else N
    per = N * w.H
    z = splitmix64(_stream_key(w.seed, STREAM_W), e0 * per, ne * per)
    r = (z >> np.uint64(32)) % np.uint64(2 * W_MAG_N)
    mag = (r % np.uint64(W_MAG_N)).astype(np.uint8) + np.uint8(W_MAG_LO)
    sign = (r // np.uint64(W_MAG_N)).astype(np.uint8) << np.uint8(7)
    w_q = (mag | sign).reshape(ne, N, w.H)
    nbs = (N // 128) * (w.H // 128)
    u = (splitmix64(_stream_key(w.seed, STREAM_W_SCALE), e0 * nbs, ne * nbs) >> np.uint64(11)).astype(np.float64)
    w_scale = ((1.0 + u * 2.0 ** -53) * 2.0 ** -8).astype(np.float32).reshape(ne, N // 128, w.H // 128)
    return w_q, w_scale


def make_weights_device(w: Workload, device, N: int | None = None):
    """All experts' weights drawn on `device` by PyTorch's seeded generator,
    same distribution as make_weights (not the same values)."""
    import torch
    N = w.H if N is None else N
    g = torch.Generator(device=device)
    g.manual_seed(w.seed * 65536 + STREAM_W)
    w_q = torch.empty((w.E, N, w.H), dtype=torch.uint8, device=device)
    for e in range(w.E):
        r = torch.randint(0, 2 * W_MAG_N, (N, w.H), generator=g, device=device, dtype=torch.int16)
        w_q[e] = ((r % W_MAG_N + W_MAG_LO) | ((r // W_MAG_N) << 7)).to(torch.uint8)
    u = torch.rand((w.E, N // 128, w.H // 128), generator=g, device=device, dtype=torch.float64)
    w_scale = ((1.0 + u) * 2.0 ** -8).to(torch.float32)
    return w_q, w_scale


def make_weights_bf16(w: Workload, e0: int = 0, ne: int | None = None, N: int | None = None) -> np.ndarray:
    """bf16 weights of the grouped GEMM for bf16 rows, experts e0..e0+ne-1:
    w[ne][N][H] bit patterns of bf16(float32(N(0,1) * 2^-5))."""
    ne = w.E - e0 if ne is None else ne
    N = w.H if N is None else N
    per = N * w.H
    v = (normals(w.seed, STREAM_W_BF16, e0 * per, ne * per) * 2.0 ** -5).astype(np.float32)
    return _to_bf16_bits(v).reshape(ne, N, w.H)


def make_weights_bf16_device(w: Workload, device, N: int | None = None):
    """All experts' bf16 weights drawn on `device` by PyTorch's seeded generator
    (same distribution as make_weights_bf16, not the same values), as int16 bits."""
    import torch
    N = w.H if N is None else N
    g = torch.Generator(device=device)
    g.manual_seed(w.seed * 65536 + STREAM_W_BF16)
    out = torch.empty((w.E, N, w.H), dtype=torch.int16, device=device)
    for e in range(w.E):
        out[e] = (torch.randn((N, w.H), generator=g, device=device, dtype=torch.float32) * 2.0 ** -5).to(
            torch.bfloat16).view(torch.int16)
    return out
