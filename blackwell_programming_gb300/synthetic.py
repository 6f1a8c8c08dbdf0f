"""Seeded synthetic inputs for the attention forward (host side, numpy).

This module holds no attention arithmetic.  It only turns a seed into bf16
tensors so that the CUDA path and the fp64 oracle are fed byte-identical
inputs.  The recipe is fixed so that any run, on any host, reproduces it:

* SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014; constants as published by Vigna) gives one 64-bit
  word per counter value ``seed + (i+1)*0x9E3779B97F4A7C15``.
* The top 53 bits give a uniform in (0, 1]: ``u = ((z >> 11) + 1) * 2**-53``.
* Box-Muller on consecutive pairs (u[2p], u[2p+1]) gives two N(0,1) samples
  ``r*cos(2*pi*u2)`` and ``r*sin(2*pi*u2)`` with ``r = sqrt(-2 ln u1)``,
  evaluated in fp64 and cast to fp32.
* The fp32 sample is multiplied by a per-tensor factor in fp32 and rounded to
  bf16 with round-to-nearest-even.
* Tensors are drawn from one stream in the order Q, K, V (V is skipped when it
  aliases the first d_v columns of K).

The workloads (shapes, scales, causal flags) are the five attention shapes of
the fused-attention study: a one-tile correctness case, a causal d=64 case with
large logits, a GQA d=128 causal case, a long-context causal case and the
head-dim 576/512 decode case.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK_PAIRS = 1 << 22


def splitmix64(counters: np.ndarray, seed: int) -> np.ndarray:
    """SplitMix64 output for each 0-based counter (uint64 array)."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (counters.astype(np.uint64) + np.uint64(1)) * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform53(counters: np.ndarray, seed: int) -> np.ndarray:
    """Uniform fp64 in (0, 1] from the top 53 bits of SplitMix64."""
    z = splitmix64(counters, seed)
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normals_f32(seed: int, start: int, count: int) -> np.ndarray:
    """Normals number ``start .. start+count-1`` of the stream, as fp32.

    Normal 2p is the cosine branch and 2p+1 the sine branch of pair p, which
    consumes uniforms 2p and 2p+1.
    """
    out = np.empty(count, dtype=np.float32)
    if count == 0:
        return out
    p0 = start // 2
    p1 = (start + count + 1) // 2
    pos = 0
    for c0 in range(p0, p1, _CHUNK_PAIRS):
        c1 = min(p1, c0 + _CHUNK_PAIRS)
        idx = np.arange(2 * c0, 2 * c1, dtype=np.uint64)
        u = uniform53(idx, seed)
        u1 = u[0::2]
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        t = (2.0 * math.pi) * u2
        pair = np.empty(2 * (c1 - c0), dtype=np.float64)
        pair[0::2] = r * np.cos(t)
        pair[1::2] = r * np.sin(t)
        lo = max(start - 2 * c0, 0)
        hi = min(start + count - 2 * c0, pair.size)
        n = hi - lo
        out[pos:pos + n] = pair[lo:hi].astype(np.float32)
        pos += n
    assert pos == count
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round-to-nearest-even) and return the uint16 bits.

    Inputs here are finite; NaN handling is not needed for the generator.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        rounding = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
        r = (b + rounding) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclass(frozen=True)
class Workload:
    """One attention forward problem: sizes, mask, scale and input recipe."""
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nkv: int
    d_qk: int
    d_v: int
    causal: bool
    scale: float
    q_factor: float = 1.0
    kv_factor: float = 1.0
    v_aliases_k: bool = False
    seed: int = 0

    @property
    def flops(self) -> float:
        """Reported FLOPs: 2*B*Hq*Nq*Nkv*(d_qk+d_v), halved when causal.

        Equal to 4*B*Hq*Nq*Nkv*d when d_qk == d_v == d.
        """
        f = 2.0 * self.B * self.Hq * self.Nq * self.Nkv * (self.d_qk + self.d_v)
        return f / 2.0 if self.causal else f

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes that must cross HBM once: Q, K, V (bf16) in, O, LSE (fp32) out."""
        q = self.B * self.Hq * self.Nq * self.d_qk * 2
        k = self.B * self.Hkv * self.Nkv * self.d_qk * 2
        v = 0 if self.v_aliases_k else self.B * self.Hkv * self.Nkv * self.d_v * 2
        o = self.B * self.Hq * self.Nq * self.d_v * 4
        lse = self.B * self.Hq * self.Nq * 4
        return q + k + v + o + lse

    def with_sizes(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    "tile_d64": Workload("tile_d64", 1, 1, 1, 128, 128, 64, 64, False, 1.0 / 8.0),
    "causal_d64_bigq": Workload("causal_d64_bigq", 2, 8, 8, 1024, 1024, 64, 64, True, 1.0 / 8.0, q_factor=8.0),
    "gqa_causal_d128": Workload("gqa_causal_d128", 4, 32, 8, 4096, 4096, 128, 128, True, 1.0 / math.sqrt(128.0)),
    "long_causal_d128": Workload("long_causal_d128", 1, 32, 8, 16384, 16384, 128, 128, True, 1.0 / math.sqrt(128.0),
                                 q_factor=1.0 / math.sqrt(2.0), kv_factor=1.0 / math.sqrt(2.0)),
    "decode_d576": Workload("decode_d576", 64, 128, 1, 1, 8192, 576, 512, False, 1.0 / math.sqrt(192.0),
                            v_aliases_k=True),
    # latent (MLA) prefill: causal, Nq = Nkv, the decode's 576/512 heads with V = K[..., :512]
    "mla_prefill_causal": Workload("mla_prefill_causal", 1, 64, 1, 4096, 4096, 576, 512, True,
                                   1.0 / math.sqrt(192.0), v_aliases_k=True),
}


@dataclass
class Inputs:
    """bf16 bit patterns (uint16) of Q, K, V in [B, H, N, d] row-major order.

    ``v`` is None when V aliases the first d_v columns of K.
    """
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray | None
    wl: Workload = field(repr=False)

    def f64(self):
        """Exact fp64 copies (V materialised from K when aliased)."""
        q = bf16_bits_to_f64(self.q)
        k = bf16_bits_to_f64(self.k)
        v = k[..., : self.wl.d_v].copy() if self.v is None else bf16_bits_to_f64(self.v)
        return q, k, v


def _draw(seed: int, start: int, shape, factor: float) -> np.ndarray:
    n = int(np.prod(shape))
    x = normals_f32(seed, start, n)
    if factor != 1.0:
        x = x * np.float32(factor)
    return f32_to_bf16_bits(x).reshape(shape)


def make_inputs(wl: Workload) -> Inputs:
    """Draw Q, K, V for a workload from its seed, in the fixed order Q, K, V."""
    qs = (wl.B, wl.Hq, wl.Nq, wl.d_qk)
    ks = (wl.B, wl.Hkv, wl.Nkv, wl.d_qk)
    vs = (wl.B, wl.Hkv, wl.Nkv, wl.d_v)
    nq = int(np.prod(qs))
    nk = int(np.prod(ks))
    q = _draw(wl.seed, 0, qs, wl.q_factor)
    k = _draw(wl.seed, nq, ks, wl.kv_factor)
    v = None if wl.v_aliases_k else _draw(wl.seed, nq + nk, vs, wl.kv_factor)
    return Inputs(q, k, v, wl)


@dataclass(frozen=True)
class GemmWorkload:
    """One projection GEMM C [M, N] = A [M, K] B [N, K]^T (bf16 in, bf16 out)."""
    name: str
    M: int
    N: int
    K: int
    seed: int = 0

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        """A and B read once, C (bf16) written once."""
        return 2 * (self.M * self.K + self.N * self.K + self.M * self.N)


GEMM_WORKLOADS = {
    # the QKV projection in front of gqa_causal_d128: 4 x 4096 tokens of a
    # 4096-wide model into 32 query + 8 key + 8 value heads of 128
    "gemm_qkv_proj": GemmWorkload("gemm_qkv_proj", 16384, 6144, 4096),
}


def make_gemm_inputs(gw: GemmWorkload):
    """bf16 bit patterns of A [M, K] and B [N, K] from the workload's seed, A first."""
    a = f32_to_bf16_bits(normals_f32(gw.seed, 0, gw.M * gw.K)).reshape(gw.M, gw.K)
    b = f32_to_bf16_bits(normals_f32(gw.seed, gw.M * gw.K, gw.N * gw.K)).reshape(gw.N, gw.K)
    return a, b


@dataclass(frozen=True)
class LayerWorkload:
    """One attention layer slice Y = Attn(X W_qkv^T) W_o^T over B sequences of N tokens.

    X ~ N(0, 1); both weights ~ N(0, 1) / sqrt(fan-in) (scaled in fp32 before
    the bf16 rounding), so Q, K, V and Y come out with unit variance, as in
    the attention workloads.
    """
    name: str
    B: int
    N: int
    d_model: int
    Hq: int
    Hkv: int
    d: int
    causal: bool
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def n_qkv(self) -> int:
        return (self.Hq + 2 * self.Hkv) * self.d

    @property
    def flops(self) -> float:
        """QKV GEMM + attention (halved when causal, as for the attention lines) + O GEMM."""
        t = self.B * self.N
        att = 4.0 * self.B * self.Hq * self.N * self.N * self.d
        if self.causal:
            att /= 2.0
        return 2.0 * t * self.n_qkv * self.d_model + att + 2.0 * t * self.d_model * self.Hq * self.d

    @property
    def algorithmic_bytes(self) -> int:
        """X, W_qkv, W_o read; QKV and O written and read back once; Y (bf16) written."""
        t = self.B * self.N
        x = t * self.d_model
        w = self.n_qkv * self.d_model + self.d_model * self.Hq * self.d
        qkv = t * self.n_qkv
        o = t * self.Hq * self.d
        return 2 * (x + w + 2 * qkv + 2 * o + t * self.d_model)

    def with_sizes(self, **kw) -> "LayerWorkload":
        d = dict(self.__dict__)
        d.update(kw)
        return LayerWorkload(**d)


LAYER_WORKLOADS = {
    # the layer around gqa_causal_d128: a 4096-wide model, 32 query and 8 KV
    # heads of 128, 4 sequences of 4096 tokens
    "layer_gqa_d128": LayerWorkload("layer_gqa_d128", 4, 4096, 4096, 32, 8, 128, True),
}


def make_layer_inputs(lw: LayerWorkload):
    """bf16 bit patterns of X [B*N, d_model], W_qkv [(Hq+2Hkv)*d, d_model] and
    W_o [d_model, Hq*d], drawn in that order from the workload's seed."""
    t = lw.B * lw.N
    nx = t * lw.d_model
    nw = lw.n_qkv * lw.d_model
    x = _draw(lw.seed, 0, (t, lw.d_model), 1.0)
    w_qkv = _draw(lw.seed, nx, (lw.n_qkv, lw.d_model), 1.0 / math.sqrt(lw.d_model))
    w_o = _draw(lw.seed, nx + nw, (lw.d_model, lw.Hq * lw.d), 1.0 / math.sqrt(lw.Hq * lw.d))
    return x, w_qkv, w_o
