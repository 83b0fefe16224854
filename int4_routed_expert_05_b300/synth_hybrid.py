"""Seeded synthetic inputs for the Gated DeltaNet decode step and gated GQA decode attention.

Like :mod:`synth`, this module only draws numbers (SplitMix64 streams, Box-Muller normals, bf16
rounding of the draws); it holds none of the two steps' arithmetic. The CUDA path and the CPU
oracle consume exactly what it returns.

Shapes. The pages fix two sizes of the 80B hybrid stack (alphalab.site, "Swiftlet 實測資料解讀",
section explaining the 80B layer mix): the 36 DeltaNet layers hold a fixed recurrent state of about
72 MiB in all, and the 12 full-attention layers keep K and V in 32-bit floats, at least 48 KiB per
token. Read with the published Qwen3-Next-80B layout, the state is 32 value heads x 128 x 128
fp32 per layer (36 x 2 MiB = 72 MiB) with 16 key heads of 128, and the cache is 2 K/V heads of 256
per layer (12 x 2 x 2 x 256 x 4 B = 48 KiB per token); 16 query heads per attention layer.

Distributions (the pages give none): state ~ N(0, 0.1^2) fp32; q, k, v, z, gate ~ N(0, 1) in
bf16; decay and write-strength inputs a, b ~ N(0, 1) fp32; A_log = ln U(1, 16) and
dt_bias ~ N(0, 0.5^2) per head; norm weight 1 + N(0, 0.1^2); cached K, V ~ N(0, 1) fp32.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .synth import bf16_bits, normal, stream_key, uniform01

# tensor ids of the hybrid steps' streams (disjoint from the MoE layer's)
T_GDN_STATE, T_GDN_Q, T_GDN_K, T_GDN_V, T_GDN_Z, T_GDN_A, T_GDN_B, T_GDN_PARAM = 101, 102, 103, 104, 105, 106, 107, 108
T_GQA_CACHE, T_GQA_Q, T_GQA_K, T_GQA_V, T_GQA_GATE = 111, 112, 113, 114, 115


@dataclass(frozen=True)
class GdnShape:
    n_key_heads: int
    n_value_heads: int
    key_dim: int
    value_dim: int

    def state_floats(self) -> int:
        return self.n_value_heads * self.value_dim * self.key_dim


@dataclass(frozen=True)
class GqaShape:
    n_q_heads: int
    n_kv_heads: int
    head_dim: int


GDN80 = GdnShape(16, 32, 128, 128)
GQA80 = GqaShape(16, 2, 256)
GDN80_LAYERS, GQA80_LAYERS = 36, 12


def _f32(key: int, n: int, sigma: float, mean: float = 0.0) -> np.ndarray:
    return (mean + sigma * normal(key, n)).astype(np.float32)


def gdn_state(sh: GdnShape, seed: int, layer: int, batch: int = 1) -> np.ndarray:
    """[batch, Hv, dv, dk] fp32."""
    n = batch * sh.state_floats()
    return _f32(stream_key(seed, T_GDN_STATE, layer), n, 0.1).reshape(
        batch, sh.n_value_heads, sh.value_dim, sh.key_dim)


def gdn_params(sh: GdnShape, seed: int, layer: int) -> dict:
    """Per-layer learned parameters: A_log, dt_bias [Hv] and norm_w [dv], fp32."""
    key = stream_key(seed, T_GDN_PARAM, layer)
    Hv = sh.n_value_heads
    A = 1.0 + 15.0 * uniform01(stream_key(key, 1), Hv)
    return {"A_log": np.log(A).astype(np.float32),
            "dt_bias": _f32(stream_key(key, 2), Hv, 0.5),
            "norm_w": _f32(stream_key(key, 3), sh.value_dim, 0.1, 1.0)}


def gdn_inputs(sh: GdnShape, seed: int, layer: int, step: int, batch: int = 1) -> dict:
    """One step's inputs: q, k [batch, Hk, dk] and v, z [batch, Hv, dv] as bf16 bit patterns
    (uint16); a, b [batch, Hv] fp32."""
    Hk, Hv, dk, dv = sh.n_key_heads, sh.n_value_heads, sh.key_dim, sh.value_dim

    def bits(tid, *shape):
        n = int(np.prod(shape))
        return bf16_bits(normal(stream_key(seed, tid, layer, step), n)).reshape(shape)

    return {"q": bits(T_GDN_Q, batch, Hk, dk), "k": bits(T_GDN_K, batch, Hk, dk),
            "v": bits(T_GDN_V, batch, Hv, dv), "z": bits(T_GDN_Z, batch, Hv, dv),
            "a": _f32(stream_key(seed, T_GDN_A, layer, step), batch * Hv, 1.0).reshape(batch, Hv),
            "b": _f32(stream_key(seed, T_GDN_B, layer, step), batch * Hv, 1.0).reshape(batch, Hv)}


def gqa_cache(sh: GqaShape, seed: int, layer: int, max_len: int, filled: int, batch: int = 1) -> np.ndarray:
    """[batch, Hkv, max_len, D] fp32: positions below ``filled`` drawn from N(0, 1), the rest 0."""
    c = np.zeros((batch, sh.n_kv_heads, max_len, sh.head_dim), np.float32)
    if filled:
        n = batch * sh.n_kv_heads * filled * sh.head_dim
        c[:, :, :filled, :] = _f32(stream_key(seed, T_GQA_CACHE, layer), n, 1.0).reshape(
            batch, sh.n_kv_heads, filled, sh.head_dim)
    return c


def gqa_inputs(sh: GqaShape, seed: int, layer: int, step: int, batch: int = 1) -> dict:
    """One step's inputs as bf16 bit patterns: q, gate [batch, Hq, D]; k, v [batch, Hkv, D]."""
    Hq, Hkv, D = sh.n_q_heads, sh.n_kv_heads, sh.head_dim

    def bits(tid, *shape):
        n = int(np.prod(shape))
        return bf16_bits(normal(stream_key(seed, tid, layer, step), n)).reshape(shape)

    return {"q": bits(T_GQA_Q, batch, Hq, D), "k": bits(T_GQA_K, batch, Hkv, D),
            "v": bits(T_GQA_V, batch, Hkv, D), "gate": bits(T_GQA_GATE, batch, Hq, D)}
