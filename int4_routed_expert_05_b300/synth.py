"""Seeded synthetic inputs for the routed-expert MoE FFN.

This module only draws numbers: integer codes, bf16 scale/bias/router bit patterns and
activations. It holds none of the layer's arithmetic (no dequantisation, no GEMV, no routing,
no packing into blobs). The CUDA path (through the tests and the benchmark) and the CPU oracle
both consume exactly what it returns, so the two sides see identical inputs.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014) used as a counter-based generator, value i of a stream being mix(key + (i+1)*gamma);
normals by the Box-Muller transform (Box and Muller, 1958). Stream keys are folded from
(seed, tensor id, layer, expert) so every tensor of every layer is an independent stream.

Value distributions follow the workload descriptions of the benchmark configurations:
int4 codes uniform on 0..15 (int8: 0..255), group 64 along each matrix's input dimension,
scale s ~ U(0.005, 0.02) rounded to bf16 and bias b = -8*s (int8: s ~ U(0.005, 0.02)/16 and
b = -128*s, so dequantised magnitudes match; a test-only switch draws b independently), router rows ~ N(0, 0.02) in bf16, shared-expert
gate vector ~ N(0, 0.02) in bf16, activations ~ N(0, 1) rounded to bf16.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
GAMMA = 0x9E3779B97F4A7C15
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)

# tensor ids that separate the streams of one layer
T_ROUTER, T_SHARED_GATE, T_ACT, T_CODES, T_SCALE, T_PERM, T_SEEDSEARCH, T_BIAS = 1, 2, 3, 4, 5, 6, 7, 8
SHARED_EXPERT = -1  # expert id used for the shared expert's stream


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _MIX1
    z = (z ^ (z >> np.uint64(27))) * _MIX2
    return z ^ (z >> np.uint64(31))


def splitmix64(key: int, n: int, start: int = 0) -> np.ndarray:
    """Values start..start+n-1 of the SplitMix64 sequence whose state starts at ``key``."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(key & 0xFFFFFFFFFFFFFFFF) + i * np.uint64(GAMMA)
        return _mix(z)


def stream_key(*parts: int) -> int:
    """Fold integers into one 64-bit stream key (each step is one SplitMix64 output)."""
    k = 0x243F6A8885A308D3
    for p in parts:
        k = int(splitmix64((k ^ (p & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF, 1)[0])
    return k


def uniform01(key: int, n: int, start: int = 0) -> np.ndarray:
    """Doubles in [0, 1) from the top 53 bits."""
    return (splitmix64(key, n, start) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(key: int, n: int) -> np.ndarray:
    """Standard normals by Box-Muller, one pair of uniforms per value."""
    u = splitmix64(key, 2 * n) >> np.uint64(11)
    u1 = (u[0::2].astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = u[1::2].astype(np.float64) * (2.0 ** -53)          # [0, 1)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def bf16_bits(x) -> np.ndarray:
    """bf16 bit patterns of float32 values, round to nearest even (finite inputs)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_value(bits) -> np.ndarray:
    """float32 values of bf16 bit patterns (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def codes(key: int, n: int, bits: int) -> np.ndarray:
    """n uniform integer codes on 0..2^bits-1 (uint8): 16 (int4) or 8 (int8) codes per draw."""
    per = 64 // bits
    z = splitmix64(key, (n + per - 1) // per)
    sh = np.arange(per, dtype=np.uint64) * np.uint64(bits)
    c = (z[:, None] >> sh[None, :]) & np.uint64((1 << bits) - 1)
    return c.reshape(-1)[:n].astype(np.uint8)


@dataclass(frozen=True)
class Shape:
    """One MoE FFN layer: hidden H, E routed experts, top-k, expert inter I, shared inter Is."""
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    shared_inter: int
    bits: int = 4
    group: int = 64
    renorm: bool = True
    # test-only: draw each bias from its own stream, U(-0.16, 0.04) (int8: / 16), independent of
    # the scale, instead of the centring b = -8 s (int8: -128 s)
    free_bias: bool = False

    def with_bits(self, bits: int) -> "Shape":
        return replace(self, bits=bits)


# hidden 256, 16 experts, top-2, inter 64 (tiny, checkable on the CPU in seconds)
TINY = Shape(256, 16, 2, 64, 64)
# Qwen3-Next-80B-A3B-shaped: hidden 2048, 512 experts, top-10, inter 512, shared 512
S80 = Shape(2048, 512, 10, 512, 512)
# Qwen3.6-35B-A3B-shaped: hidden 2048, 256 experts, top-8, inter 512, shared 512
S35 = Shape(2048, 256, 8, 512, 512)


def expert_tensors(shape: Shape, seed: int, layer: int, expert: int) -> dict:
    """Codes and bf16 scale/bias of one expert (``expert`` = SHARED_EXPERT for the shared one).

    Matrices: gate [I][H], up [I][H], down [H][I] with I = inter (or shared_inter); codes are
    uint8 arrays [out][in]; scale/bias are uint16 bf16 bit arrays [out][in/group].
    """
    H = shape.hidden
    I = shape.shared_inter if expert == SHARED_EXPERT else shape.inter
    g = shape.group
    qmax_mid = 8.0 if shape.bits == 4 else 128.0
    sdiv = 1.0 if shape.bits == 4 else 16.0
    out = {}
    for m, (rows, cols) in enumerate([(I, H), (I, H), (H, I)]):
        name = ("gate", "up", "down")[m]
        kq = stream_key(seed, T_CODES, layer, expert, m)
        out[name + "_q"] = codes(kq, rows * cols, shape.bits).reshape(rows, cols)
        ks = stream_key(seed, T_SCALE, layer, expert, m)
        s = (0.005 + 0.015 * uniform01(ks, rows * (cols // g))) / sdiv
        s_bits = bf16_bits(s.astype(np.float32)).reshape(rows, cols // g)
        if shape.free_bias:
            kb = stream_key(seed, T_BIAS, layer, expert, m)
            b = (-0.16 + 0.2 * uniform01(kb, rows * (cols // g))) / sdiv
            b_bits = bf16_bits(b.astype(np.float32)).reshape(rows, cols // g)
        else:
            b_bits = bf16_bits(-qmax_mid * bf16_value(s_bits))  # exact: power-of-two multiple
        out[name + "_s"] = s_bits
        out[name + "_b"] = b_bits
    return out


def router_bits(shape: Shape, seed: int, layer: int) -> np.ndarray:
    """Router rows Wr [E][H], N(0, 0.02), bf16 bits."""
    n = normal(stream_key(seed, T_ROUTER, layer), shape.n_experts * shape.hidden)
    return bf16_bits((0.02 * n).astype(np.float32)).reshape(shape.n_experts, shape.hidden)


def shared_gate_bits(shape: Shape, seed: int, layer: int) -> np.ndarray:
    """Shared-expert gate vector w_sg [H], N(0, 0.02), bf16 bits."""
    n = normal(stream_key(seed, T_SHARED_GATE, layer), shape.hidden)
    return bf16_bits((0.02 * n).astype(np.float32))


def activation_f32(shape: Shape, seed: int, step: int, n_tokens: int = 1) -> np.ndarray:
    """Activations [T][H], N(0, 1) rounded to bf16, returned as float32 values."""
    n = normal(stream_key(seed, T_ACT, step), n_tokens * shape.hidden)
    return bf16_value(bf16_bits(n.astype(np.float32))).reshape(n_tokens, shape.hidden)


def activation_bits(shape: Shape, seed: int, step: int, n_tokens: int = 1) -> np.ndarray:
    """The same activations as bf16 bit patterns [T][H]."""
    return bf16_bits(activation_f32(shape, seed, step, n_tokens))


def expert_map(shape: Shape, seed: int, layer: int, n_unique: int) -> np.ndarray:
    """Which of ``n_unique`` generated expert tensors sits behind expert e of ``layer``.

    Large stacks (tens of thousands of distinct experts) would take far longer to draw than to
    run, so their experts reuse a set of n_unique drawn tensors under a per-layer permutation.
    Every (layer, expert) still has its own pool slot and its own bytes in device memory.
    With n_unique >= n_experts each layer sees n_experts distinct tensors.
    """
    z = splitmix64(stream_key(seed, T_PERM, layer), max(n_unique, shape.n_experts))
    perm = np.argsort(z, kind="stable")
    return (perm[: shape.n_experts] % n_unique).astype(np.int64)
