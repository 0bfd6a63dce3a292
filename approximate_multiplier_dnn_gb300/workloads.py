"""Seeded synthetic inputs for the five layer workloads (numpy, host memory).

This module only draws random numbers; it holds none of the multiplier's
arithmetic.  The tests, the benchmark and the smoke check all take their inputs
from here so that the CUDA path and the CPU oracle see identical operands.

Shapes and distributions stand in for the layer workloads that ApproxTrain
trains on (Sec. VII/VIII: LeNet-300-100-style MLPs, CIFAR-style 3x3 conv,
ResNet 1x1 conv) plus a transformer attention head; no dataset is read.
"""
from __future__ import annotations

import numpy as np

MITCHELL_M = 7


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def uniform(shape, lo, hi, seed) -> np.ndarray:
    return rng(seed).uniform(lo, hi, size=shape).astype(np.float32)


def normal(shape, std, seed) -> np.ndarray:
    return (rng(seed).standard_normal(size=shape) * std).astype(np.float32)


def glorot_uniform(fan_in, fan_out, seed) -> np.ndarray:
    lim = np.sqrt(6.0 / (fan_in + fan_out))
    return uniform((fan_in, fan_out), -lim, lim, seed)


def he_normal(shape, fan_in, seed) -> np.ndarray:
    return normal(shape, np.sqrt(2.0 / fan_in), seed)


# ----------------------------------------------------------------- special values
def special_values_mix(n: int, seed: int) -> tuple[np.ndarray, np.ndarray]:
    """n fp32 pairs ~ U[-1,1] with 1/64 of the entries of each operand replaced
    by each special class: +0, -0, denormals (random fraction), +inf, -inf, NaN,
    and exponent-boundary values (|x| near 2^-126 and near 2^127)."""
    g = rng(seed)
    out = []
    for _ in range(2):
        x = g.uniform(-1.0, 1.0, size=n).astype(np.float32)
        bits = x.view(np.uint32)
        cls = g.integers(0, 64, size=n)
        frac = g.integers(1, 1 << 23, size=n, dtype=np.uint32)
        sign = (g.integers(0, 2, size=n, dtype=np.uint32) << 31).astype(np.uint32)
        big_e = g.integers(200, 255, size=n, dtype=np.uint32)
        small_e = g.integers(1, 40, size=n, dtype=np.uint32)
        bits[cls == 0] = 0x00000000
        bits[cls == 1] = 0x80000000
        m = cls == 2
        bits[m] = sign[m] | frac[m]                       # denormal
        bits[cls == 3] = 0x7F800000
        bits[cls == 4] = 0xFF800000
        m = cls == 5
        bits[m] = 0x7F800000 | frac[m]                    # NaN (varied payload)
        m = cls == 6
        bits[m] = sign[m] | (big_e[m] << 23) | frac[m]    # huge normals
        m = cls == 7
        bits[m] = sign[m] | (small_e[m] << 23) | frac[m]  # tiny normals
        out.append(bits.view(np.float32))
    return out[0], out[1]


# ----------------------------------------------------------------- the five workloads
def gemm_small(seed: int = 0):
    """64x128 by 128x64 GEMM, U[-1,1] (Mitchell M=7)."""
    return {"A": uniform((64, 128), -1, 1, seed), "B": uniform((128, 64), -1, 1, seed + 1)}


def elementwise_pairs(n: int = 1 << 20, seed: int = 0):
    a, b = special_values_mix(n, seed)
    return {"a": a, "b": b}


MLP_DIMS = (784, 1000, 500, 10)
MLP_BATCH = 256


def mlp(batch: int = MLP_BATCH, dims=MLP_DIMS):
    """3-layer MLP operands: X ~ N(0,1), Glorot-uniform W_l (seeds 1..3),
    per-layer output gradients dY_l ~ N(0, 0.01^2) (seed 4+l)."""
    d = {"X": normal((batch, dims[0]), 1.0, 0)}
    for l in range(3):
        d[f"W{l + 1}"] = glorot_uniform(dims[l], dims[l + 1], l + 1)
        d[f"dY{l + 1}"] = normal((batch, dims[l + 1]), 0.01, 4 + l)
    return d


CONV3X3 = dict(N=128, H=32, W=32, C=64, K=64, R=3, S=3, stride=(1, 1), pad=(1, 1), dil=(1, 1))


def conv3x3(N=128, H=32, W=32, C=64, K=64, seed=0):
    """NHWC input ~ N(0,1), RSCK 3x3 filter He-normal, NPQK dY ~ N(0, 0.01^2)."""
    return {"x": normal((N, H, W, C), 1.0, seed),
            "w": he_normal((3, 3, C, K), 9 * C, seed + 1),
            "dy": normal((N, H, W, K), 0.01, seed + 2)}


def square_gemm(n: int = 4096, seed: int = 0):
    return {"A": uniform((n, n), -1, 1, seed), "B": uniform((n, n), -1, 1, seed + 1)}


ATTN = dict(batch=32, heads=16, seq=512, dim=64)


def attention(batch=32, heads=16, seq=512, dim=64, seed=0):
    """Q, K, V ~ N(0,1), shape (batch, heads, seq, dim)."""
    shp = (batch, heads, seq, dim)
    return {"Q": normal(shp, 1.0, seed), "K": normal(shp, 1.0, seed + 1), "V": normal(shp, 1.0, seed + 2)}


CONV1X1 = dict(N=64, H=56, W=56, C=256, K=256, R=1, S=1, stride=(1, 1), pad=(0, 0), dil=(1, 1))


def conv1x1(N=64, H=56, W=56, C=256, K=256, seed=0):
    return {"x": normal((N, H, W, C), 1.0, seed), "w": he_normal((1, 1, C, K), C, seed + 1)}


# MobileNet-style depthwise 3x3 layer (depthwise convolution: ApproxTrain Table I)
DWCONV3X3 = dict(N=64, H=56, W=56, C=128, D=1, R=3, S=3, stride=(1, 1), pad=(1, 1), dil=(1, 1))


def dwconv3x3(N=64, H=56, W=56, C=128, D=1, seed=0):
    """NHWC input ~ N(0,1), 3x3 depthwise filter (R, S, C, D) He-normal over
    its 9 taps, NPQK dY ~ N(0, 0.01^2)."""
    return {"x": normal((N, H, W, C), 1.0, seed),
            "w": he_normal((3, 3, C, D), 9, seed + 1),
            "dy": normal((N, H, W, C * D), 0.01, seed + 2)}


# MobileNet-style strided depthwise layer: 112x112x64 -> 56x56x64
DWCONV3X3_S2 = dict(N=64, H=112, W=112, C=64, D=1, R=3, S=3, stride=(2, 2), pad=(1, 1), dil=(1, 1))


def dwconv3x3_s2(N=64, H=112, W=112, C=64, seed=0):
    """As dwconv3x3 for the stride-2 layer: dY is the 56x56 output's gradient."""
    P = (H + 2 - 3) // 2 + 1
    return {"x": normal((N, H, W, C), 1.0, seed),
            "w": he_normal((3, 3, C, 1), 9, seed + 1),
            "dy": normal((N, P, P, C), 0.01, seed + 2)}


# EfficientNet-style 5x5 depthwise layer: 28x28x240, padding 2
DWCONV5X5 = dict(N=64, H=28, W=28, C=240, D=1, R=5, S=5, stride=(1, 1), pad=(2, 2), dil=(1, 1))


def dwconv5x5(N=64, H=28, W=28, C=240, seed=0):
    """As dwconv3x3 for a 5x5 filter (He-normal over its 25 taps)."""
    return {"x": normal((N, H, W, C), 1.0, seed),
            "w": he_normal((5, 5, C, 1), 25, seed + 1),
            "dy": normal((N, H, W, C), 0.01, seed + 2)}

