"""4-bit group-quantised (Q4) KV blocks.

Source: Q4 edge paper summary §2.1 — per-agent KV split into fixed 256-token
blocks stored 4-bit quantised, about 72 % smaller than FP16 (ratio 0.281);
§2.2 — attention runs on the Q4 tensors directly, without a dequantise-to-FP16
pass.  The ratio 0.281 = (4 + 2*16/64)/16 fixes group 64 with an fp16 scale
and an fp16 bias per group.

Reading of the format (the pages give none beyond the ratio): affine
quantisation per 64-element group along head_dim, per (token, KV head, K|V):
scale = fp16((max - min) / 15), bias = fp16(min), computed in float32;
code = clamp(round_half_even((x - bias) / scale), 0, 15) in float32 with
scale and bias taken as their fp16 values; scale 0 gives code 0.  Element 2i
sits in the low nibble of byte i.  Dequantisation x_hat = scale * c + bias is
exact in fp64.

Layouts: codes [blocks][Hkv][B][d/2] uint8; scale/bias [blocks][Hkv][B][d/64][2]
fp16 (index 0 = scale, 1 = bias).
"""
from __future__ import annotations

import numpy as np

GROUP = 64


def quantize(x: np.ndarray):
    """x [..., d] float32 (d a multiple of 64) -> (codes uint8 [..., d/2],
    sb float16 [..., d/64, 2])."""
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    g = x.reshape(x.shape[:-1] + (d // GROUP, GROUP))
    mn = g.min(axis=-1)
    mx = g.max(axis=-1)
    scale16 = ((mx - mn) / np.float32(15.0)).astype(np.float32).astype(np.float16)
    bias16 = mn.astype(np.float16)
    s32 = scale16.astype(np.float32)[..., None]
    b32 = bias16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint((g - b32) / s32).astype(np.float32)
    q = np.where(s32 == 0, np.float32(0), q)
    q = np.clip(q, 0, 15).astype(np.uint8).reshape(x.shape)
    codes = (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)
    sb = np.stack([scale16, bias16], axis=-1)
    return codes, sb


def unpack(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    out = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = c & 0x0F
    out[..., 1::2] = c >> 4
    return out


def dequantize(codes: np.ndarray, sb: np.ndarray) -> np.ndarray:
    """fp64 values s*c + b, [..., d]."""
    c = unpack(codes).astype(np.float64)
    d = c.shape[-1]
    g = c.reshape(c.shape[:-1] + (d // GROUP, GROUP))
    s = np.asarray(sb[..., 0], dtype=np.float64)[..., None]
    b = np.asarray(sb[..., 1], dtype=np.float64)[..., None]
    return (g * s + b).reshape(c.shape)
