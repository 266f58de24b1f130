"""Seeded synthetic inputs for the KDA hot path (shared by the tests, the benchmark and the smoke check).

This module holds random numbers and dtype conversion only -- none of the method's arithmetic -- so
that the CUDA path and the CPU oracle can be fed identical inputs without sharing any code.

Generator (defined here, counter based, so any slice of any tensor can be regenerated on its own):
  * key     = mix(mix(seed + G) ^ (stream * 0xD1B54A32D192ED03))      G = 0x9E3779B97F4A7C15
  * bits_i  = mix(key + (i + 1) * G)                                  (mod 2^64)
    where mix is the splitmix64 finaliser (xor-shift 30, * 0xBF58476D1CE4E5B9, xor-shift 27,
    * 0x94D049BB133111EB, xor-shift 31).
  * element i of a standard-normal tensor uses bits_{2i}, bits_{2i+1}:  u1 = (top 24 bits + 1) / 2^24,
    u2 = top 24 bits / 2^24, x = sqrt(-2 ln u1) cos(2 pi u2) (Box-Muller), computed in fp64, stored fp32.
  * bf16 values are the fp32 values rounded to nearest even.

Workload recipes follow the five KDA configurations (tiny; decode step; chunked prefill; prefix resume;
long context): q, k, v, z, g, b_raw ~ N(0,1); the decay logit a = g + 3 (so alpha = sigmoid(N(3,1)));
conv weights N(0,1)/sqrt(W) in fp32; RMSNorm weight 1 + 0.1 N(0,1) in fp32; pool states N(0, 0.02) fp32.
"""
from __future__ import annotations

import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_S = np.uint64(0xD1B54A32D192ED03)

# stream ids of the tensors
STREAM = dict(q=1, k=2, v=3, g=4, b=5, z=6, conv_w=7, norm_w=8, pool_S=9, pool_conv=10, slots=11, misc=12)


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([seed], dtype=np.uint64) + _G
        k = _mix(s) ^ (np.array([stream], dtype=np.uint64) * _S)
        return _mix(k)[0]


def random_bits(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """uint64 bits_i for i in [offset, offset + n)."""
    idx = np.arange(offset, offset + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(_key(seed, stream) + (idx + np.uint64(1)) * _G)


def normal(seed: int, stream: int, shape, offset: int = 0) -> np.ndarray:
    """Standard normals (fp32) for elements [offset, offset + prod(shape)) of a stream."""
    n = int(np.prod(shape)) if len(np.shape(shape)) else int(shape)
    bits = random_bits(seed, stream, 2 * n, 2 * offset)
    hi = (bits >> np.uint64(40)).astype(np.float64)
    u1 = (hi[0::2] + 1.0) * (1.0 / 16777216.0)
    u2 = hi[1::2] * (1.0 / 16777216.0)
    x = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return x.astype(np.float32).reshape(shape)


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """A seeded permutation of range(n) (stable argsort of random keys)."""
    return np.argsort(random_bits(seed, stream, n), kind="stable").astype(np.int64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even; NaN -> canonical quiet NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    with np.errstate(over="ignore"):
        r = ((u + ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)) >> np.uint32(16)).astype(np.uint16)
    r[np.isnan(x)] = 0x7FC0
    return r


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(h: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(h).astype(np.float64)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Values rounded to bf16, returned as fp32."""
    return bf16_bits_to_f32(f32_to_bf16_bits(x))


def token_inputs(seed: int, T: int, H: int, dk: int, dv: int, with_z: bool = True, offset_tokens: int = 0) -> dict:
    """bf16 bit patterns of one batch of tokens: q,k [T,H,dk], v [T,H,dv], a [T,H,dk], b [T,H], z [T,H,dv].

    offset_tokens selects tokens [offset, offset + T) of the same streams, so a long sequence can be
    produced piecewise with identical values.
    """
    o = offset_tokens
    out = dict(
        q=f32_to_bf16_bits(normal(seed, STREAM["q"], (T, H, dk), o * H * dk)),
        k=f32_to_bf16_bits(normal(seed, STREAM["k"], (T, H, dk), o * H * dk)),
        v=f32_to_bf16_bits(normal(seed, STREAM["v"], (T, H, dv), o * H * dv)),
        a=f32_to_bf16_bits(normal(seed, STREAM["g"], (T, H, dk), o * H * dk) + np.float32(3.0)),
        b=f32_to_bf16_bits(normal(seed, STREAM["b"], (T, H), o * H)),
    )
    out["z"] = f32_to_bf16_bits(normal(seed, STREAM["z"], (T, H, dv), o * H * dv)) if with_z else None
    return out


def projection_inputs(seed: int, T: int, hidden: int, N: int, offset_tokens: int = 0) -> tuple:
    """bf16 bit patterns of hidden states x [T, hidden] ~ N(0, 1) and a packed projection weight W [N, hidden]
    ~ N(0, 1/hidden) (so each projected value is about N(0, 1))."""
    x = f32_to_bf16_bits(normal(seed, STREAM["misc"] + 100, (T, hidden), offset_tokens * hidden))
    w = f32_to_bf16_bits(normal(seed, STREAM["misc"] + 101, (N, hidden)) / np.float32(np.sqrt(hidden)))
    return x, w


def layer_weights(seed: int, H: int, dk: int, dv: int, W: int = 4) -> dict:
    """Per-layer constants: conv weights [H, 2dk+dv, W] and RMSNorm weight [dv], fp32."""
    Cc = 2 * dk + dv
    conv_w = normal(seed, STREAM["conv_w"], (H, Cc, W)) / np.float32(np.sqrt(W))
    norm_w = np.float32(1.0) + np.float32(0.1) * normal(seed, STREAM["norm_w"], (dv,))
    return dict(conv_w=conv_w.astype(np.float32), norm_w=norm_w.astype(np.float32))


def pool_tiles(seed: int, H: int, dk: int, dv: int, W: int, units: np.ndarray, std: float = 0.02) -> tuple:
    """Contents of pool units (unit = slot * H + head): fp32 states [n, dk, dv] and bf16 windows
    [n, W-1, 2dk+dv], each unit drawn from its own counter range."""
    units = np.asarray(units, dtype=np.int64).reshape(-1)
    Cc = 2 * dk + dv
    S = np.stack([normal(seed, STREAM["pool_S"], (dk, dv), int(u) * dk * dv) for u in units]) * np.float32(std)
    C = np.stack([f32_to_bf16_bits(normal(seed, STREAM["pool_conv"], (W - 1, Cc), int(u) * (W - 1) * Cc))
                  for u in units]) if W > 1 else np.zeros((len(units), 0, Cc), dtype=np.uint16)
    return S.astype(np.float32), C


def random_slots(seed: int, num_slots: int, n: int, draw: int = 0) -> np.ndarray:
    """n distinct slots out of num_slots (draw selects an independent draw)."""
    return permutation(seed, STREAM["slots"] + 1000 * draw, num_slots)[:n].astype(np.int32)


def fill_device_pool(pool_S, pool_conv, seed: int, unique: int = 256):
    """Fill a device pool (torch tensors S [slots,H,dk,dv] fp32, conv [slots,H,W-1,Cc] bf16) so that
    (slot, head) unit u holds the contents of generated unit u % unique.  Returns the host copies of
    the unique units (S [U,dk,dv] fp32, conv [U,W-1,Cc] uint16)."""
    import torch
    ns, H, dk, dv = pool_S.shape
    W = pool_conv.shape[2] + 1
    U = min(unique, ns * H)
    S_h, C_h = pool_tiles(seed, H, dk, dv, W, np.arange(U))
    S_d = torch.from_numpy(S_h).to(pool_S.device)
    C_d = torch.from_numpy(C_h.view(np.int16)).to(pool_S.device).view(torch.bfloat16)
    flatS = pool_S.view(ns * H, dk, dv)
    flatC = pool_conv.view(ns * H, W - 1, 2 * dk + dv)
    for start in range(0, ns * H, U):
        m = min(U, ns * H - start)
        flatS[start:start + m].copy_(S_d[:m])
        flatC[start:start + m].copy_(C_d[:m])
    return S_h, C_h


def pool_unit_values(S_h, C_h, slot: int, H: int):
    """Values held by slot `slot` (all heads) of a pool filled by fill_device_pool: S fp64, conv fp64."""
    U = S_h.shape[0]
    idx = [(slot * H + h) % U for h in range(H)]
    return S_h[idx].astype(np.float64), bf16_bits_to_f64(C_h[idx])
