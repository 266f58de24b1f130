"""Helpers shared by the GPU parity tests: moving bf16 bit patterns between numpy and torch, the
tolerance measures, and seeded pool set-up.  No method arithmetic lives here."""
import numpy as np
import torch

import kda_inputs as ki

Y_TOL = 2e-2   # bf16 outputs: max over (token, head) of max|y - y_ref| / max|y_ref|
S_TOL = 1e-3   # fp32 states: per (sequence, head) ||S - S_ref||_F / ||S_ref||_F


def to_dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_dev_to_f64(t: torch.Tensor) -> np.ndarray:
    return ki.bf16_bits_to_f64(t.detach().view(torch.int16).cpu().numpy().view(np.uint16))


def bf16_dev_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def y_err(y, ref) -> float:
    """max over vectors of max|y - ref| / max|ref| (last axis = the vector)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.abs(y - ref).max(-1)
    den = np.maximum(np.abs(ref).max(-1), 1e-30)
    return float((num / den).max()) if num.size else 0.0


def s_err(S, ref) -> float:
    """max over (.., head) of ||S - ref||_F / ||ref||_F over the last two axes."""
    S = np.asarray(S, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.sqrt(((S - ref) ** 2).sum((-1, -2)))
    den = np.maximum(np.sqrt((ref ** 2).sum((-1, -2))), 1e-30)
    return float((num / den).max()) if num.size else 0.0


def fill_pool(pool, seed: int, unique: int = 256):
    """Fill every (slot, head) unit of a device pool from `unique` host-generated units, unit u
    holding the contents of unit u % unique.  Returns the host copies (S [unique,dk,dv] fp32,
    conv [unique,W-1,Cc] uint16)."""
    ns, H, dk, dv = pool.S.shape
    W = pool.conv.shape[2] + 1
    U = min(unique, ns * H)
    S_h, C_h = ki.pool_tiles(seed, H, dk, dv, W, np.arange(U))
    S_d = torch.from_numpy(S_h).cuda()
    C_d = to_dev_bf16(C_h)
    flatS = pool.S.view(ns * H, dk, dv)
    flatC = pool.conv.view(ns * H, W - 1, 2 * dk + dv)
    for start in range(0, ns * H, U):
        m = min(U, ns * H - start)
        flatS[start:start + m].copy_(S_d[:m])
        flatC[start:start + m].copy_(C_d[:m])
    return S_h, C_h


def pool_unit_host(S_h, C_h, slot: int, H: int):
    """Host contents of slot `slot` (all heads) for a pool filled by fill_pool."""
    U = S_h.shape[0]
    idx = [(slot * H + h) % U for h in range(H)]
    return S_h[idx].astype(np.float64), ki.bf16_bits_to_f64(C_h[idx])
