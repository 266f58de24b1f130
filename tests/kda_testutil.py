"""Helpers shared by the GPU parity tests: moving bf16 bit patterns between numpy and torch, the
tolerance measures, and seeded pool set-up.  No method arithmetic lives here."""
import numpy as np
import torch

import kda_inputs as ki

Y_TOL = 2e-2   # bf16 outputs: max over (token, head) of max|y - y_ref| / max|y_ref|
S_TOL = 1e-3   # fp32 states: per (sequence, head) ||S - S_ref||_F / ||S_ref||_F
# bf16 state pools: a stored state is the bf16 rounding (nearest even, relative error <= 2^-9 per element) of
# a value computed to S_TOL, so against the unrounded reference the bar is S_TOL + 2^-9
S_TOL_BF16 = S_TOL + 2.0 ** -9


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
    return ki.fill_device_pool(pool.S, pool.conv, seed, unique)


def pool_unit_host(S_h, C_h, slot: int, H: int):
    return ki.pool_unit_values(S_h, C_h, slot, H)
