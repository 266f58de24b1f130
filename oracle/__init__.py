"""fp64 CPU oracle for the KDA serving hot path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg may
import this package.  The product path (``hybrid_linear_attention_decode_gb300``) never imports it and
shares no code with it; the only module both sides use is ``kda_inputs`` (seeded random inputs, none
of the method's arithmetic).

The arithmetic lives in ``kda_oracle.c`` (plain fp64 C, token by token).  This module builds it with
gcc, marshals numpy arrays, and states the slot-pool semantics of the three operations:

* decode step / chunked prefill ("A Preview of Production-Scale Kimi K3 Support on vLLM", section
  "KDA prefill and decode"; "vLLM Kimi K3 Support", section "Fused Kernels and Metadata
  Optimization"): the initial state of request n is gathered from pool slot ``src_slot[n]`` (zeros
  when it is -1), the final state is written to ``dst_slot[n]``;
* checkpoints (same pages, "The Hardest Part: Prefix Caching for KDA" and "Agentic Cache Retention
  Policies"): the j-th boundary of sequence n goes to ``ckpt_slots[ckpt_offsets[n] + j]`` unless that
  entry is -1;
* resume ("The Hardest Part: Prefix Caching for KDA", copy-on-write): slot ``dst[n]`` receives a copy
  of slot ``src[n]``;
* multi-token decode ("vLLM Kimi K3 Support", section "Speculative Decoding with DSpark"): L tokens per
  request in order, the state after token j kept in slot ``dst_slots[r*L + j]`` unless it is -1;
* input projections: q, k, v, a, z, b = x W^T split by rows of the packed weight.

Parity unpinned by the pages: they print no worked numeric example; every pin in the test suite comes
from algebra (closed forms, invariants, brute force, exact rational arithmetic).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkda_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into oracle/_build/libkda_oracle.so (OpenMP when the compiler has it)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


class _Cfg(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("W", ctypes.c_int32),
                ("conv_silu", ctypes.c_int32), ("l2_eps", ctypes.c_double), ("rms_eps", ctypes.c_double),
                ("scale", ctypes.c_double)]


def _configure(lib):
    """Declare the C signatures on a loaded oracle library."""
    p = ctypes.c_void_p
    lib.ora_kda_forward.argtypes = [ctypes.POINTER(_Cfg), ctypes.c_int32, p, p] + [p] * 12 + \
        [ctypes.c_int64, p, p, ctypes.c_int32]
    lib.ora_kda_forward.restype = ctypes.c_int
    lib.ora_ckpt_count.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
    lib.ora_ckpt_count.restype = ctypes.c_int64
    lib.ora_num_threads.restype = ctypes.c_int32
    lib.ora_set_threads.argtypes = [ctypes.c_int32]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(build()))
    return _lib


def num_threads() -> int:
    return int(_load().ora_num_threads())


def set_threads(n: int) -> None:
    _load().ora_set_threads(int(n))


@dataclass
class Cfg:
    """Problem shape and the constants the pages leave open (readings recorded with the design)."""
    H: int
    dk: int
    dv: int
    W: int = 4
    conv_silu: bool = True
    l2_eps: float = 1e-6
    rms_eps: float = 1e-6
    scale: float = 1.0

    @property
    def Cc(self) -> int:
        return 2 * self.dk + self.dv

    def _c(self) -> _Cfg:
        return _Cfg(self.H, self.dk, self.dv, self.W, int(bool(self.conv_silu)), self.l2_eps, self.rms_eps,
                    self.scale)


def ckpt_count(start: int, length: int, interval: int) -> int:
    """Boundaries p with p % interval == 0 and start < p <= start + length."""
    return int(_load().ora_ckpt_count(int(start), int(length), int(interval)))


def ckpt_positions(start: int, length: int, interval: int) -> list[int]:
    n = ckpt_count(start, length, interval)
    first = (start // interval + 1) * interval if interval > 0 else 0
    return [first + j * interval for j in range(n)]


def _f64(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def forward(cfg: Cfg, cu_seqlens, start_pos, q, k, v, a, b, z, conv_w, norm_w, S0, conv0,
            interval: int = 0, chunk: int = 0) -> dict:
    """Run the recurrence over a batch of sequences in fp64.

    Shapes: q,k [T,H,dk]; v [T,H,dv]; a [T,H,dk]; b [T,H]; z [T,H,dv] or None; conv_w [H,Cc,W];
    norm_w [dv]; S0 [N,H,dk,dv]; conv0 [N,H,W-1,Cc].  Returns dict with o, y [T,H,dv], S [N,H,dk,dv],
    conv [N,H,W-1,Cc], ckpt_S [n,H,dk,dv], ckpt_conv [n,H,W-1,Cc], ckpt_seq [n], ckpt_pos [n].
    """
    lib = _load()
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    sp = np.ascontiguousarray(start_pos, dtype=np.int64)
    N = len(sp)
    assert len(cu) == N + 1
    T = int(cu[-1])
    H, dk, dv, W = cfg.H, cfg.dk, cfg.dv, cfg.W
    q, k, v, a, b, z = (_f64(x) for x in (q, k, v, a, b, z))
    conv_w, norm_w = _f64(conv_w), _f64(norm_w)
    assert q.shape == (T, H, dk) and k.shape == (T, H, dk) and v.shape == (T, H, dv)
    assert a.shape == (T, H, dk) and b.shape == (T, H) and (z is None or z.shape == (T, H, dv))
    assert conv_w.shape == (H, cfg.Cc, W) and norm_w.shape == (dv,)
    S = np.array(S0, dtype=np.float64, copy=True, order="C").reshape(N, H, dk, dv)
    conv = np.array(conv0, dtype=np.float64, copy=True, order="C").reshape(N, H, W - 1, cfg.Cc)
    o = np.zeros((T, H, dv))
    y = np.zeros((T, H, dv))
    seqs, poss = [], []
    for n in range(N):
        ps = ckpt_positions(int(sp[n]), int(cu[n + 1] - cu[n]), interval) if interval > 0 else []
        seqs += [n] * len(ps)
        poss += ps
    nck = len(poss)
    ck_S = np.zeros((nck, H, dk, dv))
    ck_conv = np.zeros((nck, H, W - 1, cfg.Cc))
    c = cfg._c()
    rc = lib.ora_kda_forward(ctypes.byref(c), N, _ptr(cu), _ptr(sp), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                             _ptr(z), _ptr(conv_w), _ptr(norm_w), _ptr(S), _ptr(conv), _ptr(o), _ptr(y),
                             int(interval), _ptr(ck_S), _ptr(ck_conv), int(chunk))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return dict(o=o, y=y, S=S, conv=conv, ckpt_S=ck_S, ckpt_conv=ck_conv,
                ckpt_seq=np.array(seqs, dtype=np.int64), ckpt_pos=np.array(poss, dtype=np.int64))


def round_to_bf16(x) -> np.ndarray:
    """Value of x stored in a bf16 state pool: fp64 -> fp32 (nearest even) -> bf16 (nearest even)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + ((u >> 16) & 1) + 0x7FFF) >> 16).astype(np.uint32) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64).reshape(np.shape(x))


def _store(x, state_bf16: bool):
    return round_to_bf16(x) if state_bf16 else x


def _gather(pool_S, pool_conv, src):
    """Initial states of the requests: slot src[n], or zeros when src[n] == -1."""
    N = len(src)
    S0 = np.zeros((N,) + pool_S.shape[1:])
    C0 = np.zeros((N,) + pool_conv.shape[1:])
    for n, s in enumerate(src):
        if s >= 0:
            S0[n] = pool_S[s]
            C0[n] = pool_conv[s]
    return S0, C0


def decode_pool(cfg: Cfg, pool_S, pool_conv, src_slot, dst_slot, q, k, v, a, b, z, conv_w, norm_w,
                state_bf16: bool = False) -> dict:
    """One decode token per request on a slot pool.

    pool_S [slots,H,dk,dv] and pool_conv [slots,H,W-1,Cc] are taken as values (any float dtype); returns
    the fp64 pools after the step (only dst slots change), plus o and y [N,H,dv].  With state_bf16 the
    pool stores states in bf16: a written state is rounded to bf16 (nearest even).
    """
    N = len(src_slot)
    S0, C0 = _gather(pool_S, pool_conv, src_slot)
    r = forward(cfg, np.arange(N + 1), np.zeros(N, dtype=np.int64), q, k, v, a, b, z, conv_w, norm_w, S0, C0)
    out_S = np.array(pool_S, dtype=np.float64, copy=True)
    out_C = np.array(pool_conv, dtype=np.float64, copy=True)
    for n, d in enumerate(dst_slot):
        out_S[d] = _store(r["S"][n], state_bf16)
        out_C[d] = r["conv"][n]
    return dict(pool_S=out_S, pool_conv=out_C, o=r["o"], y=r["y"])


def project(x, w, H: int, dk: int, dv: int) -> dict:
    """The input projections of a layer: Y = x W^T in fp64, split by rows of W into q, k, v, a, z [T, H, d]
    and b [T, H] ("A Preview of Production-Scale Kimi K3 Support on vLLM", section "KDA prefill and decode":
    the input projections feeding the recurrence).  x [T, hidden], w [N, hidden], N = H*(3dk + 2dv) + H."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    y = x @ w.T
    T = x.shape[0]
    out, c = {}, 0
    for name, width, d in (("q", H * dk, dk), ("k", H * dk, dk), ("v", H * dv, dv), ("a", H * dk, dk),
                           ("z", H * dv, dv), ("b", H, 1)):
        blk = y[:, c:c + width]
        out[name] = blk.reshape(T, H) if name == "b" else blk.reshape(T, H, d)
        c += width
    assert c == w.shape[0]
    return out


def decode_multi_pool(cfg: Cfg, pool_S, pool_conv, L: int, src_slot, dst_slots, q, k, v, a, b, z, conv_w, norm_w,
                      state_bf16: bool = False) -> dict:
    """L consecutive decode tokens per request with per-position retention (speculative verification).

    Token j of request r is row r*L + j of q..z.  The recurrence runs through the L tokens of each request
    from slot src_slot[r] (zeros when -1); the state and window after token j are written to slot
    dst_slots[r*L + j] unless it is -1 (the rollback reading: every position the caller may resume from is
    kept).  Returns the fp64 pools after the call, o and y [n*L,H,dv], and the per-position states.
    """
    n = len(src_slot)
    dst = np.asarray(dst_slots, dtype=np.int64).reshape(n, L)
    S0, C0 = _gather(pool_S, pool_conv, src_slot)
    r = forward(cfg, np.arange(n + 1) * L, np.zeros(n, dtype=np.int64), q, k, v, a, b, z, conv_w, norm_w, S0, C0,
                interval=1)
    assert len(r["ckpt_pos"]) == n * L  # interval 1: a boundary after every token
    out_S = np.array(pool_S, dtype=np.float64, copy=True)
    out_C = np.array(pool_conv, dtype=np.float64, copy=True)
    for i in range(n * L):
        d = dst[i // L, i % L]
        if d >= 0:
            out_S[d] = _store(r["ckpt_S"][i], state_bf16)
            out_C[d] = r["ckpt_conv"][i]
    return dict(pool_S=out_S, pool_conv=out_C, o=r["o"], y=r["y"], pos_S=r["ckpt_S"], pos_conv=r["ckpt_conv"])


def prefill_pool(cfg: Cfg, pool_S, pool_conv, cu_seqlens, start_pos, src_slot, dst_slot, interval,
                 ckpt_slots, q, k, v, a, b, z, conv_w, norm_w, chunk: int = 0, state_bf16: bool = False) -> dict:
    """Varlen prefill on a slot pool with checkpoint emission.

    ckpt_slots lists one slot (or -1 = skip) per boundary, sequences in order, boundaries ascending.
    Returns the fp64 pools after the call, o/y [T,H,dv], and the oracle's checkpoint list.
    """
    S0, C0 = _gather(pool_S, pool_conv, src_slot)
    r = forward(cfg, cu_seqlens, start_pos, q, k, v, a, b, z, conv_w, norm_w, S0, C0, interval=interval,
                chunk=chunk)
    ckpt_slots = np.asarray(ckpt_slots, dtype=np.int64).reshape(-1)
    assert len(ckpt_slots) == len(r["ckpt_pos"]), "one ckpt slot entry per boundary"
    out_S = np.array(pool_S, dtype=np.float64, copy=True)
    out_C = np.array(pool_conv, dtype=np.float64, copy=True)
    for j, s in enumerate(ckpt_slots):
        if s >= 0:
            out_S[s] = _store(r["ckpt_S"][j], state_bf16)
            out_C[s] = r["ckpt_conv"][j]
    for n, d in enumerate(dst_slot):
        out_S[d] = _store(r["S"][n], state_bf16)
        out_C[d] = r["conv"][n]
    return dict(pool_S=out_S, pool_conv=out_C, o=r["o"], y=r["y"], ckpt_seq=r["ckpt_seq"],
                ckpt_pos=r["ckpt_pos"], ckpt_S=r["ckpt_S"], ckpt_conv=r["ckpt_conv"])


def resume_pool(pool_S, pool_conv, src_slot, dst_slot) -> dict:
    """Copy-on-write: dst[n] receives slot src[n]'s state and window."""
    out_S = np.array(pool_S, copy=True)
    out_C = np.array(pool_conv, copy=True)
    for s, d in zip(src_slot, dst_slot):
        out_S[d] = pool_S[s]
        out_C[d] = pool_conv[s]
    return dict(pool_S=out_S, pool_conv=out_C)
