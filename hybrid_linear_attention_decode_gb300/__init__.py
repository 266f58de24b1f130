"""GB300-native (sm_103a) Kimi Delta Attention serving hot path -- Python binding of ``libkda.so``.

Argument marshalling only: every step of the path runs in the CUDA kernels behind the C ABI declared in
``include/kda.h``.  PyTorch provides device memory and streams.  There is no fallback: if the library
is missing the import of an entry point raises.

Entry points (same names as the C ABI): ``kda_project_inputs``, ``kda_decode_step``, ``kda_decode_multi``,
``kda_prefill_chunked``,
``kda_resume_from_slot``, ``kda_prefill_workspace_bytes``, ``kda_checkpoint_count``,
``kda_status_string``; the host prefix index ``kda_prefix_*`` through :class:`PrefixIndex`.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkda.so")
_lib = None

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED_SHAPE, KDA_ERR_WORKSPACE, KDA_ERR_CUDA = 0, 1, 2, 3, 4
KDA_DEV_BAD_SLOT, KDA_DEV_BAD_SEQLENS, KDA_DEV_BAD_CKPT, KDA_DEV_TIMEOUT = 1, 2, 4, 16


class KdaError(RuntimeError):
    def __init__(self, rc: int, what: str, detail: str = ""):
        super().__init__(f"{what}: {kda_status_string(rc)} (status {rc})" + (f": {detail}" if detail else ""))
        self.rc = rc
        self.detail = detail


KDA_STATE_FP32, KDA_STATE_BF16 = 0, 1


class _Pool(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("conv_w", ctypes.c_int32),
                ("state_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32), ("num_slots", ctypes.c_int64),
                ("S", ctypes.c_void_p), ("conv", ctypes.c_void_p)]


class _Params(ctypes.Structure):
    _fields_ = [("conv_weight", ctypes.c_void_p), ("norm_weight", ctypes.c_void_p), ("l2_eps", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("scale", ctypes.c_float), ("conv_silu", ctypes.c_int32)]


class _PrefixPlan(ctypes.Structure):
    _fields_ = [("plan_id", ctypes.c_uint64), ("src_slot", ctypes.c_int32), ("private_slot", ctypes.c_int32),
                ("start_pos", ctypes.c_int64), ("num_ckpts", ctypes.c_int32), ("reserved", ctypes.c_int32)]


KDA_RETAIN_INTERVAL, KDA_RETAIN_SECOND_HIT = 0, 1


def load_library(path: str | None = None):
    """Load libkda.so (built in-tree by ``hybrid_linear_attention_decode_gb300/build.py``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libkda.so not built ({p}); run __graft_entry__.build() first")
    lib = ctypes.CDLL(p)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.kda_decode_step.argtypes = [ctypes.POINTER(_Pool), ctypes.POINTER(_Params), i32] + [vp] * 11
    lib.kda_decode_step.restype = ctypes.c_int
    lib.kda_decode_multi.argtypes = [ctypes.POINTER(_Pool), ctypes.POINTER(_Params), i32, i32] + [vp] * 11
    lib.kda_decode_multi.restype = ctypes.c_int
    lib.kda_project_inputs.argtypes = [i64, i32, i32, i32, i32] + [vp] * 10
    lib.kda_project_inputs.restype = ctypes.c_int
    lib.kda_checkpoint_count.argtypes = [i64, i64, i64]
    lib.kda_checkpoint_count.restype = i64
    lib.kda_prefill_workspace_bytes.argtypes = [ctypes.POINTER(_Pool), i32, i64, i32]
    lib.kda_prefill_workspace_bytes.restype = ctypes.c_size_t
    lib.kda_prefill_chunked.argtypes = [ctypes.POINTER(_Pool), ctypes.POINTER(_Params), i32, i64, vp, vp, vp, vp, i32,
                                        i64, vp, vp] + [vp] * 7 + [vp, ctypes.c_size_t, vp, vp]
    lib.kda_prefill_chunked.restype = ctypes.c_int
    lib.kda_prefill_chunked_noalloc.argtypes = [ctypes.POINTER(_Pool), ctypes.POINTER(_Params), i32, i64, vp, vp, vp,
                                                vp, i32, i64, vp, vp] + [vp] * 7 + [vp, vp]
    lib.kda_prefill_chunked_noalloc.restype = ctypes.c_int
    lib.kda_resume_from_slot.argtypes = [ctypes.POINTER(_Pool), i32, vp, vp, vp, vp]
    lib.kda_resume_from_slot.restype = ctypes.c_int
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_version.restype = ctypes.c_int
    lib.kda_last_error_string.argtypes = []
    lib.kda_last_error_string.restype = ctypes.c_char_p
    lib.kda_check_slots.argtypes = [i64, i32, vp, vp, i32, vp]
    lib.kda_check_slots.restype = ctypes.c_int
    lib.kda_selftest_wait_timeout.argtypes = [i64, vp, vp]
    lib.kda_selftest_wait_timeout.restype = ctypes.c_int
    lib.kda_prefix_index_create.argtypes = [i32, i32, i32, i64]
    lib.kda_prefix_index_create.restype = vp
    lib.kda_prefix_index_destroy.argtypes = [vp]
    lib.kda_prefix_index_destroy.restype = None
    lib.kda_prefix_index_free_slots.argtypes = [vp]
    lib.kda_prefix_index_free_slots.restype = i32
    lib.kda_prefix_plan.argtypes = [vp, vp, i64, ctypes.POINTER(_PrefixPlan), vp, i32]
    lib.kda_prefix_plan.restype = ctypes.c_int
    lib.kda_prefix_commit.argtypes = [vp, ctypes.c_uint64]
    lib.kda_prefix_commit.restype = ctypes.c_int
    lib.kda_prefix_abort.argtypes = [vp, ctypes.c_uint64]
    lib.kda_prefix_abort.restype = ctypes.c_int
    lib.kda_prefix_release_slot.argtypes = [vp, i32]
    lib.kda_prefix_release_slot.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libkda must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


@dataclass
class StatePool:
    """The state-slot pool: S [num_slots, H, dk, dv] fp32 or bf16, conv [num_slots, H, W-1, 2dk+dv] bf16."""
    S: torch.Tensor
    conv: torch.Tensor

    @staticmethod
    def empty(num_slots: int, H: int, dk: int, dv: int, W: int = 4, device="cuda",
              state_dtype=torch.float32) -> "StatePool":
        return StatePool(torch.zeros(num_slots, H, dk, dv, dtype=state_dtype, device=device),
                         torch.zeros(num_slots, H, W - 1, 2 * dk + dv, dtype=torch.bfloat16, device=device))

    @property
    def num_slots(self) -> int:
        return int(self.S.shape[0])

    def c(self) -> _Pool:
        ns, H, dk, dv = self.S.shape
        if self.S.dtype == torch.float32:
            sd = KDA_STATE_FP32
        elif self.S.dtype == torch.bfloat16:
            sd = KDA_STATE_BF16
        else:
            raise TypeError("state pool dtype must be float32 or bfloat16")
        return _Pool(H, dk, dv, self.conv.shape[2] + 1, sd, 0, ns, _ptr(self.S), _ptr(self.conv))


@dataclass
class LayerParams:
    """conv_weight [H, 2dk+dv, W] fp32, norm_weight [dv] fp32 and the layer's constants."""
    conv_weight: torch.Tensor
    norm_weight: torch.Tensor
    l2_eps: float = 1e-6
    rms_eps: float = 1e-6
    scale: float = 1.0
    conv_silu: bool = True

    def c(self) -> _Params:
        return _Params(_ptr(self.conv_weight), _ptr(self.norm_weight), self.l2_eps, self.rms_eps, self.scale,
                       int(bool(self.conv_silu)))


def kda_status_string(rc: int) -> str:
    return load_library().kda_status_string(int(rc)).decode()


def kda_checkpoint_count(start_pos: int, length: int, interval: int) -> int:
    return int(load_library().kda_checkpoint_count(int(start_pos), int(length), int(interval)))


def kda_prefill_workspace_bytes(pool: StatePool, nseq: int, total_tokens: int, chunk: int) -> int:
    pc = pool.c()
    return int(load_library().kda_prefill_workspace_bytes(ctypes.byref(pc), int(nseq), int(total_tokens), int(chunk)))


def kda_last_error_string() -> str:
    return load_library().kda_last_error_string().decode()


def _check(rc: int, what: str, detail: bool = True) -> None:
    if rc != KDA_OK:
        raise KdaError(rc, what, kda_last_error_string() if detail else "")


def _host_i32(x):
    import numpy as np
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32).reshape(-1))


def kda_check_slots(num_slots: int, src_slot, dst_slot, ckpt_slots=None) -> None:
    """Host check of one call's slot-aliasing contract (kda_check_slots in the C ABI); raises KdaError naming
    the first violation.  Arrays may be host or device tensors or sequences (device ones are copied)."""
    s, d, c = _host_i32(src_slot), _host_i32(dst_slot), _host_i32(ckpt_slots)
    if len(s) != len(d):
        raise ValueError("src_slot and dst_slot differ in length")
    vp = ctypes.c_void_p
    rc = load_library().kda_check_slots(int(num_slots), len(s), s.ctypes.data_as(vp), d.ctypes.data_as(vp),
                                        0 if c is None else len(c), None if c is None else c.ctypes.data_as(vp))
    _check(rc, "kda_check_slots")


def kda_selftest_wait_timeout(limit_ns: int, dev_status, stream=None) -> None:
    """Run the bounded-wait check: a wait that never completes gives up after limit_ns and sets
    KDA_DEV_TIMEOUT in dev_status (int32 [1] on the GPU)."""
    _check(load_library().kda_selftest_wait_timeout(int(limit_ns), _ptr(dev_status), _stream(stream)),
           "kda_selftest_wait_timeout")


# KDA_CHECK_SLOTS=1: every call checks its slot arrays on the host first (copies them from the device and
# synchronises; for debugging only).
_DEBUG_SLOTS = os.environ.get("KDA_CHECK_SLOTS", "0") not in ("", "0")


def kda_decode_step(pool: StatePool, params: LayerParams, q, k, v, a, b, z, y, src_slot, dst_slot, dev_status,
                    stream=None) -> None:
    """One fused decode token per request; see include/kda.h.  Tensors: q,k,a [n,H,dk] bf16, v,z,y
    [n,H,dv] bf16, b [n,H] bf16, src_slot/dst_slot [n] int32, dev_status [1] int32 (all on the GPU)."""
    n = int(src_slot.shape[0])
    if _DEBUG_SLOTS:
        kda_check_slots(pool.num_slots, src_slot, dst_slot)
    pc, pp = pool.c(), params.c()
    rc = load_library().kda_decode_step(ctypes.byref(pc), ctypes.byref(pp), n, _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                                        _ptr(b), _ptr(z), _ptr(y), _ptr(src_slot), _ptr(dst_slot),
                                        _ptr(dev_status), _stream(stream))
    _check(rc, "kda_decode_step")


def projection_width(H: int, dk: int, dv: int) -> int:
    """Rows of the packed projection weight: q, k, v, a, z and b."""
    return H * (3 * dk + 2 * dv) + H


def kda_project_inputs(x, w, H: int, dk: int, dv: int, q, k, v, a, b, z, dev_status, stream=None) -> None:
    """The six input projections in one GEMM (see include/kda.h): x [T, hidden] bf16, w [N, hidden] bf16 with
    the rows of q, k, v, a, z, b; outputs q, k, a [T, H, dk], v, z [T, H, dv], b [T, H] bf16 (z may be None)."""
    T, hidden = int(x.shape[0]), int(x.shape[1])
    rc = load_library().kda_project_inputs(T, hidden, int(H), int(dk), int(dv), _ptr(x), _ptr(w), _ptr(q), _ptr(k),
                                           _ptr(v), _ptr(a), _ptr(b), _ptr(z), _ptr(dev_status), _stream(stream))
    _check(rc, "kda_project_inputs")


DECODE_MULTI_MAX_L = 8  # KDA_DECODE_MULTI_MAX_L in kda.h


def kda_decode_multi(pool: StatePool, params: LayerParams, L: int, q, k, v, a, b, z, y, src_slot, dst_slots,
                     dev_status, stream=None) -> None:
    """L consecutive decode tokens per request with per-position state retention (speculative verification);
    see include/kda.h.  q,k,a [n*L,H,dk], v,z,y [n*L,H,dv], b [n*L,H] bf16 (row r*L+j = token j of request r);
    src_slot [n] int32; dst_slots [n*L] int32 (-1 = position not kept)."""
    n = int(src_slot.shape[0])
    if _DEBUG_SLOTS:
        kept = _host_i32(dst_slots)
        kda_check_slots(pool.num_slots, [], [], kept)
        src_h = _host_i32(src_slot)
        for r, s_ in enumerate(src_h):
            others = set(kept[:r * L].tolist()) | set(kept[(r + 1) * L:].tolist())
            if s_ >= 0 and int(s_) in others:
                raise KdaError(KDA_ERR_INVALID_ARG, "kda_decode_multi",
                               f"src_slot[{r}] = {s_} is kept by another request")
    pc, pp = pool.c(), params.c()
    rc = load_library().kda_decode_multi(ctypes.byref(pc), ctypes.byref(pp), n, int(L), _ptr(q), _ptr(k), _ptr(v),
                                         _ptr(a), _ptr(b), _ptr(z), _ptr(y), _ptr(src_slot), _ptr(dst_slots),
                                         _ptr(dev_status), _stream(stream))
    _check(rc, "kda_decode_multi")


def kda_prefill_chunked(pool: StatePool, params: LayerParams, cu_seqlens, start_pos, src_slot, dst_slot, chunk: int,
                        ckpt_interval: int, ckpt_offsets, ckpt_slots, q, k, v, a, b, z, y, workspace, dev_status,
                        stream=None) -> None:
    """Chunked prefill with checkpoint emission; see include/kda.h.  cu_seqlens/ckpt_offsets int32
    [nseq+1], start_pos int64 [nseq], slots int32, workspace a uint8 tensor of
    kda_prefill_workspace_bytes() bytes."""
    nseq = int(start_pos.shape[0])
    T = int(q.shape[0]) if q is not None else 0
    if _DEBUG_SLOTS:
        kda_check_slots(pool.num_slots, src_slot, dst_slot, ckpt_slots if ckpt_interval > 0 else None)
    pc, pp = pool.c(), params.c()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load_library().kda_prefill_chunked(
        ctypes.byref(pc), ctypes.byref(pp), nseq, T, _ptr(cu_seqlens), _ptr(start_pos), _ptr(src_slot),
        _ptr(dst_slot), int(chunk), int(ckpt_interval), _ptr(ckpt_offsets), _ptr(ckpt_slots), _ptr(q), _ptr(k),
        _ptr(v), _ptr(a), _ptr(b), _ptr(z), _ptr(y), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(rc, "kda_prefill_chunked")


# Size of the fixed scratch behind kda_prefill_chunked_noalloc (KDA_NOALLOC_SCRATCH_BYTES in kda.h).
NOALLOC_SCRATCH_BYTES = 64 << 20


def kda_prefill_chunked_noalloc(pool: StatePool, params: LayerParams, cu_seqlens, start_pos, src_slot, dst_slot,
                                chunk: int, ckpt_interval: int, ckpt_offsets, ckpt_slots, q, k, v, a, b, z, y,
                                dev_status, stream=None) -> None:
    """kda_prefill_chunked for callers that cannot allocate device memory: the workspace is the library's
    fixed scratch (NOALLOC_SCRATCH_BYTES per GPU).  Calls that overlap on the GPU race on that scratch;
    the first call on a device (nseq = 0 does only that set-up) should come at start-up, before any stream
    capture.  See include/kda.h."""
    nseq = int(start_pos.shape[0])
    T = int(q.shape[0]) if q is not None else 0
    if _DEBUG_SLOTS and nseq > 0:
        kda_check_slots(pool.num_slots, src_slot, dst_slot, ckpt_slots if ckpt_interval > 0 else None)
    pc, pp = pool.c(), params.c()
    rc = load_library().kda_prefill_chunked_noalloc(
        ctypes.byref(pc), ctypes.byref(pp), nseq, T, _ptr(cu_seqlens), _ptr(start_pos), _ptr(src_slot),
        _ptr(dst_slot), int(chunk), int(ckpt_interval), _ptr(ckpt_offsets), _ptr(ckpt_slots), _ptr(q), _ptr(k),
        _ptr(v), _ptr(a), _ptr(b), _ptr(z), _ptr(y), _ptr(dev_status), _stream(stream))
    _check(rc, "kda_prefill_chunked_noalloc")


def kda_resume_from_slot(pool: StatePool, src_slot, dst_slot, dev_status, stream=None) -> None:
    """Copy-on-write: slot dst_slot[i] receives a bit-exact copy of slot src_slot[i] (int32 [n])."""
    if _DEBUG_SLOTS:
        kda_check_slots(pool.num_slots, src_slot, dst_slot)
    pc = pool.c()
    rc = load_library().kda_resume_from_slot(ctypes.byref(pc), int(src_slot.shape[0]), _ptr(src_slot),
                                             _ptr(dst_slot), _ptr(dev_status), _stream(stream))
    _check(rc, "kda_resume_from_slot")


@dataclass
class PrefixPlan:
    """What one prompt needs: resume from ``src_slot`` (or start fresh when it is -1) into ``private_slot``,
    prefill tokens [start_pos, len) with checkpoint interval = the match unit and the ``ckpt_slots`` table
    (one entry per match-unit boundary in (start_pos, len]: a pool slot, or -1 to skip)."""
    plan_id: int
    src_slot: int
    private_slot: int
    start_pos: int
    ckpt_slots: list


class PrefixIndex:
    """Host prefix index over a state pool (``kda_prefix_index_*`` in the C ABI): chained match-unit hashes
    to checkpoint slots, copy-on-write private slots, LRU eviction, interval or second-hit retention."""

    def __init__(self, num_slots: int, match_unit: int = 128, policy: int = KDA_RETAIN_INTERVAL,
                 interval: int = 0):
        self._lib = load_library()
        self._h = self._lib.kda_prefix_index_create(int(num_slots), int(match_unit), int(policy), int(interval))
        if not self._h:
            raise KdaError(KDA_ERR_INVALID_ARG, "kda_prefix_index_create")
        self.match_unit = int(match_unit)

    def close(self) -> None:
        if self._h:
            self._lib.kda_prefix_index_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def free_slots(self) -> int:
        return int(self._lib.kda_prefix_index_free_slots(self._h))

    def plan(self, tokens) -> PrefixPlan:
        import numpy as np
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        cap = max(1, len(t) // self.match_unit)
        ck = np.empty(cap, dtype=np.int32)
        out = _PrefixPlan()
        rc = self._lib.kda_prefix_plan(self._h, t.ctypes.data_as(ctypes.c_void_p), len(t), ctypes.byref(out),
                                       ck.ctypes.data_as(ctypes.c_void_p), cap)
        _check(rc, "kda_prefix_plan", detail=False)
        return PrefixPlan(int(out.plan_id), int(out.src_slot), int(out.private_slot), int(out.start_pos),
                          [int(x) for x in ck[:out.num_ckpts]])

    def commit(self, plan: PrefixPlan) -> None:
        _check(self._lib.kda_prefix_commit(self._h, plan.plan_id), "kda_prefix_commit", detail=False)

    def abort(self, plan: PrefixPlan) -> None:
        _check(self._lib.kda_prefix_abort(self._h, plan.plan_id), "kda_prefix_abort", detail=False)

    def release_slot(self, slot: int) -> None:
        _check(self._lib.kda_prefix_release_slot(self._h, int(slot)), "kda_prefix_release_slot", detail=False)
