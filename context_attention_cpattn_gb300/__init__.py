"""cpattn - packed variable-length context-parallel attention on one GB300.

Thin Python binding of ``libcpattn.so`` (C ABI in ``include/cpattn.h``).  The
functions keep the C names and only marshal arguments: torch tensors are
passed as device pointers and the current CUDA stream as the stream handle.
Every step of the computation runs in the library's CUDA kernels; there is no
Python or CPU fallback, and a missing library raises ``ImportError``.
"""

from __future__ import annotations

import ctypes
import math
import os
import re
from typing import Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# CPATTN_LIB loads another prebuilt copy of the library instead of the in-tree
# one (build() always writes the in-tree library).
LIB_PATH = os.environ.get("CPATTN_LIB") or os.path.join(_PKG, "lib", "libcpattn.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "cpattn.h")

OK, INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA_ERROR, DEVICE_FAULT = range(6)
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE", 4: "CUDA_ERROR", 5: "DEVICE_FAULT"}
MODES = {"zigzag": 0, "grid2d": 1, "contiguous": 2, "ulysses2d": 3, "paired": 4}
DTYPE_FP32, DTYPE_BF16 = 0, 1
MASK_SKIP, MASK_FULL, MASK_DIAG, MASK_KV_HEAD, MASK_Q_TAIL = range(5)


class CpattnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class _Grid(ctypes.Structure):
    _fields_ = [("frames", ctypes.c_int32), ("height", ctypes.c_int32), ("width", ctypes.c_int32)]


class _PlanInfo(ctypes.Structure):
    _fields_ = [("total_tokens", ctypes.c_int64), ("n_chunks", ctypes.c_int64), ("max_rank_tokens", ctypes.c_int64),
                ("n_seqs", ctypes.c_int32), ("cp_size", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("split_h", ctypes.c_int32), ("split_w", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class _DcpConfig(ctypes.Structure):
    _fields_ = [("max_cp", ctypes.c_int32), ("reserved", ctypes.c_int32), ("cap_tokens", ctypes.c_int64),
                ("attn_coef", ctypes.c_int64), ("lin_coef", ctypes.c_int64)]


_lib = None
_P, _I32, _I64, _SZ, _F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float

_SIGNATURES = {
    "cpattn_plan": [_P, _I32, _I32, _I32, _P, _P],
    "cpattn_plan_2d": [_P, _I32, _I32, _I32, _P],
    "cpattn_plan_paired": [_P, _I32, _I32, _I32, _P],
    "cpattn_plan_allowed_pairs": [_P, _I32, _P],
    "cpattn_plan_destroy": [_P],
    "cpattn_plan_get_a2a_map": [_P, _P, _I64],
    "cpattn_plan_get_worklist": [_P, _I32, _I32, _I32, _I32, _I32, _P, _I64, _P, _I64, _P, _P],
    "cpattn_plan_get_info": [_P, _P],
    "cpattn_plan_get_chunk_offsets": [_P, _P, _I64],
    "cpattn_plan_get_chunk_ranks": [_P, _P, _I64],
    "cpattn_plan_get_rank_offsets": [_P, _P, _I64],
    "cpattn_plan_get_local_cu_seqlens": [_P, _I32, _P, _I64],
    "cpattn_plan_get_index_map": [_P, _P, _I64],
    "cpattn_plan_get_ring_schedule": [_P, _I32, _P, _P, _I64],
    "cpattn_workspace_size": [_P, _I32, _I32, _I32, _I32, _I32, _P],
    "cpattn_fwd": [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _F32, _I32, _P, _P, _P, _SZ, _P],
    "cpattn_fwd_static": [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _F32, _I32, _P, _P, _P],
    "cpattn_block_fwd": [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _F32, _I32, _I32, _I32, _P, _P, _P, _SZ, _P],
    "cpattn_bwd_workspace_size": [_P, _I32, _I32, _I32, _I32, _I32, _P],
    "cpattn_bwd": [_P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _F32, _I32, _P, _P, _P, _P, _SZ, _P],
    "cpattn_block_bwd": [_P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _F32, _I32, _I32, _I32, _P, _P, _P, _P,
                         _SZ, _P],
    "cpattn_merge": [_I32, _P, _P, _I64, _I32, _I32, _P, _I64, _P, _I32, _P, _P],
    "cpattn_gather_rows": [_P, _I64, _P, _P, _I64, _I64, _P],
    "cpattn_scatter_rows": [_P, _P, _I64, _P, _I64, _I64, _P],
    "cpattn_token_loss_norm": [_P, _P, _I64, _P, _P, _P, _P],
    "cpattn_fwd_flops": [_P, _I32, _I32, _I32, _I32, _P, _P],
    "cpattn_dcp_quotas": [_P, _I32, _I32, _I32, ctypes.c_double, _P],
    "cpattn_dcp_schedule": [_P, _I64, _P, _I32, _P, _P, _P, _P, _P],
    "cpattn_dcp_sweep": [_P, _I64, _P, _I32, _I32, _I32, _I32, _P, _P, _P],
    "cpattn_sync_status": [_P, _P],
    "cpattn_static_sync_status": [_P],
    "cpattn_debug_wait_fault": [ctypes.c_uint32, _I32],
    "cpattn_copy": [_P, _P, _SZ, _I32, _P],
    "cpattn_last_error_string": [],
    "cpattn_version": [],
}


def build(force: bool = False) -> str:
    """Compile libcpattn.so for sm_103a in-tree (nvcc)."""
    from ._build import build as _build
    return _build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded library; raises ImportError if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with context_attention_cpattn_gb300.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_char_p if name in ("cpattn_last_error_string", "cpattn_version") else ctypes.c_int
        _lib = L
    return _lib


def header_functions() -> list:
    """Names of every function declared in include/cpattn.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cpattn_[a-z0-9_]+)\s*\(", text)))


def _check(status: int):
    if status != OK:
        msg = lib().cpattn_last_error_string().decode()
        raise CpattnError(status, msg)


def version() -> str:
    return lib().cpattn_version().decode()


# ------------------------------------------------------------------ plans

class Plan:
    """A context-parallel split (library-owned host object)."""

    def __init__(self, handle, cu_seqlens, cp, mode, grid):
        self._h = handle
        self.cu_seqlens = np.asarray(cu_seqlens, dtype=np.int32)
        self.cp = cp
        self.mode = mode
        self.grid = grid

    @property
    def handle(self):
        return self._h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _lib is not None:
            _lib.cpattn_plan_destroy(h)
            self._h = None

    def info(self) -> dict:
        out = _PlanInfo()
        _check(lib().cpattn_plan_get_info(self._h, ctypes.byref(out)))
        return {f: getattr(out, f) for f, _ in _PlanInfo._fields_ if f != "reserved"}

    def _get(self, fn, n, dtype, *pre):
        out = np.empty(n, dtype=dtype)
        _check(getattr(lib(), fn)(self._h, *pre, out.ctypes.data, n))
        return out

    def chunk_offsets(self):
        return self._get("cpattn_plan_get_chunk_offsets", self.info()["n_chunks"] + 1, np.int64)

    def chunk_ranks(self):
        return self._get("cpattn_plan_get_chunk_ranks", self.info()["n_chunks"], np.int32)

    def rank_offsets(self):
        return self._get("cpattn_plan_get_rank_offsets", self.cp + 1, np.int64)

    def local_cu_seqlens(self, rank: int):
        return self._get("cpattn_plan_get_local_cu_seqlens", len(self.cu_seqlens), np.int32, rank)

    def index_map(self):
        return self._get("cpattn_plan_get_index_map", int(self.cu_seqlens[-1]), np.int64)

    def allowed_pairs(self, causal: bool = True) -> int:
        out = ctypes.c_uint64()
        _check(lib().cpattn_plan_allowed_pairs(self._h, int(bool(causal)), ctypes.byref(out)))
        return int(out.value)

    def a2a_map(self):
        """ULYSSES2D and PAIRED plans: the all-to-all row gather map [u*T]."""
        return self._get("cpattn_plan_get_a2a_map", self.info()["split_h"] * int(self.cu_seqlens[-1]), np.int64)

    def worklist(self, backward: bool, dtype, causal: bool = True, q_rank: int = -1, ring_step: int = 0):
        """The work list a call hands its kernel: (tiles int32 [n, 8] with
        columns row0, pos0, out_row0, rows, run_begin, run_end, pieces, rank;
        runs int32 [m, 4] with columns row0, pos0, len, masked)."""
        args = (self._h, int(bool(backward)), _dtype_code_of(dtype), int(bool(causal)), int(q_rank), int(ring_step))
        nt, nr = ctypes.c_int64(), ctypes.c_int64()
        _check(lib().cpattn_plan_get_worklist(*args, None, 0, None, 0, ctypes.byref(nt), ctypes.byref(nr)))
        tiles = np.zeros((nt.value, 8), dtype=np.int32)
        runs = np.zeros((nr.value, 4), dtype=np.int32)
        _check(lib().cpattn_plan_get_worklist(*args, tiles.ctypes.data, nt.value, runs.ctypes.data, nr.value,
                                              ctypes.byref(nt), ctypes.byref(nr)))
        return tiles, runs

    def ring_schedule(self, causal: bool):
        n = self.cp * self.cp
        kv = np.empty(n, dtype=np.int32)
        kind = np.empty(n, dtype=np.int32)
        _check(lib().cpattn_plan_get_ring_schedule(self._h, int(bool(causal)), kv.ctypes.data, kind.ctypes.data, n))
        return kv.reshape(self.cp, self.cp), kind.reshape(self.cp, self.cp)


def cpattn_plan(cu_seqlens, cp_size: int, mode="zigzag", grid=None) -> Plan:
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    g = _Grid(*grid) if grid is not None else None
    h = ctypes.c_void_p()
    _check(lib().cpattn_plan(cu.ctypes.data, len(cu) - 1, int(cp_size), m,
                             ctypes.byref(g) if g is not None else None, ctypes.byref(h)))
    return Plan(h.value, cu, int(cp_size), m, grid)


def cpattn_plan_2d(cu_seqlens, ulysses: int, ring: int) -> Plan:
    """2D-Attention mesh of ulysses x ring virtual ranks (mode ulysses2d)."""
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    h = ctypes.c_void_p()
    _check(lib().cpattn_plan_2d(cu.ctypes.data, len(cu) - 1, int(ulysses), int(ring), ctypes.byref(h)))
    return Plan(h.value, cu, int(ulysses) * int(ring), MODES["ulysses2d"], (int(ulysses), int(ring)))


def cpattn_plan_paired(cu_seqlens, cp_size: int, n_chunks: int) -> Plan:
    """Clean/noisy time-chunk pairs for teacher forcing (mode paired)."""
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    h = ctypes.c_void_p()
    _check(lib().cpattn_plan_paired(cu.ctypes.data, len(cu) - 1, int(cp_size), int(n_chunks), ctypes.byref(h)))
    return Plan(h.value, cu, int(cp_size), MODES["paired"], (int(n_chunks),))


# ------------------------------------------------------------------ attention

def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_FP32
    raise CpattnError(UNSUPPORTED, f"dtype {t.dtype}")


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def cpattn_workspace_size(plan: Plan, H: int, Hkv: int, D: int, dtype, causal: bool) -> int:
    code = dtype if isinstance(dtype, int) else _dtype_code_of(dtype)
    out = ctypes.c_size_t()
    _check(lib().cpattn_workspace_size(plan.handle, H, Hkv, D, code, int(bool(causal)), ctypes.byref(out)))
    return out.value


def _dtype_code_of(dtype) -> int:
    import torch
    return {torch.bfloat16: DTYPE_BF16, torch.float32: DTYPE_FP32, "bf16": DTYPE_BF16, "fp32": DTYPE_FP32}[dtype]


def cpattn_fwd(plan: Plan, q, k, v, o, lse, workspace, scale: Optional[float] = None, causal: bool = True,
               stream=None):
    """Whole packed forward.  q [T,H,D], k/v [T,Hkv,D], o [T,H,D], lse fp32 [H,T],
    workspace a uint8 device tensor of at least cpattn_workspace_size bytes."""
    T, H, D = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    _check(lib().cpattn_fwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), H, Hkv, D, scale,
                            int(bool(causal)), _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel(),
                            _stream(stream)))


def cpattn_fwd_static(plan: Plan, q, k, v, o, lse, scale: Optional[float] = None, causal: bool = True,
                      stream=None):
    """cpattn_fwd without a workspace, for callers that cannot allocate device
    memory: the scratch is a fixed 8 MiB array inside the library, shared by
    every call (serialise calls; make the first call on a device before any
    stream capture)."""
    T, H, D = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    _check(lib().cpattn_fwd_static(plan.handle, _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), H, Hkv, D, scale,
                                   int(bool(causal)), _ptr(o), _ptr(lse), _stream(stream)))


def cpattn_block_fwd(plan: Plan, q, k, v, o_partial, lse_partial, workspace, q_rank: int, ring_step: int,
                     scale: Optional[float] = None, causal: bool = True, stream=None):
    """One ring step of one virtual rank: fp32 partial O [T_r,H,D] and LSE [H,T_r]."""
    T, H, D = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    _check(lib().cpattn_block_fwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), H, Hkv, D, scale,
                                  int(bool(causal)), int(q_rank), int(ring_step), _ptr(o_partial),
                                  _ptr(lse_partial), _ptr(workspace), workspace.numel(), _stream(stream)))


def cpattn_bwd_workspace_size(plan: Plan, H: int, Hkv: int, D: int, dtype, causal: bool) -> int:
    out = ctypes.c_size_t()
    _check(lib().cpattn_bwd_workspace_size(plan.handle, H, Hkv, D, _dtype_code_of(dtype), int(bool(causal)),
                                           ctypes.byref(out)))
    return int(out.value)


def cpattn_bwd(plan: Plan, q, k, v, o, lse, dout, dq, dk, dv, workspace, scale: Optional[float] = None,
               causal: bool = True, stream=None):
    """Whole packed backward: dq [T,H,D], dk, dv [T,Hkv,D] in the input dtype."""
    T, H, D = q.shape
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    _check(lib().cpattn_bwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                            _dtype_code(q), H, k.shape[1], D, scale, int(bool(causal)), _ptr(dq), _ptr(dk), _ptr(dv),
                            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def cpattn_block_bwd(plan: Plan, q, k, v, o, lse, dout, dq_acc, dk_acc, dv_acc, workspace, q_rank: int,
                     ring_step: int, scale: Optional[float] = None, causal: bool = True, stream=None):
    """One ring step of the backward, added to fp32 accumulators at global rows."""
    T, H, D = q.shape
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    _check(lib().cpattn_block_bwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                  _dtype_code(q), H, k.shape[1], D, scale, int(bool(causal)), q_rank, ring_step,
                                  _ptr(dq_acc), _ptr(dk_acc), _ptr(dv_acc), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def cpattn_merge(o_parts: Sequence, lse_parts: Sequence, o_out, lse_out, out_rows=None, stream=None):
    """Exact LSE merge of fp32 partials o_parts[i] [rows,H,D], lse_parts[i] [H,rows]
    into o_out [out_rows_total,H,D] (fp32 or bf16) and lse_out [H,out_rows_total]."""
    n = len(o_parts)
    rows, H, D = o_parts[0].shape
    op = (ctypes.c_void_p * n)(*[t.data_ptr() for t in o_parts])
    lp = (ctypes.c_void_p * n)(*[t.data_ptr() for t in lse_parts])
    _check(lib().cpattn_merge(n, op, lp, rows, H, D, _ptr(out_rows), o_out.shape[0], _ptr(o_out),
                              _dtype_code(o_out), _ptr(lse_out), _stream(stream)))


def cpattn_gather_rows(src, dst, index, stream=None):
    """dst[i] = src[index[i]] (rows of equal byte size)."""
    row_bytes = dst[0].numel() * dst.element_size() if dst.shape[0] else 16
    _check(lib().cpattn_gather_rows(_ptr(src), src.shape[0], _ptr(dst), _ptr(index), index.numel(), row_bytes,
                                    _stream(stream)))


def cpattn_scatter_rows(src, dst, index, stream=None):
    """dst[index[i]] = src[i] (rows of equal byte size)."""
    row_bytes = src[0].numel() * src.element_size() if src.shape[0] else 16
    _check(lib().cpattn_scatter_rows(_ptr(src), _ptr(dst), dst.shape[0], _ptr(index), index.numel(), row_bytes,
                                     _stream(stream)))


def cpattn_token_loss_norm(loss, valid, out_loss, out_count, out_loss_f32=None, stream=None):
    """out_loss (fp64 [1]) = mean of loss over valid tokens; out_count (int64 [1]) = valid tokens."""
    _check(lib().cpattn_token_loss_norm(_ptr(loss), _ptr(valid), loss.numel(), _ptr(out_loss), _ptr(out_count),
                                        _ptr(out_loss_f32), _stream(stream)))


def cpattn_fwd_flops(cu_seqlens, H: int, D: int, causal: bool) -> int:
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    out = ctypes.c_uint64()
    _check(lib().cpattn_fwd_flops(cu.ctypes.data, len(cu) - 1, H, D, int(bool(causal)), ctypes.byref(out), None))
    return int(out.value)


def cpattn_sync_status(workspace=None, stream=None):
    _check(lib().cpattn_sync_status(_ptr(workspace), _stream(stream)))


def cpattn_copy(dst, src, n_blocks: int = 0, stream=None):
    """dst <- src with a copy kernel; either tensor may be pinned host memory
    (read or written by the GPU over the host link)."""
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("dst and src sizes differ")
    _check(lib().cpattn_copy(_ptr(dst), _ptr(src), nbytes, int(n_blocks), _stream(stream)))


def cpattn_debug_wait_fault(wait_limit_us: int, withhold_first_v: bool = False):
    """Fault-path test support: a short limit on every bounded kernel wait and,
    optionally, a withheld V load in the bf16 forward (see the C header)."""
    _check(lib().cpattn_debug_wait_fault(int(wait_limit_us), int(bool(withhold_first_v))))


def cpattn_static_sync_status(stream=None):
    """Fault word of cpattn_fwd_static's static array on the current device."""
    _check(lib().cpattn_static_sync_status(_stream(stream)))


# ------------------------------------------------------ Dynamic-CP scheduler

def _dcp_config(max_cp, cap_tokens, attn_coef, lin_coef):
    return _DcpConfig(int(max_cp), 0, int(cap_tokens), int(attn_coef), int(lin_coef))


def _seqlens(lengths):
    return np.ascontiguousarray(np.asarray(lengths, dtype=np.int64))


def cpattn_dcp_quotas(m, vpp: int, pp: int, total: float) -> np.ndarray:
    """Per-micro-batch workload of each DP rank from its micro-batch count m[i] (Eq. 1-3)."""
    mm = np.ascontiguousarray(np.asarray(m, dtype=np.int32))
    out = np.empty(len(mm), dtype=np.float64)
    _check(lib().cpattn_dcp_quotas(mm.ctypes.data, len(mm), vpp, pp, float(total), out.ctypes.data))
    return out


def cpattn_dcp_schedule(lengths, n_micro: int, max_cp: int, cap_tokens: int, attn_coef: int, lin_coef: int = 0):
    """Micro-batch and CP size of each sample, and each micro-batch's CP size, workload and tokens."""
    L = _seqlens(lengths)
    n = len(L)
    cfg = _dcp_config(max_cp, cap_tokens, attn_coef, lin_coef)
    out = {"sample_micro": np.empty(n, np.int32), "sample_cp": np.empty(n, np.int32),
           "micro_cp": np.empty(n_micro, np.int32), "micro_work": np.empty(n_micro, np.int64),
           "micro_tokens": np.empty(n_micro, np.int64)}
    _check(lib().cpattn_dcp_schedule(L.ctypes.data, n, ctypes.byref(cfg), n_micro,
                                     *[out[k].ctypes.data for k in ("sample_micro", "sample_cp", "micro_cp",
                                                                     "micro_work", "micro_tokens")]))
    return out


def cpattn_dcp_sweep(lengths, dp: int, pp: int, vpp: int, mult: int, max_cp: int, cap_tokens: int,
                     attn_coef: int, lin_coef: int = 0):
    """Budget curve over m = pp..mult*pp micro-batches per DP rank, its knee and the chosen m."""
    L = _seqlens(lengths)
    cfg = _dcp_config(max_cp, cap_tokens, attn_coef, lin_coef)
    budgets = np.empty((mult - 1) * pp + 1, np.int64)
    knee, best = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().cpattn_dcp_sweep(L.ctypes.data, len(L), ctypes.byref(cfg), dp, pp, vpp, mult,
                                  budgets.ctypes.data, ctypes.byref(knee), ctypes.byref(best)))
    return {"m": np.arange(pp, mult * pp + 1), "budgets": budgets, "knee_m": knee.value, "best_m": best.value}


def dcp_micro_batches(lengths, schedule) -> list:
    """Each micro-batch as (sample ids in ascending order, cu_seqlens, cp size), ready for cpattn_plan."""
    L = _seqlens(lengths)
    out = []
    for b, cp in enumerate(schedule["micro_cp"]):
        ids = np.flatnonzero(schedule["sample_micro"] == b)
        cu = np.concatenate([[0], np.cumsum(L[ids])]).astype(np.int32)
        out.append((ids, cu, int(cp)))
    return out
