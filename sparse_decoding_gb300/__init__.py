"""GB300-native bitmask N:M decode SpMV (the decode kernel of SparseDecoding).

This package is a thin ctypes binding over ``libnmspmv.so`` (C ABI in
``include/nmspmv.h``). Every step of the computation runs in the library's
CUDA kernels; this module only checks tensor types and passes pointers, sizes
and the current CUDA stream. PyTorch supplies device memory and streams.

There is no fallback: if the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# NM_LIBRARY may name another build of the library (the bounds-checking one).
LIB_PATH = os.environ.get("NM_LIBRARY") or os.path.join(_HERE, "libnmspmv.so")

NM_OK = 0
NM_ERR_INVALID_ARG = 1
NM_ERR_SHAPE = 2
NM_ERR_ALIGN = 3
NM_ERR_UNSUPPORTED = 4
NM_ERR_NOT_NM = 5
NM_ERR_CUDA = 6
NM_ERR_TIMEOUT = 7
NM_ERR_NOT_PD = 8
NM_ERR_BOUNDS = 9

PATTERNS = ((2, 4), (4, 8), (8, 16), (16, 32))

NM_STACK_DENSE = 1
NM_STACK_PERSISTENT = 2
NM_LINEAR_SWIGLU = 1
NM_LINEAR_QKV = 2
NM_OBS_SGEMM = 1

# Every symbol the header declares (the CPU test checks they are exported).
EXPORTS = ("nm_abi_version", "nm_status_str", "nm_pack_host", "nm_select", "nm_pack", "nm_spmv",
           "nm_spmv_f32out", "dense_gemv", "dense_gemv_f32out", "nm_spmv_stack", "dense_gemv_stack",
           "nm_device_status", "nm_spmv_noalloc", "nm_stack_plan_create", "nm_stack_plan_run",
           "nm_stack_plan_destroy", "nm_pack_swiglu", "nm_spmv_swiglu", "nm_obs_hessian", "nm_obs_prune",
           "nm_spmv_f32out_atomic", "nm_select_pack", "nm_spmv_qkv", "nm_obs_release_workspace")


class NmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} (status {status})")


class NmLinear(ctypes.Structure):
    """Mirror of ``nm_linear`` in include/nmspmv.h."""
    _fields_ = [("masks", ctypes.c_void_p), ("values", ctypes.c_void_p), ("W", ctypes.c_void_p),
                ("x", ctypes.c_void_p), ("y", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("K", ctypes.c_int64), ("flags", ctypes.c_uint32), ("y_k", ctypes.c_void_p),
                ("y_v", ctypes.c_void_p), ("rows_q", ctypes.c_int64), ("rows_k", ctypes.c_int64)]


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load libnmspmv.so (built by ``sparse_decoding_gb300.build``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -m sparse_decoding_gb300.build` "
                           "(or __graft_entry__.build()) first")
    L = ctypes.CDLL(LIB_PATH)
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    sig = {
        "nm_abi_version": ([], i32),
        "nm_status_str": ([i32], ctypes.c_char_p),
        "nm_pack_host": ([p, i64, i64, i32, i32, p, p], i32),
        "nm_select": ([p, p, i64, i64, i32, i32, p, p], i32),
        "nm_pack": ([p, i64, i64, i32, i32, p, p, p], i32),
        "nm_select_pack": ([p, p, i64, i64, i32, i32, p, p, p], i32),
        "nm_spmv": ([p, p, p, p, i64, i64, i32, p], i32),
        "nm_spmv_f32out": ([p, p, p, p, i64, i64, i32, p], i32),
        "nm_spmv_f32out_atomic": ([p, p, p, p, i64, i64, i32, p], i32),
        "nm_spmv_qkv": ([p, p, p, p, p, p, i64, i64, i64, i64, i32, p], i32),
        "dense_gemv": ([p, p, p, i64, i64, i32, p], i32),
        "dense_gemv_f32out": ([p, p, p, i64, i64, i32, p], i32),
        "nm_spmv_stack": ([ctypes.POINTER(NmLinear), i32, i32, p], i32),
        "dense_gemv_stack": ([ctypes.POINTER(NmLinear), i32, i32, p], i32),
        "nm_device_status": ([p], i32),
        "nm_spmv_noalloc": ([p, p, p, p, i64, i64, i32, p], i32),
        "nm_stack_plan_create": ([ctypes.POINTER(NmLinear), i32, i32, ctypes.c_uint, ctypes.POINTER(p)], i32),
        "nm_stack_plan_run": ([p, p], i32),
        "nm_stack_plan_destroy": ([p], i32),
        "nm_pack_swiglu": ([p, p, i64, i64, i32, i32, p, p, p], i32),
        "nm_spmv_swiglu": ([p, p, p, p, i64, i64, i32, p], i32),
        "nm_obs_hessian": ([p, i64, i64, p, i32, p], i32),
        "nm_obs_prune": ([p, p, i64, i64, i32, i32, ctypes.c_float, ctypes.c_uint, p, p, p, p], i32),
        "nm_obs_release_workspace": ([], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def status_str(status: int) -> str:
    return lib().nm_status_str(int(status)).decode()


def _check(status: int, where: str):
    if status != NM_OK:
        raise NmError(status, where)


def _stream(t: Optional[torch.Tensor] = None) -> int:
    dev = t.device if t is not None else None
    return torch.cuda.current_stream(dev).cuda_stream


def _cuda(t: torch.Tensor, dtype, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise TypeError(f"{name} must be contiguous")
    return t


def _x2d(x: torch.Tensor) -> torch.Tensor:
    return x.unsqueeze(0) if x.dim() == 1 else x


# --- calls ---------------------------------------------------------------------

def init(device: Optional[torch.device] = None) -> None:
    """Allocate the per-device scratch now (do this before any CUDA graph capture)."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _check(lib().nm_device_status(ctypes.c_void_p(_stream())), "nm_device_status")


def device_status() -> int:
    """Wait for the current stream; return and clear the device status word."""
    return lib().nm_device_status(ctypes.c_void_p(_stream()))


def select(W: torch.Tensor, a: torch.Tensor, N: int, M: int, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Wanda N:M selection on the GPU: keep the N largest |W|*a_j per M-column subgroup."""
    _cuda(W, torch.bfloat16, "W")
    _cuda(a, torch.float32, "a")
    rows, K = W.shape
    out = torch.empty_like(W) if out is None else _cuda(out, torch.bfloat16, "out")
    _check(lib().nm_select(W.data_ptr(), a.data_ptr(), rows, K, N, M, out.data_ptr(),
                           ctypes.c_void_p(_stream(W))), "nm_select")
    return out


def select_pack(W: torch.Tensor, a: torch.Tensor, N: int, M: int):
    """Wanda N:M selection and pack in one pass: dense W (bf16, CUDA) and column norms a (fp32)
    -> (masks int32-viewed uint32 [rows][K/32], values bf16 [rows][K/2]); equal to pack(select(W, a))."""
    _cuda(W, torch.bfloat16, "W")
    _cuda(a, torch.float32, "a")
    rows, K = W.shape
    masks = torch.empty(rows, K // 32, dtype=torch.int32, device=W.device)
    values = torch.empty(rows, K // 2, dtype=torch.bfloat16, device=W.device)
    _check(lib().nm_select_pack(W.data_ptr(), a.data_ptr(), rows, K, N, M, masks.data_ptr(), values.data_ptr(),
                                ctypes.c_void_p(_stream(W))), "nm_select_pack")
    return masks, values


def pack(W: torch.Tensor, N: int, M: int):
    """Pruned dense W (bf16, CUDA) -> (masks int32-viewed uint32 [rows][K/32], values bf16 [rows][K/2])."""
    _cuda(W, torch.bfloat16, "W")
    rows, K = W.shape
    masks = torch.empty(rows, K // 32, dtype=torch.int32, device=W.device)
    values = torch.empty(rows, K // 2, dtype=torch.bfloat16, device=W.device)
    _check(lib().nm_pack(W.data_ptr(), rows, K, N, M, masks.data_ptr(), values.data_ptr(),
                         ctypes.c_void_p(_stream(W))), "nm_pack")
    return masks, values


def pack_host(W: torch.Tensor, N: int, M: int):
    """Host packer: CPU bf16 W -> CPU (masks int32-viewed uint32, values bf16)."""
    if W.is_cuda or W.dtype != torch.bfloat16 or not W.is_contiguous():
        raise TypeError("W must be a contiguous CPU bf16 tensor")
    rows, K = W.shape
    masks = torch.empty(rows, K // 32, dtype=torch.int32)
    values = torch.empty(rows, K // 2, dtype=torch.bfloat16)
    _check(lib().nm_pack_host(W.data_ptr(), rows, K, N, M, masks.data_ptr(), values.data_ptr()), "nm_pack_host")
    return masks, values


def spmv(masks: torch.Tensor, values: torch.Tensor, x: torch.Tensor, out: Optional[torch.Tensor] = None,
         f32: bool = False, atomic: bool = False) -> torch.Tensor:
    """y[b][r] = sum_j W[r][j] x[b][j] over the bitmask format; bf16 (or fp32 with f32=True).

    atomic=True (fp32 only): the split-K variant that combines row-block parts
    with atomicAdd (nm_spmv_f32out_atomic)."""
    if atomic and not f32:
        raise ValueError("the atomicAdd split-K variant writes fp32 (f32=True)")
    _cuda(masks, torch.int32, "masks")
    _cuda(values, torch.bfloat16, "values")
    x = _cuda(_x2d(x), torch.bfloat16, "x")
    rows = masks.shape[0]
    K = masks.shape[1] * 32
    batch = x.shape[0]
    if values.shape != (rows, K // 2) or x.shape[1] != K:
        raise ValueError("shape mismatch between masks, values and x")
    odt = torch.float32 if f32 else torch.bfloat16
    out = torch.empty(batch, rows, dtype=odt, device=x.device) if out is None else _cuda(out, odt, "out")
    name = "nm_spmv_f32out_atomic" if atomic else "nm_spmv_f32out" if f32 else "nm_spmv"
    _check(getattr(lib(), name)(masks.data_ptr(), values.data_ptr(), x.data_ptr(), out.data_ptr(), rows, K, batch,
                                ctypes.c_void_p(_stream(x))), name)
    return out


def spmv_qkv(masks: torch.Tensor, values: torch.Tensor, x: torch.Tensor, rows_q: int, rows_k: int,
             out: Optional[Sequence[torch.Tensor]] = None):
    """The SpMV of a fused q/k/v matrix (q rows, then k rows, then v rows) into three bf16
    buffers q [batch][rows_q], k [batch][rows_k], v [batch][rows_v]; returns (q, k, v)."""
    _cuda(masks, torch.int32, "masks")
    _cuda(values, torch.bfloat16, "values")
    x = _cuda(_x2d(x), torch.bfloat16, "x")
    rows = masks.shape[0]
    K = masks.shape[1] * 32
    batch = x.shape[0]
    rows_v = rows - rows_q - rows_k
    if values.shape != (rows, K // 2) or x.shape[1] != K or rows_q < 0 or rows_k < 0 or rows_v < 0:
        raise ValueError("shape mismatch between masks, values, x and the q/k/v row counts")
    if out is None:
        out = [torch.empty(batch, r, dtype=torch.bfloat16, device=x.device) for r in (rows_q, rows_k, rows_v)]
    q, k, v = (_cuda(t, torch.bfloat16, n) for t, n in zip(out, ("q", "k", "v")))
    _check(lib().nm_spmv_qkv(masks.data_ptr(), values.data_ptr(), x.data_ptr(), q.data_ptr(), k.data_ptr(),
                             v.data_ptr(), rows_q, rows_k, rows_v, K, batch, ctypes.c_void_p(_stream(x))),
           "nm_spmv_qkv")
    return q, k, v


def pack_swiglu(W_gate: torch.Tensor, W_up: torch.Tensor, N: int, M: int):
    """Pruned gate and up matrices (bf16, CUDA, [rows_h][K]) -> (masks, values) in the pair
    layout of nm_pack_swiglu: [2*rows_h][K/32] and [2*rows_h][K/2]."""
    _cuda(W_gate, torch.bfloat16, "W_gate")
    _cuda(W_up, torch.bfloat16, "W_up")
    if W_gate.shape != W_up.shape:
        raise ValueError("W_gate and W_up must have the same shape")
    rows_h, K = W_gate.shape
    masks = torch.empty(2 * rows_h, K // 32, dtype=torch.int32, device=W_gate.device)
    values = torch.empty(2 * rows_h, K // 2, dtype=torch.bfloat16, device=W_gate.device)
    _check(lib().nm_pack_swiglu(W_gate.data_ptr(), W_up.data_ptr(), rows_h, K, N, M, masks.data_ptr(),
                                values.data_ptr(), ctypes.c_void_p(_stream(W_gate))), "nm_pack_swiglu")
    return masks, values


def spmv_swiglu(masks: torch.Tensor, values: torch.Tensor, x: torch.Tensor,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """h[b][r] = bf16(silu(g) * u), g and u the gate and up rows of a pair-layout matrix times x."""
    _cuda(masks, torch.int32, "masks")
    _cuda(values, torch.bfloat16, "values")
    x = _cuda(_x2d(x), torch.bfloat16, "x")
    rows = masks.shape[0]
    K = masks.shape[1] * 32
    batch = x.shape[0]
    if values.shape != (rows, K // 2) or x.shape[1] != K or rows % 32 != 0:
        raise ValueError("shape mismatch between masks, values and x (rows must be a multiple of 32)")
    out = torch.empty(batch, rows // 2, dtype=torch.bfloat16, device=x.device) if out is None else \
        _cuda(out, torch.bfloat16, "out")
    _check(lib().nm_spmv_swiglu(masks.data_ptr(), values.data_ptr(), x.data_ptr(), out.data_ptr(), rows // 2, K,
                                batch, ctypes.c_void_p(_stream(x))), "nm_spmv_swiglu")
    return out


def dense_gemv(W: torch.Tensor, x: torch.Tensor, out: Optional[torch.Tensor] = None,
               f32: bool = False) -> torch.Tensor:
    """Dense bf16 reference: y[b][r] = sum_j W[r][j] x[b][j]."""
    _cuda(W, torch.bfloat16, "W")
    x = _cuda(_x2d(x), torch.bfloat16, "x")
    rows, K = W.shape
    batch = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("shape mismatch between W and x")
    odt = torch.float32 if f32 else torch.bfloat16
    out = torch.empty(batch, rows, dtype=odt, device=x.device) if out is None else _cuda(out, odt, "out")
    fn = lib().dense_gemv_f32out if f32 else lib().dense_gemv
    _check(fn(W.data_ptr(), x.data_ptr(), out.data_ptr(), rows, K, batch, ctypes.c_void_p(_stream(x))),
           "dense_gemv")
    return out


def _linear_array(ops: Sequence[dict]) -> ctypes.Array:
    arr = (NmLinear * len(ops))()
    for i, op in enumerate(ops):
        t = arr[i]
        for f in ("masks", "values", "W", "x", "y"):
            v = op.get(f)
            setattr(t, f, v.data_ptr() if v is not None else None)
        t.rows = int(op["rows"])
        t.K = int(op["K"])
        t.flags = int(op.get("flags", 0))
        for f in ("y_k", "y_v"):
            v = op.get(f)
            setattr(t, f, v.data_ptr() if v is not None else None)
        t.rows_q = int(op.get("rows_q", 0))
        t.rows_k = int(op.get("rows_k", 0))
    return arr


def spmv_stack(ops: Sequence[dict], batch: int) -> None:
    """Run a decode-token linear stack: ops[i] = {masks, values, x, y, rows, K}, in order."""
    arr = _linear_array(ops)
    _check(lib().nm_spmv_stack(arr, len(ops), batch, ctypes.c_void_p(_stream())), "nm_spmv_stack")


def dense_gemv_stack(ops: Sequence[dict], batch: int) -> None:
    """Dense counterpart of spmv_stack: ops[i] = {W, x, y, rows, K}."""
    arr = _linear_array(ops)
    _check(lib().dense_gemv_stack(arr, len(ops), batch, ctypes.c_void_p(_stream())), "dense_gemv_stack")


class StackPlan:
    """A decode-token stack prepared once (``nm_stack_plan``); ``run()`` launches it.

    By default each op is its own kernel, chained with programmatic dependent
    launch; with ``persistent=True`` the whole stack is one persistent kernel
    launch with a grid barrier between ops (when every op is on the TMA path).
    The plan holds the ops' device pointers: it keeps their tensors alive
    until ``close()``.
    """

    def __init__(self, ops: Sequence[dict], batch: int, dense: bool = False, persistent: bool = False):
        self._keep = list(ops)
        self.batch = batch
        self.dense = dense
        arr = _linear_array(self._keep)
        flags = (NM_STACK_DENSE if dense else 0) | (NM_STACK_PERSISTENT if persistent else 0)
        h = ctypes.c_void_p()
        _check(lib().nm_stack_plan_create(arr, len(self._keep), batch, flags, ctypes.byref(h)),
               "nm_stack_plan_create")
        self._h = h

    def run(self) -> None:
        if self._h is None:
            raise RuntimeError("StackPlan is closed")
        _check(lib().nm_stack_plan_run(self._h, ctypes.c_void_p(_stream())), "nm_stack_plan_run")

    def close(self) -> None:
        if getattr(self, "_h", None) is not None:
            h, self._h = self._h, None
            _check(lib().nm_stack_plan_destroy(h), "nm_stack_plan_destroy")
            self._keep = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# --- N:M pruning by the OBS rule --------------------------------------------------

def obs_hessian(X: torch.Tensor, H: Optional[torch.Tensor] = None, accumulate: bool = False) -> torch.Tensor:
    """H = 2 X^T X (or H += 2 X^T X) for calibration inputs X, bf16 [T][K] -> fp32 [K][K]."""
    _cuda(X, torch.bfloat16, "X")
    T, K = X.shape
    if H is None:
        if accumulate:
            raise ValueError("accumulate needs H")
        H = torch.empty(K, K, dtype=torch.float32, device=X.device)
    _cuda(H, torch.float32, "H")
    if tuple(H.shape) != (K, K):
        raise ValueError("H must be [K][K]")
    _check(lib().nm_obs_hessian(X.data_ptr(), T, K, H.data_ptr(), int(bool(accumulate)),
                                ctypes.c_void_p(_stream(X))), "nm_obs_hessian")
    return H


def obs_prune(W: torch.Tensor, H: torch.Tensor, N: int, M: int, percdamp: float = 0.01, sgemm: bool = False,
              masks: bool = True, f32: bool = False):
    """OBS N:M pruning of W (bf16 [rows][K]) against H (fp32 [K][K]). Synchronous.

    Returns (W_pruned bf16 [rows][K], keep masks int32-viewed uint32 [rows][K/32] or
    None, W_pruned fp32 or None)."""
    _cuda(W, torch.bfloat16, "W")
    _cuda(H, torch.float32, "H")
    rows, K = W.shape
    if tuple(H.shape) != (K, K):
        raise ValueError("H must be [K][K]")
    out = torch.empty_like(W)
    m = torch.empty(rows, K // 32, dtype=torch.int32, device=W.device) if masks else None
    wf = torch.empty(rows, K, dtype=torch.float32, device=W.device) if f32 else None
    _check(lib().nm_obs_prune(W.data_ptr(), H.data_ptr(), rows, K, N, M, float(percdamp),
                              NM_OBS_SGEMM if sgemm else 0, out.data_ptr(),
                              m.data_ptr() if m is not None else None,
                              wf.data_ptr() if wf is not None else None,
                              ctypes.c_void_p(_stream(W))), "nm_obs_prune")
    return out, m, wf


def obs_release_workspace():
    """Return the memory the OBS calls keep for their workspaces on the current device."""
    _check(lib().nm_obs_release_workspace(), "nm_obs_release_workspace")
