"""CPU oracle for the bitmask N:M decode SpMV (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product library never calls it and shares no
code with it. The arithmetic lives in ``nm_oracle.c`` (plain C, fp64), which
cites the pages it follows; this file only compiles it with gcc and marshals
numpy arrays into it.

bf16 tensors cross this boundary as ``numpy.uint16`` arrays of raw bits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nm_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libnm_oracle.so")

_STATUS = {0: "ok", 1: "bad argument", 2: "bad shape", 4: "unsupported N:M",
           5: "more than N nonzeros in an M-subgroup", 7: "mask word without 16 set bits"}


class OracleError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {_STATUS.get(code, code)} (status {code})")
        self.code = code


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no CUDA, no -ffast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        _lib.oracle_select.argtypes = [p, p, i64, i64, i32, i32, p]
        _lib.oracle_pack.argtypes = [p, i64, i64, i32, i32, p, p]
        _lib.oracle_unpack.argtypes = [p, p, i64, i64, p]
        _lib.oracle_spmv_f64.argtypes = [p, p, i64, i64, i32, p, p]
        _lib.oracle_swiglu_f64.argtypes = [p, p, i64, p]
        _lib.oracle_pair_rows.argtypes = [p, p, i64, i64, p]
        for f in (_lib.oracle_select, _lib.oracle_pack, _lib.oracle_unpack, _lib.oracle_spmv_f64,
                  _lib.oracle_swiglu_f64, _lib.oracle_pair_rows):
            f.restype = ctypes.c_int
    return _lib


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected raw bf16 bits as uint16, got {a.dtype}")
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(code: int, where: str):
    if code != 0:
        raise OracleError(code, where)


def select(W_bits, a, N: int, M: int) -> np.ndarray:
    """Wanda N:M selection: keep the N largest |W|*a_j per aligned M-subgroup."""
    W_bits = _u16(W_bits)
    rows, K = W_bits.shape
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    assert a.shape == (K,)
    out = np.empty_like(W_bits)
    _check(lib().oracle_select(_ptr(W_bits), _ptr(a), rows, K, N, M, _ptr(out)), "oracle_select")
    return out


def pack(W_bits, N: int, M: int):
    """Pruned dense W -> (masks uint32[rows][K/32], values uint16[rows][K/2])."""
    W_bits = _u16(W_bits)
    rows, K = W_bits.shape
    masks = np.empty((rows, K // 32), dtype=np.uint32)
    values = np.empty((rows, K // 2), dtype=np.uint16)
    _check(lib().oracle_pack(_ptr(W_bits), rows, K, N, M, _ptr(masks), _ptr(values)), "oracle_pack")
    return masks, values


def unpack(masks, values, K: int) -> np.ndarray:
    """(masks, values) -> dense bf16 bits, +0 at pruned positions."""
    masks = np.ascontiguousarray(np.asarray(masks, dtype=np.uint32))
    values = _u16(values)
    rows = masks.shape[0]
    assert masks.shape == (rows, K // 32) and values.shape == (rows, K // 2)
    W = np.empty((rows, K), dtype=np.uint16)
    _check(lib().oracle_unpack(_ptr(masks), _ptr(values), rows, K, _ptr(W)), "oracle_unpack")
    return W


def spmv_f64(W_bits, x_bits):
    """y[b][r] = sum_j W[r][j] x[b][j] in fp64 (index order), and S = sum |W x|.

    ``x_bits`` is ``[batch][K]``; returns (y, S), both ``[batch][rows]`` float64.
    """
    W_bits = _u16(W_bits)
    x_bits = _u16(x_bits)
    if x_bits.ndim == 1:
        x_bits = x_bits[None, :]
    rows, K = W_bits.shape
    batch = x_bits.shape[0]
    assert x_bits.shape == (batch, K)
    y = np.empty((batch, rows), dtype=np.float64)
    S = np.empty((batch, rows), dtype=np.float64)
    _check(lib().oracle_spmv_f64(_ptr(W_bits), _ptr(x_bits), rows, K, batch, _ptr(y), _ptr(S)),
           "oracle_spmv_f64")
    return y, S


def spmv_packed_f64(masks, values, x_bits, K: int):
    """The oracle's product from the packed format: decode, then the dense fp64 product."""
    return spmv_f64(unpack(masks, values, K), x_bits)


def swiglu_f64(g, u) -> np.ndarray:
    """h = silu(g) * u elementwise in fp64, silu(g) = g / (1 + exp(-g))."""
    g = np.ascontiguousarray(np.asarray(g, dtype=np.float64))
    u = np.ascontiguousarray(np.asarray(u, dtype=np.float64))
    assert g.shape == u.shape
    h = np.empty_like(g)
    _check(lib().oracle_swiglu_f64(_ptr(g), _ptr(u), g.size, _ptr(h)), "oracle_swiglu_f64")
    return h


def pair_rows(Wg_bits, Wu_bits) -> np.ndarray:
    """The pair layout: row block t holds gate rows 16t..16t+15, then up rows 16t..16t+15."""
    Wg_bits = _u16(Wg_bits)
    Wu_bits = _u16(Wu_bits)
    assert Wg_bits.shape == Wu_bits.shape
    rows_h, K = Wg_bits.shape
    out = np.empty((2 * rows_h, K), dtype=np.uint16)
    _check(lib().oracle_pair_rows(_ptr(Wg_bits), _ptr(Wu_bits), rows_h, K, _ptr(out)), "oracle_pair_rows")
    return out


def spmv_swiglu_f64(Wg_bits, Wu_bits, x_bits):
    """The fused gate/up SpMV with SwiGLU: (h, g, u, Sg, Su), each [batch][rows_h] float64."""
    g, Sg = spmv_f64(Wg_bits, x_bits)
    u, Su = spmv_f64(Wu_bits, x_bits)
    return swiglu_f64(g, u), g, u, Sg, Su
