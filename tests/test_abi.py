"""CPU checks of the C ABI: the library loads, exports every symbol that
include/nmspmv.h declares, validates arguments before touching the GPU, and
its host packer is bit-exact with the oracle's packer. No GPU compute here."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.bits import to_bits

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nmspmv.h")


@pytest.fixture(scope="module")
def nm():
    from sparse_decoding_gb300 import build
    build.build()
    import sparse_decoding_gb300 as nm
    nm.lib()
    return nm


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(\w+)\s*\([^;{]*\)\s*;", text)) - {"if", "sizeof"})


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("nm_pack_host", "nm_select", "nm_pack", "nm_spmv", "nm_spmv_f32out", "dense_gemv",
              "nm_spmv_stack", "dense_gemv_stack", "nm_device_status", "nm_status_str", "nm_abi_version"):
        assert n in names, n


def test_linear_struct_matches_header(nm):
    """nm_linear: five pointers, two int64, one uint32 (padded to 8 bytes), then the
    q/k/v split fields: two pointers, two int64."""
    assert ctypes.sizeof(nm.NmLinear) == 5 * 8 + 2 * 8 + 8 + 2 * 8 + 2 * 8
    assert nm.NmLinear.y_k.offset == 64 and nm.NmLinear.rows_k.offset == 88
    assert nm.lib().nm_abi_version() == 4
    text = open(HEADER).read()
    assert "uint32_t flags;" in text and "#define NM_LINEAR_SWIGLU 1u" in text and "#define NM_LINEAR_QKV 2u" in text
    body = text[text.index("typedef struct nm_linear {"):text.index("} nm_linear;")]
    fields = re.findall(r"(\w+);", re.sub(r"/\*.*?\*/", "", body, flags=re.S))
    assert fields == ["masks", "values", "W", "x", "y", "rows", "K", "flags", "y_k", "y_v", "rows_q", "rows_k"], fields


def test_library_exports_every_declared_symbol(nm):
    L = nm.lib()
    for name in declared_functions():
        assert hasattr(L, name), f"libnmspmv.so does not export {name}"
    assert set(declared_functions()) <= set(nm.EXPORTS), set(declared_functions()) - set(nm.EXPORTS)
    assert L.nm_abi_version() == 4


def test_status_strings(nm):
    for code in range(10):
        assert nm.status_str(code) != "unknown status"
    assert nm.status_str(10) == "unknown status"
    assert nm.status_str(5).startswith("an M-subgroup")


@pytest.mark.parametrize("N,M", synth.PATTERNS)
def test_host_pack_bit_exact_with_oracle(nm, N, M):
    rows, K = 67, 4096
    W = synth.weights(rows, K, seed=21)
    a = synth.col_norms(K, seed=21).numpy()
    Wp = oracle.select(to_bits(W), a, N, M)
    om, ov = oracle.pack(Wp, N, M)
    Wt = torch.from_numpy(Wp.view(np.int16)).view(torch.bfloat16)
    masks, values = nm.pack_host(Wt, N, M)
    np.testing.assert_array_equal(masks.numpy().view(np.uint32), om)
    np.testing.assert_array_equal(to_bits(values), ov)


def test_host_pack_fill_rule_and_errors(nm):
    W = np.zeros((2, 64), dtype=np.uint16)
    W[0, 2] = 0x4000
    W[0, 0] = 0x8000  # -0.0: zero, becomes the filler
    W[1, :] = 0x3F80  # every entry nonzero: more than N
    Wt = torch.from_numpy(W[:1].copy().view(np.int16)).view(torch.bfloat16)
    masks, values = nm.pack_host(Wt, 8, 16)
    om, ov = oracle.pack(W[:1], 8, 16)
    np.testing.assert_array_equal(masks.numpy().view(np.uint32), om)
    np.testing.assert_array_equal(to_bits(values), ov)
    bad = torch.from_numpy(W[1:].copy().view(np.int16)).view(torch.bfloat16)
    with pytest.raises(nm.NmError) as e:
        nm.pack_host(bad, 8, 16)
    assert e.value.status == nm.NM_ERR_NOT_NM
    with pytest.raises(nm.NmError) as e:
        nm.pack_host(bad, 3, 8)
    assert e.value.status == nm.NM_ERR_UNSUPPORTED


def test_argument_validation_before_any_cuda_call(nm):
    """These calls must fail on their arguments alone (no device is touched)."""
    L = nm.lib()
    buf = (ctypes.c_uint8 * 4096)()
    p = ctypes.addressof(buf)
    p16 = (p + 15) & ~15
    # K not a multiple of 32
    assert L.nm_spmv(p16, p16, p16, p16, 4, 48, 1, None) == nm.NM_ERR_SHAPE
    assert L.dense_gemv(p16, p16, p16, 4, 48, 1, None) == nm.NM_ERR_SHAPE
    # batch outside 1..8
    assert L.nm_spmv(p16, p16, p16, p16, 4, 64, 9, None) == nm.NM_ERR_UNSUPPORTED
    assert L.nm_spmv(p16, p16, p16, p16, 4, 64, 0, None) == nm.NM_ERR_UNSUPPORTED
    # misaligned pointer
    assert L.nm_spmv(p16 + 2, p16, p16, p16, 4, 64, 1, None) == nm.NM_ERR_ALIGN
    assert L.nm_spmv_f32out(p16, p16, p16, p16 + 4, 4, 64, 1, None) == nm.NM_ERR_ALIGN
    assert L.dense_gemv(p16, p16 + 8, p16, 4, 64, 1, None) == nm.NM_ERR_ALIGN
    # NULL data pointer
    assert L.nm_spmv(None, p16, p16, p16, 4, 64, 1, None) == nm.NM_ERR_INVALID_ARG
    # unsupported pattern
    assert L.nm_pack(p16, 4, 64, 3, 4, p16, p16, None) == nm.NM_ERR_UNSUPPORTED
    assert L.nm_select(p16, p16, 4, 64, 2, 8, p16, None) == nm.NM_ERR_UNSUPPORTED
    # empty problems succeed without work
    assert L.nm_spmv(None, None, None, None, 0, 64, 1, None) == nm.NM_OK
    assert L.nm_pack(None, 0, 64, 2, 4, None, None, None) == nm.NM_OK
    # negative sizes
    assert L.nm_spmv(p16, p16, p16, p16, -1, 64, 1, None) == nm.NM_ERR_SHAPE
    # a stack is validated as a whole before anything is launched
    ops = (nm.NmLinear * 2)()
    for o in ops:
        o.masks = o.values = o.x = o.y = p16
        o.rows, o.K = 4, 64
    ops[1].K = 40
    assert L.nm_spmv_stack(ops, 2, 1, None) == nm.NM_ERR_SHAPE
    assert L.nm_spmv_stack(None, 1, 1, None) == nm.NM_ERR_INVALID_ARG
    # a plan is validated before any device work as well
    h = ctypes.c_void_p()
    assert L.nm_stack_plan_create(ops, 2, 1, 0, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_stack_plan_create(ops, -1, 1, 0, ctypes.byref(h)) == nm.NM_ERR_INVALID_ARG
    assert L.nm_stack_plan_create(ops, 2, 1, 0, ctypes.byref(h)) == nm.NM_ERR_SHAPE
    assert L.nm_stack_plan_create(ops, 1, 9, 0, ctypes.byref(h)) == nm.NM_ERR_UNSUPPORTED
    assert L.nm_stack_plan_create(None, 0, 0, 0, ctypes.byref(h)) == nm.NM_ERR_UNSUPPORTED
    assert L.nm_stack_plan_create(ops, 1, 1, 4, ctypes.byref(h)) == nm.NM_ERR_INVALID_ARG  # unknown flag
    assert h.value is None  # not set on error
    assert L.nm_stack_plan_run(None, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_stack_plan_destroy(None) == nm.NM_OK
    # the SwiGLU pair calls: rows_h must be a multiple of 16
    assert L.nm_spmv_swiglu(p16, p16, p16, p16, 8, 64, 1, None) == nm.NM_ERR_SHAPE
    assert L.nm_spmv_swiglu(p16, p16, p16, p16, 16, 48, 1, None) == nm.NM_ERR_SHAPE
    assert L.nm_spmv_swiglu(p16, p16, p16, p16, 16, 64, 9, None) == nm.NM_ERR_UNSUPPORTED
    assert L.nm_spmv_swiglu(None, p16, p16, p16, 16, 64, 1, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_spmv_swiglu(None, None, None, None, 0, 64, 1, None) == nm.NM_OK
    assert L.nm_pack_swiglu(p16, p16, 8, 64, 2, 4, p16, p16, None) == nm.NM_ERR_SHAPE
    assert L.nm_pack_swiglu(p16, p16, 16, 64, 3, 4, p16, p16, None) == nm.NM_ERR_UNSUPPORTED
    assert L.nm_pack_swiglu(p16, None, 16, 64, 2, 4, p16, p16, None) == nm.NM_ERR_INVALID_ARG
    # a stack op's flags: unknown bits, or SwiGLU on a row count that is not a multiple of 32
    ops[1].K = 64
    ops[0].flags = 4
    assert L.nm_spmv_stack(ops, 2, 1, None) == nm.NM_ERR_INVALID_ARG
    ops[0].flags = nm.NM_LINEAR_SWIGLU
    ops[0].rows = 16
    assert L.nm_spmv_stack(ops, 2, 1, None) == nm.NM_ERR_SHAPE
    ops[0].W = p16
    assert L.dense_gemv_stack(ops, 2, 1, None) == nm.NM_ERR_INVALID_ARG


def test_no_fallback_when_library_missing(monkeypatch):
    import sparse_decoding_gb300 as nm
    monkeypatch.setattr(nm, "_lib", None)
    monkeypatch.setattr(nm, "LIB_PATH", "/nonexistent/libnmspmv.so")
    with pytest.raises(RuntimeError, match="not built"):
        nm.lib()


def test_obs_argument_validation_before_any_cuda_call(nm):
    L = nm.lib()
    buf = (ctypes.c_uint8 * 4096)()
    p16 = (ctypes.addressof(buf) + 15) & ~15
    prune = L.nm_obs_prune
    # shape: K % 32, negative sizes
    assert prune(p16, p16, 4, 48, 2, 4, 0.01, 0, p16, None, None, None) == nm.NM_ERR_SHAPE
    assert prune(p16, p16, -1, 64, 2, 4, 0.01, 0, p16, None, None, None) == nm.NM_ERR_SHAPE
    # pattern: M must divide 32, 1 <= N <= M
    for N, M in ((2, 6), (0, 4), (5, 4), (2, 64)):
        assert prune(p16, p16, 4, 64, N, M, 0.01, 0, p16, None, None, None) == nm.NM_ERR_UNSUPPORTED
    # damping must be finite and >= 0; unknown flag
    for d in (-0.1, float("nan"), float("inf")):
        assert prune(p16, p16, 4, 64, 2, 4, d, 0, p16, None, None, None) == nm.NM_ERR_INVALID_ARG
    assert prune(p16, p16, 4, 64, 2, 4, 0.01, 2, p16, None, None, None) == nm.NM_ERR_INVALID_ARG
    # NULL and misaligned pointers
    assert prune(None, p16, 4, 64, 2, 4, 0.01, 0, p16, None, None, None) == nm.NM_ERR_INVALID_ARG
    assert prune(p16, p16, 4, 64, 2, 4, 0.01, 0, None, None, None, None) == nm.NM_ERR_INVALID_ARG
    assert prune(p16, p16 + 4, 4, 64, 2, 4, 0.01, 0, p16, None, None, None) == nm.NM_ERR_ALIGN
    assert prune(p16, p16, 4, 64, 2, 4, 0.01, 0, p16, p16 + 4, None, None) == nm.NM_ERR_ALIGN
    assert prune(p16, p16, 4, 64, 2, 4, 0.01, 0, p16, None, p16 + 8, None) == nm.NM_ERR_ALIGN
    # empty problems succeed without work
    assert prune(None, None, 0, 64, 2, 4, 0.01, 0, None, None, None, None) == nm.NM_OK
    assert prune(None, None, 4, 0, 2, 4, 0.01, 0, None, None, None, None) == nm.NM_OK
    hess = L.nm_obs_hessian
    assert hess(p16, 8, 48, p16, 0, None) == nm.NM_ERR_SHAPE
    assert hess(p16, -1, 64, p16, 0, None) == nm.NM_ERR_SHAPE
    assert hess(p16, 8, 64, None, 0, None) == nm.NM_ERR_INVALID_ARG
    assert hess(None, 8, 64, p16, 0, None) == nm.NM_ERR_INVALID_ARG
    assert hess(p16 + 2, 8, 64, p16, 0, None) == nm.NM_ERR_ALIGN
    assert hess(None, 0, 64, p16, 1, None) == nm.NM_OK  # nothing to add
    assert hess(None, 8, 0, None, 0, None) == nm.NM_OK


def test_atomic_splitk_argument_validation(nm):
    L = nm.lib()
    buf = (ctypes.c_uint8 * 4096)()
    p16 = (ctypes.addressof(buf) + 15) & ~15
    f = L.nm_spmv_f32out_atomic
    assert f(p16, p16, p16, p16, 4, 48, 1, None) == nm.NM_ERR_SHAPE
    assert f(p16, p16, p16, p16, 4, 64, 9, None) == nm.NM_ERR_UNSUPPORTED
    assert f(p16, p16, p16, p16 + 4, 4, 64, 1, None) == nm.NM_ERR_ALIGN
    assert f(None, p16, p16, p16, 4, 64, 1, None) == nm.NM_ERR_INVALID_ARG
    assert f(None, None, None, None, 0, 64, 1, None) == nm.NM_OK
