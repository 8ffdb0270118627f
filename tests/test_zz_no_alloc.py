"""nm_spmv_noalloc: the SpMV for callers that may not allocate device memory.

Such a caller (for example code running inside another framework's memory
pool) cannot let the library cudaMalloc its scratch on first use, so this entry
point keeps that scratch in a fixed device array instead. The tests check,
through the C ABI, that it gives nm_spmv's result bit for bit (same kernel,
same summation order) and the oracle's within the decode tolerance, call after
call; and, in a fresh process where nothing else of the library has run, that
its first call leaves the library's own scratch unallocated. The file is named
to run last, so that a run stopping at the first failure has run everything
else first; it also passes alone in a fresh process.
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.bits import bf16_ulp, bits_to_f32, from_bits, to_bits

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TOL = 1e-4


@pytest.fixture(scope="module")
def nm():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sparse_decoding_gb300 import build
    build.build()
    import sparse_decoding_gb300 as nm
    return nm


def _call(fn, m, v, x, y, rows, K, batch):
    return fn(m.data_ptr(), v.data_ptr(), x.data_ptr(), y.data_ptr(), rows, K, batch,
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _check_oracle(y_bits, y64, S, what):
    """bf16 within one ulp of the fp64 oracle (plus 1e-4*S where |y64| < 1e-4*S)."""
    yb = bits_to_f32(y_bits).astype(np.float64)
    bound = bf16_ulp(y64) + np.where(np.abs(y64) >= TOL * S, 0.0, TOL * S)
    bad = ~(np.abs(yb - y64) <= bound)
    assert not bad.any(), f"{what}: off the oracle at {np.argwhere(bad)[:5]}"


# Shapes covering whole-row-block CTAs, row blocks split between CTAs
# (the scratch in use), K = 128 and the fallback kernel (K % 128 != 0).
@pytest.mark.parametrize("rows,K,batch", [(4096, 4096, 1), (6144, 4096, 1), (4096, 14336, 3),
                                          (10000, 128, 2), (333, 96, 1), (28672, 4096, 1)])
def test_noalloc_matches_nm_spmv_and_oracle_twice(nm, rows, K, batch):
    Wp = to_bits(synth.nm_structured(rows, K, 2, 4, seed=rows + K))
    masks, values = oracle.pack(Wp, 2, 4)
    xb = to_bits(synth.activations(batch, K, seed=7))
    y64, S = oracle.spmv_f64(Wp, xb)
    m = torch.from_numpy(masks.view(np.int32)).cuda()
    v = from_bits(values).cuda()
    x = from_bits(xb).cuda()
    L = nm.lib()
    y_ref = torch.empty(batch, rows, dtype=torch.bfloat16, device="cuda")
    assert _call(L.nm_spmv, m, v, x, y_ref, rows, K, batch) == nm.NM_OK
    for call in range(2):  # the second call finds the array as the first left it
        y = torch.full((batch, rows), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call(L.nm_spmv_noalloc, m, v, x, y, rows, K, batch) == nm.NM_OK
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref), f"call {call}: nm_spmv_noalloc differs from nm_spmv"
        _check_oracle(to_bits(y.cpu()), y64, S, f"call {call}")
    assert nm.device_status() == nm.NM_OK


def test_noalloc_rejects_bad_arguments(nm):
    L = nm.lib()
    buf = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.nm_spmv_noalloc(p, p, p, p, 4, 48, 1, s) == nm.NM_ERR_SHAPE
    assert L.nm_spmv_noalloc(p, p, p, p, 4, 64, 9, s) == nm.NM_ERR_UNSUPPORTED
    assert L.nm_spmv_noalloc(p + 2, p, p, p, 4, 64, 1, s) == nm.NM_ERR_ALIGN
    assert L.nm_spmv_noalloc(None, p, p, p, 4, 64, 1, s) == nm.NM_ERR_INVALID_ARG


# Run in a fresh process: only nm_spmv_noalloc has been called when the device's
# free memory is read, so if that call had allocated the library scratch (about
# 2 MB), the first allocating call made afterwards (nm_spmv) would find it there
# and allocate nothing. It must instead take at least the scratch's bytes.
_FRESH = textwrap.dedent("""
    import ctypes, sys
    sys.path.insert(0, {root!r})
    import numpy as np, torch
    import oracle, synth
    from tests.bits import from_bits, to_bits
    import sparse_decoding_gb300 as nm
    torch.cuda.set_device(0)
    rows, K = 4096, 14336
    Wp = to_bits(synth.nm_structured(rows, K, 2, 4, seed=11))
    masks, values = oracle.pack(Wp, 2, 4)
    m = torch.from_numpy(masks.view(np.int32)).cuda()
    v = from_bits(values).cuda()
    x = synth.activations(1, K, seed=12).cuda()
    y1 = torch.empty(1, rows, dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty(1, rows, dtype=torch.bfloat16, device="cuda")
    y3 = torch.empty(1, rows, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    L = nm.lib()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = lambda y: (m.data_ptr(), v.data_ptr(), x.data_ptr(), y.data_ptr(), rows, K, 1, s)
    assert L.nm_spmv_noalloc(*args(y1)) == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    assert L.nm_spmv_noalloc(*args(y2)) == 0      # later calls allocate nothing either
    assert L.nm_device_status(s) == 0             # and the status query, after noalloc only
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert L.nm_spmv(*args(y3)) == 0              # the library scratch is allocated now
    torch.cuda.synchronize()
    free2 = torch.cuda.mem_get_info()[0]
    assert torch.equal(y1, y3) and torch.equal(y2, y3)
    print("FREE", free0, free1, free2)
""")


def test_noalloc_first_call_allocates_nothing_in_a_fresh_process(nm):
    r = subprocess.run([sys.executable, "-c", _FRESH.format(root=ROOT)], capture_output=True, text=True,
                       cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("FREE")][-1]
    free0, free1, free2 = map(int, line.split()[1:])
    assert free1 == free0, "a later nm_spmv_noalloc call (or the status query) changed free device memory"
    scratch_bytes = 256 + 4 * 1024 + 4 * 1024 * 2 * 8 * 32  # status, counters, partial sums
    assert free1 - free2 >= scratch_bytes, (
        f"nm_spmv took {free1 - free2} bytes: the library scratch already existed, "
        "so nm_spmv_noalloc must have allocated it")
