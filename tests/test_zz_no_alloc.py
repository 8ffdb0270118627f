"""nm_spmv_noalloc: the SpMV for callers that may not allocate device memory.

Such a caller (for example code running inside another framework's memory
pool) cannot let the library cudaMalloc its scratch on first use, so this entry
point keeps that scratch in a fixed device array instead. It must give the
same result as nm_spmv, call after call, through the C ABI. The file is named
to run last, so that a run stopping at the first failure has run everything
else first; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.bits import bf16_ulp, bits_to_f32, from_bits, to_bits

pytestmark = pytest.mark.gpu


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


# Shapes covering whole-row-block CTAs, row blocks split between CTAs
# (the scratch in use), K = 128 and the fallback kernel (K % 128 != 0).
@pytest.mark.parametrize("rows,K,batch", [(4096, 4096, 1), (6144, 4096, 1), (4096, 14336, 3),
                                          (10000, 128, 2), (333, 96, 1), (28672, 4096, 1)])
def test_noalloc_matches_nm_spmv_twice(nm, rows, K, batch):
    Wp = to_bits(synth.nm_structured(rows, K, 2, 4, seed=rows + K))
    masks, values = oracle.pack(Wp, 2, 4)
    m = torch.from_numpy(masks.view(np.int32)).cuda()
    v = from_bits(values).cuda()
    x = synth.activations(batch, K, seed=7).cuda()
    L = nm.lib()
    y_ref = torch.empty(batch, rows, dtype=torch.bfloat16, device="cuda")
    assert _call(L.nm_spmv, m, v, x, y_ref, rows, K, batch) == nm.NM_OK
    ref = bits_to_f32(to_bits(y_ref)).astype(np.float64)
    for _ in range(2):  # the second call finds the array as the first left it
        y = torch.full((batch, rows), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call(L.nm_spmv_noalloc, m, v, x, y, rows, K, batch) == nm.NM_OK
        torch.cuda.synchronize()
        got = bits_to_f32(to_bits(y)).astype(np.float64)
        assert np.all(np.abs(got - ref) <= bf16_ulp(ref)), "nm_spmv_noalloc differs from nm_spmv"
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
