"""GPU parity of the split-K variant that combines row-block parts with
atomicAdd (nm_spmv_f32out_atomic) against the CPU oracle.

The variant splits the K range of every row block over all CTA slots, so
almost every row is the sum of several CTAs' parts. Its result obeys the fp32
bound of the default path, |y32 - y64| <= 1e-4 * S; with dyadic weights and
small-integer activations every partial sum is exact, so the result must equal
the oracle exactly whatever order the additions take -- which also shows that
each part is added exactly once.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.bits import to_bits
from tests.test_gpu_parity import check_close, dev, oracle_case, sampled_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nm():
    from sparse_decoding_gb300 import build
    build.build()
    import sparse_decoding_gb300 as nm
    nm.init()
    return nm


def run_atomic(nm, masks, values, x, fill=None):
    m = torch.from_numpy(masks.view(np.int32)).cuda()
    v, xd = dev(values), dev(x)
    out = torch.empty(x.shape[0], masks.shape[0], dtype=torch.float32, device="cuda")
    if fill is not None:
        out.fill_(fill)
    nm.spmv(m, v, xd, out=out, f32=True, atomic=True)
    torch.cuda.synchronize()
    return out.cpu().numpy()


SHAPES = [(1, 128), (31, 256), (100, 512), (64, 4096), (257, 1024), (1, 4096), (33, 8192), (96, 28672),
          (4900, 4096), (6144, 4096), (20000, 384), (33, 96), (5, 3968)]


@pytest.mark.parametrize("rows,K", SHAPES)
def test_atomic_matches_oracle(nm, rows, K):
    for batch in (1, 2, 8):
        _, masks, values, x, y64, S = oracle_case(rows, K, 8, 16, batch, seed=rows * 3 + K, select=False)
        y32 = run_atomic(nm, masks, values, x, fill=float("nan"))
        check_close(y32, None, y64, S, f"atomic {rows}x{K} b{batch}")


@pytest.mark.parametrize("N,M", synth.PATTERNS)
def test_atomic_exact_dyadic(nm, N, M):
    for rows, K, batch in ((4096, 4096, 1), (100, 14336, 8), (64, 28672, 3)):
        Wp = to_bits(synth.nm_structured(rows, K, N, M, seed=15, dyadic=True))
        masks, values = oracle.pack(Wp, N, M)
        x = to_bits(synth.small_int_activations(batch, K, seed=15))
        y64, _ = oracle.spmv_f64(Wp, x)
        y32 = run_atomic(nm, masks, values, x, fill=123.0)
        np.testing.assert_array_equal(y32.astype(np.float64), y64)


@pytest.mark.parametrize("name,batch", [("o", 8), ("down", 8), ("down", 1), ("qkv", 4)])
def test_atomic_llama8b_sampled(nm, name, batch):
    rows, K = synth.LLAMA31_8B[name]
    W = synth.nm_structured(rows, K, 2, 4, seed=17, device="cuda")
    m, v = nm.pack(W, 2, 4)
    x = synth.activations(batch, K, seed=18, device="cuda")
    y = nm.spmv(m, v, x, f32=True, atomic=True)
    torch.cuda.synchronize()
    idx = sampled_rows(rows, 17)
    y64, S = oracle.spmv_f64(to_bits(W[torch.from_numpy(idx).cuda()].cpu()), to_bits(x.cpu()))
    check_close(y.cpu().numpy()[:, idx], None, y64, S, f"atomic 8b {name} b{batch}")


def test_atomic_needs_fp32_and_handles_empty(nm):
    m = torch.zeros(4, 2, dtype=torch.int32, device="cuda")
    v = torch.zeros(4, 32, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(1, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        nm.spmv(m, v, x, atomic=True)
    m0 = torch.zeros(5, 0, dtype=torch.int32, device="cuda")
    v0 = torch.zeros(5, 0, dtype=torch.bfloat16, device="cuda")
    x0 = torch.zeros(2, 0, dtype=torch.bfloat16, device="cuda")
    y0 = torch.full((2, 5), 7.0, dtype=torch.float32, device="cuda")
    nm.spmv(m0, v0, x0, out=y0, f32=True, atomic=True)
    assert torch.equal(y0, torch.zeros_like(y0))
    assert nm.device_status() == nm.NM_OK
