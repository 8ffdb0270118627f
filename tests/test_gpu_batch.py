"""GPU parity of the decode SpMV at batch 2..8 against the CPU oracle.

At batch 2, byte-regular words take the byte tables with both batch rows
shuffled as one bf16 pair; otherwise each warp walks its units with x from a
bf16 [column][batch] window in shared memory. The shapes cover: row blocks of
one CTA, partial row blocks (rows not a multiple of 32), row blocks whose K is
split over many CTAs (the fix-up across CTAs), every batch size, matrices
mixing 2:4 rows with 4:8, 8:16 and 16:32 rows, activations holding Inf and
NaN, exact sums, and repeatability. Tolerances are the SpMV's (fp32 within
1e-4 S elementwise, bf16 within one ulp of y64 and equal to rn(fp32)).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.bits import bits_to_f32, to_bits
from tests.test_gpu_parity import bf16_round_np, check_close, dev, nm, oracle_case, run_spmv  # noqa: F401

pytestmark = pytest.mark.gpu

# rows, K: one CTA's row blocks, partial row blocks, 128 x 14336 and
# 1000 x 28672 split few row blocks' K over many CTAs; 4097 x 4096 is
# stream-K with a one-row last row block
BATCH_SHAPES = [(1, 128), (33, 256), (128, 128), (129, 512), (200, 1024), (640, 4096), (4097, 4096),
             (128, 14336), (1000, 28672)]


@pytest.mark.parametrize("rows,K", BATCH_SHAPES)
@pytest.mark.parametrize("batch", [2, 4, 8])
def test_batch_24_shapes(nm, rows, K, batch):
    _, masks, values, x, y64, S = oracle_case(rows, K, 2, 4, batch, seed=rows + K + batch, select=False)
    y32, ybf = run_spmv(nm, masks, values, x)
    check_close(y32, ybf, y64, S, f"2:4 {rows}x{K} b{batch}")


@pytest.mark.parametrize("batch", [3, 5, 6, 7])
def test_batch_24_odd_batches(nm, batch):
    for rows, K in ((257, 1024), (4096, 4096)):
        _, masks, values, x, y64, S = oracle_case(rows, K, 2, 4, batch, seed=batch * 13 + rows, select=False)
        y32, ybf = run_spmv(nm, masks, values, x)
        check_close(y32, ybf, y64, S, f"2:4 {rows}x{K} b{batch}")


@pytest.mark.parametrize("batch", [2, 4, 8])
def test_batch_mixed_patterns(nm, batch):
    """Row groups of different patterns in one matrix at batch > 1, interleaved
    at several granularities, in the same CTAs and the same fix-ups."""
    K = 4096
    parts = []
    for i, (n, m_) in enumerate([(2, 4), (16, 32), (4, 8), (2, 4), (8, 16), (2, 4), (16, 32)]):
        rows = [64, 96, 32, 160, 1000, 33, 40][i]
        parts.append((n, m_, to_bits(synth.nm_structured(rows, K, n, m_, seed=50 + i))))
    Wp = np.concatenate([w for _, _, w in parts])
    masks = np.concatenate([oracle.pack(w, n, m_)[0] for n, m_, w in parts])
    values = np.concatenate([oracle.pack(w, n, m_)[1] for n, m_, w in parts])
    x = to_bits(synth.activations(batch, K, seed=51))
    y64, S = oracle.spmv_f64(Wp, x)
    y32, ybf = run_spmv(nm, masks, values, x)
    check_close(y32, ybf, y64, S, f"mixed units b{batch}")


@pytest.mark.parametrize("batch", [1, 2, 4, 8])
def test_nonfinite_x_reaches_only_rows_that_keep_its_column(nm, batch):
    """x holding +Inf, -Inf and NaN at a few columns. The format's sum has a
    term for kept values only, so such a column reaches just the rows that keep
    it (the dense product over the pruned W, which the oracle computes, would
    also multiply the pruned zeros: 0 * Inf = NaN). Rows that keep the column
    agree with the oracle's non-finite value; the other rows equal the oracle
    with those x entries set to 0."""
    rows, K = 1000, 4096
    Wp = to_bits(synth.nm_structured(rows, K, 2, 4, seed=61))
    masks, values = oracle.pack(Wp, 2, 4)
    x = to_bits(synth.activations(batch, K, seed=62))
    cols = [5, 700, 4095]
    specials = [0x7F80, 0xFF80, 0x7FC0]  # +Inf, -Inf, NaN
    bad_rows = list(range(batch))  # every batch row gets one special value
    for b in bad_rows:
        x[b, cols[b % 3]] = specials[b % 3]
    y64, _ = oracle.spmv_f64(Wp, x)
    xz = x.copy()
    for b in bad_rows:
        xz[b, cols[b % 3]] = 0
    yz, Sz = oracle.spmv_f64(Wp, xz)
    y32, ybf = run_spmv(nm, masks, values, x)
    for b in bad_rows:
        c = cols[b % 3]
        keeps = Wp[:, c] != 0  # nonzero kept weight at column c (2:4 packs no kept zeros here)
        assert keeps.any() and (~keeps).any()
        got = y32[b]
        np.testing.assert_array_equal(np.isnan(got[keeps]), np.isnan(y64[b][keeps]))
        np.testing.assert_array_equal(np.isposinf(got[keeps]), np.isposinf(y64[b][keeps]))
        np.testing.assert_array_equal(np.isneginf(got[keeps]), np.isneginf(y64[b][keeps]))
        assert np.all(np.isfinite(got[~keeps])), f"b{batch} row {b}: a non-finite x leaked into rows that prune it"
        check_close(got[None, ~keeps], ybf[b][None, ~keeps], yz[b][None, ~keeps], Sz[b][None, ~keeps],
                    f"finite rows b{batch}")


@pytest.mark.parametrize("batch", [2, 4, 8])
def test_batch_exact_dyadic(nm, batch):
    """Dyadic weights, small-integer x: every partial sum is exact in fp32, so
    the result equals the fp64 one exactly."""
    for rows, K in ((4096, 4096), (300, 14336)):
        Wp = to_bits(synth.nm_structured(rows, K, 2, 4, seed=7, dyadic=True))
        masks, values = oracle.pack(Wp, 2, 4)
        x = to_bits(synth.small_int_activations(batch, K, seed=7))
        y64, _ = oracle.spmv_f64(Wp, x)
        y32, ybf = run_spmv(nm, masks, values, x)
        np.testing.assert_array_equal(y32.astype(np.float64), y64)
        np.testing.assert_array_equal(ybf, bf16_round_np(y64.astype(np.float32)))


@pytest.mark.parametrize("batch", [2, 8])
def test_batch_repeatable(nm, batch):
    """Each warp's order of products is fixed and the fix-up adds parts in
    warp and CTA order: repeated calls give identical bits."""
    _, masks, values, x, _, _ = oracle_case(4096, 14336, 2, 4, batch, seed=9, select=False)
    m = torch.from_numpy(masks.view(np.int32)).cuda()
    v, xd = dev(values), dev(x)
    ys = [nm.spmv(m, v, xd, f32=True) for _ in range(3)]
    for y in ys[1:]:
        assert torch.equal(y, ys[0])
    yb = [to_bits(nm.spmv(m, v, xd)) for _ in range(2)]
    np.testing.assert_array_equal(yb[0], yb[1])
    np.testing.assert_array_equal(yb[0], bf16_round_np(ys[0].cpu().numpy()))


def test_batch_zero_x_and_ones(nm):
    """Closed forms at batch > 1: x = 0 gives 0; 2:4 rows of ones times x = 1
    give K / 2."""
    rows, K = 300, 2048
    keep = synth.random_nm_keep(rows, K, 2, 4, seed=8).numpy()
    Wp = np.where(keep, np.uint16(0x3F80), np.uint16(0))
    masks, values = oracle.pack(Wp, 2, 4)
    y32, _ = run_spmv(nm, masks, values, np.full((4, K), 0x3F80, dtype=np.uint16))
    assert np.all(y32 == K / 2)
    y32, ybf = run_spmv(nm, masks, values, np.zeros((8, K), dtype=np.uint16))
    assert np.all(y32 == 0) and np.all(bits_to_f32(ybf) == 0)
