"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Tolerances (the fp32 and bf16 bounds of the decode SpMV):
  * masks, values, selection: bit-exact;
  * fp32 output: |y32 - y64| <= 1e-4 * S elementwise, S = sum_j |W_rj x_bj|;
  * bf16 output: within one bf16 ulp of y64, and equal to bf16_rn(y32) of the
    same kernel (where |y64| < 1e-4 * S only the fp32 bound applies);
  * integer-valued cases (dyadic W, small-integer x): exact.
Inputs for the CUDA path come from synth (seeded) or from the oracle; no
oracle input comes from the CUDA path.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.bits import bf16_ulp, bits_to_f32, from_bits, to_bits

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module")
def nm():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sparse_decoding_gb300 import build
    build.build()
    import sparse_decoding_gb300 as nm
    nm.init()
    return nm


def dev(bits: np.ndarray) -> torch.Tensor:
    return from_bits(bits).cuda()


def masks_np(m: torch.Tensor) -> np.ndarray:
    return m.cpu().numpy().view(np.uint32)


def bf16_round_np(y32: np.ndarray) -> np.ndarray:
    return to_bits(torch.from_numpy(np.ascontiguousarray(y32, dtype=np.float32)).to(torch.bfloat16))


def check_close(y32: np.ndarray, ybf: np.ndarray, y64: np.ndarray, S: np.ndarray, what: str):
    err = np.abs(y32.astype(np.float64) - y64)
    bad = err > TOL * S
    assert not bad.any(), f"{what}: fp32 error {err[bad][:5]} > 1e-4*S {TOL * S[bad][:5]}"
    if ybf is not None:
        np.testing.assert_array_equal(ybf, bf16_round_np(y32), err_msg=f"{what}: bf16 != rn(fp32)")
        yb = bits_to_f32(ybf).astype(np.float64)
        strict = np.abs(y64) >= TOL * S
        ulp_err = np.abs(yb - y64)
        bad = strict & (ulp_err > bf16_ulp(y64))
        assert not bad.any(), f"{what}: bf16 more than 1 ulp off at {np.argwhere(bad)[:5]}"


def oracle_case(rows, K, N, M, batch, seed, select=True):
    """Oracle-side inputs: pruned W (bits), masks, values, x (bits), y64, S."""
    if select:
        W = to_bits(synth.weights(rows, K, seed=seed))
        a = synth.col_norms(K, seed=seed).numpy()
        Wp = oracle.select(W, a, N, M)
    else:
        Wp = to_bits(synth.nm_structured(rows, K, N, M, seed=seed))
    masks, values = oracle.pack(Wp, N, M)
    x = to_bits(synth.activations(batch, K, seed=seed + 1))
    y64, S = oracle.spmv_f64(Wp, x)
    return Wp, masks, values, x, y64, S


def run_spmv(nm, masks, values, x):
    m = torch.from_numpy(masks.view(np.int32)).cuda()
    v, xd = dev(values), dev(x)
    y32 = nm.spmv(m, v, xd, f32=True)
    ybf = nm.spmv(m, v, xd)
    torch.cuda.synchronize()
    return y32.cpu().numpy(), to_bits(ybf)


# --- SpMV -------------------------------------------------------------------------

SMALL_SHAPES = [(1, 128), (31, 128), (33, 256), (100, 512), (64, 4096), (257, 1024),  # TMA path
                (1, 32), (31, 64), (33, 96), (70, 160), (5, 4000 // 32 * 32)]          # fallback path


@pytest.mark.parametrize("rows,K", SMALL_SHAPES)
@pytest.mark.parametrize("N,M", synth.PATTERNS)
def test_spmv_small_shapes(nm, rows, K, N, M):
    for batch in (1, 3):
        _, masks, values, x, y64, S = oracle_case(rows, K, N, M, batch, seed=rows * 7 + K)
        y32, ybf = run_spmv(nm, masks, values, x)
        check_close(y32, ybf, y64, S, f"{rows}x{K} {N}:{M} b{batch}")


# More row blocks than SMs, so CTAs share row blocks (stream-K fix-up across
# CTAs), with 1, 3, 9 and 32 units per row block.
STREAM_K_SHAPES = [(5000, 128), (10000, 128), (20000, 384), (4900, 4096), (9999, 1152), (6144, 4096),
                   # few row blocks, long K: row blocks shared by many CTAs
                   (64, 14336), (96, 28672), (33, 8192), (250, 4096), (1, 4096)]


@pytest.mark.parametrize("rows,K", STREAM_K_SHAPES)
def test_spmv_stream_k_shapes(nm, rows, K):
    for batch in (1, 2, 5):
        _, masks, values, x, y64, S = oracle_case(rows, K, 8, 16, batch, seed=rows + K, select=False)
        y32, ybf = run_spmv(nm, masks, values, x)
        check_close(y32, ybf, y64, S, f"{rows}x{K} b{batch}")


def test_spmv_mixed_patterns_in_one_matrix(nm):
    """Row groups packed with different patterns: byte-regular words (2:4, 4:8)
    and irregular ones (8:16, 16:32) in one matrix, interleaved at several
    granularities, so warps meet both kinds of unit."""
    K = 4096
    parts = []
    for i, (n, m_) in enumerate([(2, 4), (16, 32), (4, 8), (8, 16), (2, 4), (16, 32)]):
        rows = [64, 96, 32, 160, 1000, 33][i]
        parts.append((n, m_, to_bits(synth.nm_structured(rows, K, n, m_, seed=40 + i))))
    Wp = np.concatenate([w for _, _, w in parts])
    masks = np.concatenate([oracle.pack(w, n, m_)[0] for n, m_, w in parts])
    values = np.concatenate([oracle.pack(w, n, m_)[1] for n, m_, w in parts])
    x = to_bits(synth.activations(1, K, seed=41))
    y64, S = oracle.spmv_f64(Wp, x)
    y32, ybf = run_spmv(nm, masks, values, x)
    check_close(y32, ybf, y64, S, "mixed patterns")


@pytest.mark.parametrize("rows,K", STREAM_K_SHAPES)
def test_dense_stream_k_shapes(nm, rows, K):
    Wp = to_bits(synth.nm_structured(rows, K, 2, 4, seed=rows))
    x = to_bits(synth.activations(3, K, seed=rows))
    y64, S = oracle.spmv_f64(Wp, x)
    y32 = nm.dense_gemv(dev(Wp), dev(x), f32=True).cpu().numpy()
    check_close(y32, None, y64, S, f"dense {rows}x{K}")


@pytest.mark.parametrize("batch", range(1, 9))
def test_spmv_every_batch(nm, batch):
    for rows, K in ((96, 1024), (45, 96)):
        _, masks, values, x, y64, S = oracle_case(rows, K, 16, 32, batch, seed=batch)
        y32, ybf = run_spmv(nm, masks, values, x)
        check_close(y32, ybf, y64, S, f"{rows}x{K} b{batch}")


@pytest.mark.parametrize("N,M", synth.PATTERNS)
def test_spmv_single_4096(nm, N, M):
    """4096 x 4096, batch 1, seed 0: the single-linear workload."""
    _, masks, values, x, y64, S = oracle_case(4096, 4096, N, M, 1, seed=0)
    y32, ybf = run_spmv(nm, masks, values, x)
    check_close(y32, ybf, y64, S, f"4096x4096 {N}:{M}")


@pytest.mark.parametrize("name", ["qkv", "o", "gate_up", "down"])
@pytest.mark.parametrize("N,M", [(2, 4), (16, 32)])
def test_spmv_llama8b_linears(nm, name, N, M):
    rows, K = synth.LLAMA31_8B[name]
    _, masks, values, x, y64, S = oracle_case(rows, K, N, M, 1, seed=11, select=False)
    y32, ybf = run_spmv(nm, masks, values, x)
    check_close(y32, ybf, y64, S, f"{name} {N}:{M}")


# The other model shapes at full size (Qwen3-14B/32B with 4:8 and 8:16;
# Llama-3.3-70B with 2:4 and 16:32): W is drawn on the GPU by the seeded
# generator, packed and multiplied there; the oracle recomputes a sample of
# rows (the first and last row block and 32 scattered rows) from the same
# generator's rows copied back.
MODEL_CASES = [("qwen3-14b", (4, 8)), ("qwen3-14b", (8, 16)), ("qwen3-32b", (4, 8)), ("qwen3-32b", (8, 16)),
               ("llama3.3-70b", (2, 4)), ("llama3.3-70b", (16, 32))]


def sampled_rows(rows: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    idx = np.concatenate([np.arange(min(32, rows)), np.arange(max(0, rows - 32), rows),
                          rng.integers(0, rows, 32)])
    return np.unique(idx)


def check_sampled(nm, rows, K, N, M, batch, seed, what):
    W = synth.nm_structured(rows, K, N, M, seed=seed, device="cuda")
    m, v = nm.pack(W, N, M)
    x = synth.activations(batch, K, seed=seed + 1, device="cuda")
    y32 = nm.spmv(m, v, x, f32=True)
    ybf = nm.spmv(m, v, x)
    torch.cuda.synchronize()
    idx = sampled_rows(rows, seed)
    Wp = to_bits(W[torch.from_numpy(idx).cuda()].cpu())
    y64, S = oracle.spmv_f64(Wp, to_bits(x.cpu()))
    check_close(y32.cpu().numpy()[:, idx], to_bits(ybf)[:, idx], y64, S, what)
    del W, m, v


@pytest.mark.parametrize("model,pattern", MODEL_CASES)
@pytest.mark.parametrize("name", ["qkv", "o", "gate_up", "down"])
def test_spmv_model_linears_sampled(nm, model, pattern, name):
    rows, K = synth.MODELS[model][name]
    N, M = pattern
    check_sampled(nm, rows, K, N, M, 1, seed=rows % 1000 + K % 997, what=f"{model} {name} {N}:{M}")


@pytest.mark.parametrize("batch", [2, 4, 8])
@pytest.mark.parametrize("name", ["o", "down"])
def test_spmv_70b_batch_sweep_sampled(nm, batch, name):
    rows, K = synth.LLAMA33_70B[name]
    check_sampled(nm, rows, K, 2, 4, batch, seed=31 + batch, what=f"70b {name} b{batch}")


# The 8B stack's two largest linears at full size at the batch sizes of the
# batch-4 and batch-8 timings (the batch > 1 kernel: bf16 x window, per-warp
# ranges, fix-ups between warps and CTAs), all four patterns.
@pytest.mark.parametrize("batch", [4, 8])
@pytest.mark.parametrize("name", ["gate_up", "down"])
@pytest.mark.parametrize("N,M", synth.PATTERNS)
def test_spmv_llama8b_batch_sampled(nm, batch, name, N, M):
    rows, K = synth.LLAMA31_8B[name]
    check_sampled(nm, rows, K, N, M, batch, seed=61 + batch + N, what=f"8b {name} {N}:{M} b{batch}")


@pytest.mark.parametrize("N,M", synth.PATTERNS)
def test_spmv_exact_dyadic(nm, N, M):
    """Dyadic weights, small-integer x: fp32 is exact in any summation order."""
    for rows, K, batch in ((4096, 4096, 1), (100, 14336, 4), (33, 96, 2)):
        Wp = to_bits(synth.nm_structured(rows, K, N, M, seed=5, dyadic=True))
        masks, values = oracle.pack(Wp, N, M)
        x = to_bits(synth.small_int_activations(batch, K, seed=5))
        y64, _ = oracle.spmv_f64(Wp, x)
        y32, ybf = run_spmv(nm, masks, values, x)
        np.testing.assert_array_equal(y32.astype(np.float64), y64)
        np.testing.assert_array_equal(ybf, bf16_round_np(y64.astype(np.float32)))


def test_spmv_one_hot_columns(nm):
    rows, K = 77, 512
    Wp = to_bits(synth.nm_structured(rows, K, 4, 8, seed=6))
    masks, values = oracle.pack(Wp, 4, 8)
    cols = [0, 1, 31, 32, 127, 128, 300, 511]
    x = np.zeros((len(cols), K), dtype=np.uint16)
    for b, j in enumerate(cols):
        x[b, j] = 0x3F80
    y32, ybf = run_spmv(nm, masks, values, x)
    for b, j in enumerate(cols):
        np.testing.assert_array_equal(y32[b], bits_to_f32(Wp[:, j]))
        np.testing.assert_array_equal(ybf[b], Wp[:, j])


def test_spmv_closed_forms(nm):
    rows, K = 40, 1024
    keep = synth.random_nm_keep(rows, K, 8, 16, seed=7).numpy()
    Wp = np.where(keep, np.uint16(0x3F80), np.uint16(0))
    masks, values = oracle.pack(Wp, 8, 16)
    ones = np.full((2, K), 0x3F80, dtype=np.uint16)
    y32, _ = run_spmv(nm, masks, values, ones)
    assert np.all(y32 == K / 2)
    y32, ybf = run_spmv(nm, masks, values, np.zeros((1, K), dtype=np.uint16))
    assert np.all(y32 == 0) and np.all(ybf == 0)


def test_spmv_nan_stays_in_its_row(nm):
    rows, K = 64, 256
    Wp = to_bits(synth.nm_structured(rows, K, 2, 4, seed=8))
    c = int(np.nonzero(Wp[5])[0][3])
    Wp[5, c] = 0x7FC0
    masks, values = oracle.pack(Wp, 2, 4)
    x = to_bits(synth.activations(1, K, seed=8))
    y64, S = oracle.spmv_f64(Wp, x)
    y32, ybf = run_spmv(nm, masks, values, x)
    assert np.isnan(y32[0, 5]) and np.isnan(bits_to_f32(ybf[0, 5]))
    ok = np.arange(rows) != 5
    check_close(y32[:, ok], ybf[:, ok], y64[:, ok], S[:, ok], "nan rows")


def test_spmv_repeatable(nm):
    """Fixed summation order: repeated calls give identical bits."""
    _, masks, values, x, _, _ = oracle_case(6144, 4096, 2, 4, 1, seed=9, select=False)
    m = torch.from_numpy(masks.view(np.int32)).cuda()
    v, xd = dev(values), dev(x)
    ys = [nm.spmv(m, v, xd, f32=True) for _ in range(3)]
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


@pytest.mark.parametrize("batch", [1, 4])
@pytest.mark.parametrize("N,M", [(2, 4), (16, 32)])
def test_spmv_row_and_k_shards(nm, batch, N, M):
    """The path shards by rows (x replicated) or by K (partial sums added):
    concatenated row shards, and the fp32 sum of K shards, meet the same bound
    against the fp64 oracle as the unsharded product. (A row's summation order
    follows how its row block is split over CTAs, which depends on the shard's
    shape, so the shards are not required to repeat the unsharded bits.)"""
    rows, K = 4096, 4096
    _, masks, values, x, y64, S = oracle_case(rows, K, N, M, batch, seed=21, select=False)
    m = torch.from_numpy(masks.view(np.int32)).cuda()
    v, xd = dev(values), dev(x)
    full = nm.spmv(m, v, xd, f32=True).cpu().numpy()
    check_close(full, None, y64, S, "unsharded")
    for cuts in ([0, 2048, 4096], [0, 1024, 3072, 4096], [0, 32, 4096]):
        parts = [nm.spmv(m[a:b].contiguous(), v[a:b].contiguous(), xd, f32=True) for a, b in zip(cuts, cuts[1:])]
        y = torch.cat(parts, dim=1).cpu().numpy()
        check_close(y, None, y64, S, f"row shards {cuts}")
        # two fp32 results of the same rows, each within 1e-4 S of y64
        assert np.all(np.abs(y.astype(np.float64) - full) <= 2 * TOL * S)
    for cut in (2048, 1024, 128):
        ya = nm.spmv(m[:, :cut // 32].contiguous(), v[:, :cut // 2].contiguous(), xd[:, :cut].contiguous(), f32=True)
        yb = nm.spmv(m[:, cut // 32:].contiguous(), v[:, cut // 2:].contiguous(), xd[:, cut:].contiguous(), f32=True)
        check_close((ya + yb).cpu().numpy(), None, y64, S, f"K shards at {cut}")


def test_spmv_empty_and_k0(nm):
    m = torch.zeros(0, 4, dtype=torch.int32, device="cuda")
    v = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(1, 128, dtype=torch.bfloat16, device="cuda")
    y = nm.spmv(m, v, x)
    assert y.shape == (1, 0)
    # K == 0: every output is the empty sum, +0
    m0 = torch.zeros(5, 0, dtype=torch.int32, device="cuda")
    v0 = torch.zeros(5, 0, dtype=torch.bfloat16, device="cuda")
    x0 = torch.zeros(2, 0, dtype=torch.bfloat16, device="cuda")
    y0 = torch.full((2, 5), 7.0, dtype=torch.bfloat16, device="cuda")
    nm.spmv(m0, v0, x0, out=y0)
    assert torch.equal(y0, torch.zeros_like(y0))


# --- pack and select ---------------------------------------------------------------

PACK_SHAPES = [(1, 32), (31, 64), (33, 96), (257, 1024), (4096, 4096), (128, 14336)]


@pytest.mark.parametrize("rows,K", PACK_SHAPES)
@pytest.mark.parametrize("N,M", synth.PATTERNS)
def test_select_and_pack_bit_exact(nm, rows, K, N, M):
    W = synth.weights(rows, K, seed=rows + K)
    a = synth.col_norms(K, seed=rows + K)
    Wp = oracle.select(to_bits(W), a.numpy(), N, M)
    om, ov = oracle.pack(Wp, N, M)
    Wg = nm.select(W.cuda(), a.cuda(), N, M)
    np.testing.assert_array_equal(to_bits(Wg), Wp)
    gm, gv = nm.pack(Wg, N, M)
    np.testing.assert_array_equal(masks_np(gm), om)
    np.testing.assert_array_equal(to_bits(gv), ov)
    # in-place selection gives the same result
    Wi = W.cuda()
    nm.select(Wi, a.cuda(), N, M, out=Wi)
    np.testing.assert_array_equal(to_bits(Wi), Wp)


def test_select_ties_and_special_values(nm):
    rows, K = 64, 256
    rng = np.random.default_rng(3)
    W = np.array([0x3F80, 0xBF80, 0x4000, 0x0000, 0x8000], dtype=np.uint16)[rng.integers(0, 5, (rows, K))]
    a = np.ones(K, dtype=np.float32)
    a[::7] = 0.0
    for N, M in synth.PATTERNS:
        Wp = oracle.select(W, a, N, M)
        got = nm.select(dev(W), torch.from_numpy(a).cuda(), N, M)
        np.testing.assert_array_equal(to_bits(got), Wp)
        om, ov = oracle.pack(Wp, N, M)
        gm, gv = nm.pack(dev(Wp), N, M)
        np.testing.assert_array_equal(masks_np(gm), om)
        np.testing.assert_array_equal(to_bits(gv), ov)


# --- selection and pack fused in one pass (nm_select_pack) ----------------------------

@pytest.mark.parametrize("rows,K", PACK_SHAPES)
@pytest.mark.parametrize("N,M", synth.PATTERNS)
def test_select_pack_bit_exact(nm, rows, K, N, M):
    W = synth.weights(rows, K, seed=rows + K)
    a = synth.col_norms(K, seed=rows + K)
    om, ov = oracle.pack(oracle.select(to_bits(W), a.numpy(), N, M), N, M)
    gm, gv = nm.select_pack(W.cuda(), a.cuda(), N, M)
    np.testing.assert_array_equal(masks_np(gm), om)
    np.testing.assert_array_equal(to_bits(gv), ov)


def test_select_pack_ties_zeros_and_nan_scores(nm):
    # weights +-1, 2, +0, -0 (ties, kept zeros with their sign), a column norm
    # of 0 (a nonzero weight whose score ties the zeros), NaN weights and a NaN
    # norm (NaN scores rank above every number)
    rows, K = 96, 512
    rng = np.random.default_rng(4)
    W = np.array([0x3F80, 0xBF80, 0x4000, 0x0000, 0x8000], dtype=np.uint16)[rng.integers(0, 5, (rows, K))]
    W[rng.integers(0, rows, 40), rng.integers(0, K, 40)] = 0x7FC0
    a = np.ones(K, dtype=np.float32)
    a[::7] = 0.0
    a[5] = np.nan
    for N, M in synth.PATTERNS:
        om, ov = oracle.pack(oracle.select(W, a, N, M), N, M)
        gm, gv = nm.select_pack(dev(W), torch.from_numpy(a).cuda(), N, M)
        np.testing.assert_array_equal(masks_np(gm), om, err_msg=f"{N}:{M} masks")
        np.testing.assert_array_equal(to_bits(gv), ov, err_msg=f"{N}:{M} values")


@pytest.mark.parametrize("N,M", [(2, 4), (16, 32)])
def test_select_pack_llama_gate_up_sampled(nm, N, M):
    # full-size 28672 x 4096 on the GPU; rows sampled for the oracle
    rows, K = synth.LLAMA31_8B["gate_up"]
    W = synth.weights(rows, K, 0, 77, device="cuda")
    a = synth.col_norms(K, 0, 78, device="cuda")
    gm, gv = nm.select_pack(W, a, N, M)
    idx = torch.from_numpy(np.random.default_rng(5).choice(rows, 64, replace=False)).cuda()
    om, ov = oracle.pack(oracle.select(to_bits(W[idx].cpu()), a.cpu().numpy(), N, M), N, M)
    np.testing.assert_array_equal(masks_np(gm[idx]), om)
    np.testing.assert_array_equal(to_bits(gv[idx].cpu()), ov)


def test_select_pack_rejects_bad_arguments(nm):
    W = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    a = torch.ones(64, dtype=torch.float32, device="cuda")
    with pytest.raises(nm.NmError) as e:
        nm.select_pack(W, a, 1, 4)
    assert e.value.status == nm.NM_ERR_UNSUPPORTED
    with pytest.raises(nm.NmError) as e:
        nm.select_pack(torch.zeros(4, 48, dtype=torch.bfloat16, device="cuda"), a[:48].contiguous(), 2, 4)
    assert e.value.status == nm.NM_ERR_SHAPE


def test_pack_fill_rule_and_signed_zero(nm):
    Wp = np.zeros((3, 64), dtype=np.uint16)
    Wp[0, 2] = 0x4000
    Wp[0, 0] = 0x8000
    Wp[1, 40] = 0x7FC0       # NaN counts as nonzero and is kept bit for bit
    Wp[2, :] = 0x0000        # all zero: the first N of every subgroup
    for N, M in synth.PATTERNS:
        om, ov = oracle.pack(Wp, N, M)
        gm, gv = nm.pack(dev(Wp), N, M)
        np.testing.assert_array_equal(masks_np(gm), om)
        np.testing.assert_array_equal(to_bits(gv), ov)


def test_pack_reports_not_nm(nm):
    Wp = np.full((4, 64), 0x3F80, dtype=np.uint16)
    with pytest.raises(nm.NmError) as e:
        nm.pack(dev(Wp), 2, 4)
    assert e.value.status == nm.NM_ERR_NOT_NM
    # the next valid pack is not affected by the previous error
    ok = to_bits(synth.nm_structured(4, 64, 2, 4, seed=1))
    nm.pack(dev(ok), 2, 4)


def test_misaligned_pointer_is_rejected(nm):
    _, masks, values, x, _, _ = oracle_case(32, 128, 2, 4, 1, seed=1, select=False)
    m = torch.from_numpy(masks.view(np.int32)).cuda()
    v = dev(values)
    xbig = torch.zeros(2, 136, dtype=torch.bfloat16, device="cuda")
    xs = xbig.view(-1)[1:129]  # 2-byte offset
    y = torch.empty(1, 32, dtype=torch.bfloat16, device="cuda")
    st = nm.lib().nm_spmv(m.data_ptr(), v.data_ptr(), xs.data_ptr(), y.data_ptr(), 32, 128, 1, None)
    assert st == nm.NM_ERR_ALIGN


# --- dense reference ------------------------------------------------------------------

@pytest.mark.parametrize("rows,K,batch", [(1, 32, 1), (33, 96, 3), (4096, 4096, 1), (4096, 14336, 1),
                                           (100, 512, 8), (6144, 4096, 4)])
def test_dense_gemv(nm, rows, K, batch):
    Wp = to_bits(synth.nm_structured(rows, K, 2, 4, seed=rows))
    x = to_bits(synth.activations(batch, K, seed=rows))
    y64, S = oracle.spmv_f64(Wp, x)
    Wd, xd = dev(Wp), dev(x)
    y32 = nm.dense_gemv(Wd, xd, f32=True).cpu().numpy()
    ybf = to_bits(nm.dense_gemv(Wd, xd))
    check_close(y32, ybf, y64, S, f"dense {rows}x{K} b{batch}")


# --- stacks and graphs -------------------------------------------------------------------

def _stack_inputs(nm, batch=1, layers=2):
    ops_s, ops_d, refs = [], [], []
    for layer in range(layers):
        for mi, name in enumerate(synth.MATRICES):
            rows, K = synth.LLAMA31_8B[name]
            rows = rows // 8  # keep the test quick; the shapes keep their K
            W = synth.nm_structured(rows, K, 16, 32, seed=layer * 4 + mi).cuda()
            m, v = nm.pack(W, 16, 32)
            x = synth.activations(batch, K, seed=100 + layer * 4 + mi).cuda()
            y = torch.empty(batch, rows, dtype=torch.bfloat16, device="cuda")
            yd = torch.empty(batch, rows, dtype=torch.bfloat16, device="cuda")
            ops_s.append(dict(masks=m, values=v, x=x, y=y, rows=rows, K=K))
            ops_d.append(dict(W=W, x=x, y=yd, rows=rows, K=K))
            refs.append((m, v, x, W))
    return ops_s, ops_d, refs


@pytest.mark.parametrize("batch", [1, 4])
def test_stack_equals_single_calls(nm, batch):
    ops_s, ops_d, refs = _stack_inputs(nm, batch)
    nm.spmv_stack(ops_s, batch)
    nm.dense_gemv_stack(ops_d, batch)
    torch.cuda.synchronize()
    for op, opd, (m, v, x, W) in zip(ops_s, ops_d, refs):
        assert torch.equal(op["y"], nm.spmv(m, v, x))
        assert torch.equal(opd["y"], nm.dense_gemv(W, x))


def test_stack_in_cuda_graph(nm):
    ops_s, _, refs = _stack_inputs(nm, 1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        nm.spmv_stack(ops_s, 1)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        nm.spmv_stack(ops_s, 1)
    for op in ops_s:
        op["y"].zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for op, (m, v, x, _) in zip(ops_s, refs):
        assert torch.equal(op["y"], nm.spmv(m, v, x))


# --- stack plans: the whole stack as one persistent launch ------------------------------------

def check_bf16(ybf: np.ndarray, y64: np.ndarray, S: np.ndarray, what: str):
    """bf16 output alone: within one ulp of y64 (plus 1e-4*S where |y64| < 1e-4*S)."""
    yb = bits_to_f32(ybf).astype(np.float64)
    err = np.abs(yb - y64)
    bound = bf16_ulp(y64) + np.where(np.abs(y64) >= TOL * S, 0.0, TOL * S)
    bad = ~(err <= bound)
    assert not bad.any(), f"{what}: {np.argwhere(bad)[:5]} err {err[bad][:5]} bound {bound[bad][:5]}"


@pytest.mark.parametrize("batch", [1, 4])
@pytest.mark.parametrize("dense", [False, True])
@pytest.mark.parametrize("persistent", [False, True])
def test_plan_matches_oracle(nm, batch, dense, persistent):
    ops_s, ops_d, refs = _stack_inputs(nm, batch)
    ops = ops_d if dense else ops_s
    for op in ops:
        op["y"].fill_(float("nan"))
    plan = nm.StackPlan(ops, batch, dense=dense, persistent=persistent)
    plan.run()
    torch.cuda.synchronize()
    for i, (op, (_, _, x, W)) in enumerate(zip(ops, refs)):
        y64, S = oracle.spmv_f64(to_bits(W.cpu()), to_bits(x.cpu()))
        check_bf16(to_bits(op["y"]), y64, S, f"plan op {i} {'dense' if dense else 'sparse'} b{batch}")
    plan.close()
    assert nm.device_status() == nm.NM_OK


# A chain in which op i+1 reads op i's output: an op that read its x before the
# previous op had stored all of it would see NaN (outputs start as NaN) or a
# stale value, and miss the oracle computed on what it actually read.
@pytest.mark.parametrize("batch", [1, 3])
@pytest.mark.parametrize("persistent", [False, True])
def test_plan_chained_dependency(nm, batch, persistent):
    shapes = [(1024, 4096), (2048, 1024), (512, 2048), (4096, 512), (896, 4096), (4096, 896),
              (128, 4096), (6144, 128), (4096, 6144), (4096, 4096), (32, 4096), (4096, 32)]
    shapes = [(r, k) for r, k in shapes if k % 128 == 0]
    for (r0, _), (_, k1) in zip(shapes, shapes[1:]):
        assert r0 == k1
    x0 = synth.activations(batch, shapes[0][1], seed=5).cuda()
    ops, Ws, x = [], [], x0
    for i, (rows, K) in enumerate(shapes):
        W = synth.nm_structured(rows, K, 2, 4, seed=50 + i)
        # keep the chain's values O(1): scale by 1/sqrt(K/2 * 0.02^2)
        W = (W.float() * (1.0 / (0.02 * (K / 2) ** 0.5))).to(torch.bfloat16)
        m, v = nm.pack(W.cuda(), 2, 4)
        y = torch.full((batch, rows), float("nan"), dtype=torch.bfloat16, device="cuda")
        ops.append(dict(masks=m, values=v, x=x, y=y, rows=rows, K=K))
        Ws.append(W)
        x = y
    plan = nm.StackPlan(ops, batch, persistent=persistent)
    for rep in range(3):
        for op in ops:
            op["y"].fill_(float("nan"))
        plan.run()
        torch.cuda.synchronize()
        for i, (op, W) in enumerate(zip(ops, Ws)):
            xin = to_bits(op["x"].cpu())  # what op i actually read: op i-1's output
            assert not np.isnan(bits_to_f32(xin)).any(), f"op {i}: input still NaN"
            y64, S = oracle.spmv_f64(to_bits(W), xin)
            check_bf16(to_bits(op["y"]), y64, S, f"chain op {i} rep {rep}")
    plan.close()
    assert nm.device_status() == nm.NM_OK


@pytest.mark.parametrize("persistent", [False, True])
def test_plan_repeats_and_graph_replay_bit_exact(nm, persistent):
    ops_s, _, _ = _stack_inputs(nm, 1)
    plan = nm.StackPlan(ops_s, 1, persistent=persistent)
    plan.run()
    torch.cuda.synchronize()
    first = [op["y"].clone() for op in ops_s]
    for _ in range(20):
        plan.run()
    torch.cuda.synchronize()
    for op, f in zip(ops_s, first):
        assert torch.equal(op["y"], f)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            plan.run()
    torch.cuda.current_stream().wait_stream(s)
    for op in ops_s:
        op["y"].zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for op, f in zip(ops_s, first):
        assert torch.equal(op["y"], f)
    plan.close()
    assert nm.device_status() == nm.NM_OK


def test_plans_of_different_sizes_interleave(nm):
    # a persistent plan with many ops, then one with a single op (less shared
    # memory), then both run: creating the small plan must not break the large one
    ops_s, _, refs = _stack_inputs(nm, 1)
    big = nm.StackPlan(ops_s, 1, persistent=True)
    small = nm.StackPlan(ops_s[:1], 1, persistent=True)
    for op in ops_s:
        op["y"].fill_(float("nan"))
    big.run()
    small.run()
    big.run()
    torch.cuda.synchronize()
    for i, (op, (_, _, x, W)) in enumerate(zip(ops_s, refs)):
        y64, S = oracle.spmv_f64(to_bits(W.cpu()), to_bits(x.cpu()))
        check_bf16(to_bits(op["y"]), y64, S, f"large plan op {i}")
    big.close()
    small.close()
    assert nm.device_status() == nm.NM_OK


def test_plan_falls_back_to_chained_launches(nm):
    # K = 96 is off the TMA path: the plan runs the ops as nm_spmv_stack would
    ops_s, _, refs = _stack_inputs(nm, 2, layers=1)
    W = synth.nm_structured(40, 96, 2, 4, seed=3).cuda()
    m, v = nm.pack(W, 2, 4)
    x = synth.activations(2, 96, seed=4).cuda()
    ops = ops_s + [dict(masks=m, values=v, x=x, y=torch.empty(2, 40, dtype=torch.bfloat16, device="cuda"),
                        rows=40, K=96)]
    refs = refs + [(m, v, x, W)]
    plan = nm.StackPlan(ops, 2, persistent=True)
    plan.run()
    torch.cuda.synchronize()
    for op, (m, v, x, _) in zip(ops, refs):
        assert torch.equal(op["y"], nm.spmv(m, v, x))
    plan.close()


# --- q/k/v projection stored in three buffers (nm_spmv_qkv) ------------------------------------

@pytest.mark.parametrize("batch", [1, 3, 8])
@pytest.mark.parametrize("rows_q,rows_k,rows_v,K", [(4096, 1024, 1024, 4096), (96, 32, 32, 256),
                                                    (100, 20, 30, 96), (0, 64, 64, 128), (64, 0, 40, 128)])
def test_spmv_qkv(nm, rows_q, rows_k, rows_v, K, batch):
    rows = rows_q + rows_k + rows_v
    Wp = to_bits(synth.nm_structured(rows, K, 2, 4, seed=rows + K))
    masks, values = oracle.pack(Wp, 2, 4)
    xb = to_bits(synth.activations(batch, K, seed=batch + K))
    y64, S = oracle.spmv_f64(Wp, xb)
    m = torch.from_numpy(masks.view(np.int32)).cuda()
    v, x = dev(values), dev(xb)
    q, k, vv = nm.spmv_qkv(m, v, x, rows_q, rows_k)
    y = nm.spmv(m, v, x)
    torch.cuda.synchronize()
    assert q.shape == (batch, rows_q) and k.shape == (batch, rows_k) and vv.shape == (batch, rows_v)
    cat = torch.cat([q, k, vv], dim=1)
    assert torch.equal(cat, y), "the three parts differ from nm_spmv's y"
    check_bf16(to_bits(cat.cpu()), y64, S, f"qkv {rows_q}/{rows_k}/{rows_v} b{batch}")


def test_qkv_op_in_a_plan_feeds_the_next_op(nm):
    # qkv of a small layer stores q, k, v apart; the next op reads v as its x
    rq, rk, rv, K = 256, 128, 128, 512
    W1 = synth.nm_structured(rq + rk + rv, K, 4, 8, seed=41)
    W2 = synth.nm_structured(96, rv, 4, 8, seed=42)
    W2 = (W2.float() * (1.0 / (0.02 * (rv / 2) ** 0.5))).to(torch.bfloat16)
    m1, v1 = nm.pack(W1.cuda(), 4, 8)
    m2, v2 = nm.pack(W2.cuda(), 4, 8)
    x = synth.activations(2, K, seed=43).cuda()
    q = torch.full((2, rq), float("nan"), dtype=torch.bfloat16, device="cuda")
    k = torch.full((2, rk), float("nan"), dtype=torch.bfloat16, device="cuda")
    vv = torch.full((2, rv), float("nan"), dtype=torch.bfloat16, device="cuda")
    y2 = torch.full((2, 96), float("nan"), dtype=torch.bfloat16, device="cuda")
    ops = [dict(masks=m1, values=v1, x=x, y=q, y_k=k, y_v=vv, rows=rq + rk + rv, K=K, flags=nm.NM_LINEAR_QKV,
                rows_q=rq, rows_k=rk),
           dict(masks=m2, values=v2, x=vv, y=y2, rows=96, K=rv)]
    for persistent in (False, True):  # persistent plans store plain y only: this one runs as a chain
        plan = nm.StackPlan(ops, 2, persistent=persistent)
        plan.run()
        torch.cuda.synchronize()
        full = nm.spmv(m1, v1, x)
        assert torch.equal(torch.cat([q, k, vv], dim=1), full)
        y64, S = oracle.spmv_f64(to_bits(W2), to_bits(vv.cpu()))
        check_bf16(to_bits(y2.cpu()), y64, S, "op after qkv")
        plan.close()
    assert nm.device_status() == nm.NM_OK


def test_spmv_qkv_rejects_bad_arguments(nm):
    m = torch.zeros(64, 4, dtype=torch.int32, device="cuda")
    v = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(1, 128, dtype=torch.bfloat16, device="cuda")
    L = nm.lib()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    o = torch.zeros(1, 64, dtype=torch.bfloat16, device="cuda").data_ptr()
    assert L.nm_spmv_qkv(m.data_ptr(), v.data_ptr(), x.data_ptr(), o, o, o, -1, 32, 32, 128, 1, s) == nm.NM_ERR_SHAPE
    assert L.nm_spmv_qkv(m.data_ptr(), v.data_ptr(), x.data_ptr(), o, None, o, 32, 16, 16, 128, 1, s) == \
        nm.NM_ERR_INVALID_ARG
    assert L.nm_spmv_qkv(m.data_ptr(), v.data_ptr(), x.data_ptr(), o + 2, o, o, 32, 16, 16, 128, 1, s) == \
        nm.NM_ERR_ALIGN
    assert L.nm_spmv_qkv(m.data_ptr(), v.data_ptr(), x.data_ptr(), o, o, o, 32, 16, 16, 128, 9, s) == \
        nm.NM_ERR_UNSUPPORTED


# --- gate/up SpMV with the SwiGLU epilogue ---------------------------------------------------

def check_swiglu(hbf: np.ndarray, h64, g64, u64, Sg, Su, what: str):
    """h = silu(g) * u from fp32 g, u (each within 1e-4 * S of the oracle) in fp32, rounded to bf16.
    |silu'| <= 1.1, so |h32 - h64| <= 1.1 dg (|u| + du) + (|silu(g)| + 1.1 dg) du + 1e-6 |h|
    (fp32 evaluation), dg = 1e-4 Sg, du = 1e-4 Su; bf16 adds one ulp."""
    dg, du = TOL * Sg, TOL * Su
    silu = np.abs(oracle.swiglu_f64(g64, np.ones_like(g64)))
    bound = 1.1 * dg * (np.abs(u64) + du) + (silu + 1.1 * dg) * du + 1e-6 * np.abs(h64)
    bound = bound + bf16_ulp(np.abs(h64) + bound)
    err = np.abs(bits_to_f32(hbf).astype(np.float64) - h64)
    bad = ~(err <= bound)
    assert not bad.any(), f"{what}: {np.argwhere(bad)[:5]} err {err[bad][:5]} bound {bound[bad][:5]}"


def swiglu_case(rows_h, K, N, M, batch, seed):
    Wg = synth.nm_structured(rows_h, K, N, M, seed=seed)
    Wu = synth.nm_structured(rows_h, K, N, M, seed=seed + 1)
    x = synth.activations(batch, K, seed=seed + 2)
    return Wg, Wu, x


@pytest.mark.parametrize("N,M", synth.PATTERNS)
def test_pack_swiglu_bit_exact(nm, N, M):
    Wg, Wu, _ = swiglu_case(48, 256, N, M, 1, seed=7)
    masks, values = nm.pack_swiglu(Wg.cuda(), Wu.cuda(), N, M)
    om, ov = oracle.pack(oracle.pair_rows(to_bits(Wg), to_bits(Wu)), N, M)
    np.testing.assert_array_equal(masks_np(masks), om)
    np.testing.assert_array_equal(to_bits(values), ov)


# TMA path (K % 128 == 0) and fallback path; one row-block pair up to many
@pytest.mark.parametrize("rows_h,K", [(16, 128), (48, 512), (256, 4096), (1024, 1024), (16, 96), (80, 160)])
@pytest.mark.parametrize("batch", [1, 3, 8])
def test_spmv_swiglu(nm, rows_h, K, batch):
    Wg, Wu, x = swiglu_case(rows_h, K, 2, 4, batch, seed=rows_h + K)
    masks, values = nm.pack_swiglu(Wg.cuda(), Wu.cuda(), 2, 4)
    h = nm.spmv_swiglu(masks, values, x.cuda())
    torch.cuda.synchronize()
    h64, g64, u64, Sg, Su = oracle.spmv_swiglu_f64(to_bits(Wg), to_bits(Wu), to_bits(x))
    check_swiglu(to_bits(h), h64, g64, u64, Sg, Su, f"swiglu {rows_h}x{K} b{batch}")


@pytest.mark.parametrize("N,M", [(2, 4), (16, 32)])
def test_spmv_swiglu_llama_gate_up_sampled(nm, N, M):
    rows_h, K = synth.LLAMA31_8B["gate_up"][0] // 2, synth.LLAMA31_8B["gate_up"][1]
    Wg = synth.nm_structured(rows_h, K, N, M, seed=21, device="cuda")
    Wu = synth.nm_structured(rows_h, K, N, M, seed=22, device="cuda")
    x = synth.activations(1, K, seed=23, device="cuda")
    masks, values = nm.pack_swiglu(Wg, Wu, N, M)
    h = nm.spmv_swiglu(masks, values, x)
    torch.cuda.synchronize()
    idx = sampled_rows(rows_h, 24)
    sel = torch.from_numpy(idx).cuda()
    h64, g64, u64, Sg, Su = oracle.spmv_swiglu_f64(to_bits(Wg[sel].cpu()), to_bits(Wu[sel].cpu()), to_bits(x.cpu()))
    check_swiglu(to_bits(h)[:, idx], h64, g64, u64, Sg, Su, f"llama gate_up swiglu {N}:{M}")


@pytest.mark.parametrize("persistent", [False, True])
def test_swiglu_op_feeds_down_in_a_stack(nm, persistent):
    """gate_up with the SwiGLU epilogue, then down reading h: an MLP of one decode layer."""
    rows_h, K = 1024, 512
    Wg, Wu, x = swiglu_case(rows_h, K, 2, 4, 1, seed=40)
    Wd = synth.nm_structured(K, rows_h, 2, 4, seed=43)
    mgu, vgu = nm.pack_swiglu(Wg.cuda(), Wu.cuda(), 2, 4)
    md, vd = nm.pack(Wd.cuda(), 2, 4)
    h = torch.full((1, rows_h), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = torch.full((1, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    ops = [dict(masks=mgu, values=vgu, x=x.cuda(), y=h, rows=2 * rows_h, K=K, flags=nm.NM_LINEAR_SWIGLU),
           dict(masks=md, values=vd, x=h, y=y, rows=K, K=rows_h)]
    plan = nm.StackPlan(ops, 1, persistent=persistent)  # a SwiGLU op keeps the plan on chained launches
    plan.run()
    torch.cuda.synchronize()
    h64, g64, u64, Sg, Su = oracle.spmv_swiglu_f64(to_bits(Wg), to_bits(Wu), to_bits(x))
    check_swiglu(to_bits(h), h64, g64, u64, Sg, Su, "stack swiglu")
    y64, S = oracle.spmv_f64(to_bits(Wd), to_bits(h.cpu()))  # down on what it actually read
    check_bf16(to_bits(y), y64, S, "stack down")
    plan.close()


def test_no_bounded_wait_ran_out(nm):
    assert nm.device_status() == nm.NM_OK


@pytest.mark.parametrize("batch", [1, 3])
def test_plan_reads_current_inputs_each_run(nm, batch):
    """The chained plan replays a graph captured at creation: each run must read
    x as it is then (no values are frozen into the graph), on any stream."""
    ops_s, _, refs = _stack_inputs(nm, batch, layers=1)
    plan = nm.StackPlan(ops_s, batch)
    for trial in range(3):
        for i, op in enumerate(ops_s):
            op["x"].copy_(synth.activations(batch, op["K"], seed=700 + 10 * trial + i).cuda())
            op["y"].fill_(float("nan"))
        s = torch.cuda.Stream() if trial == 2 else torch.cuda.current_stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            plan.run()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for i, (op, (_, _, _, W)) in enumerate(zip(ops_s, refs)):
            y64, S = oracle.spmv_f64(to_bits(W.cpu()), to_bits(op["x"].cpu()))
            check_bf16(to_bits(op["y"]), y64, S, f"plan run {trial} op {i} b{batch}")
    plan.close()
    assert nm.device_status() == nm.NM_OK
