"""Pins for the CPU oracle, checked against what the pages and mathematics fix.

None of these tests compares the oracle with itself: expected values come from
independent constructions (enumerated masks, numpy's float64 matmul, exact
integer arithmetic, closed forms, numpy's stable argsort) or from numbers the
pages state (tests/golden/format_facts.json).
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.bits import bits_to_f32, bits_to_f64, popcount32, to_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
PATTERNS = synth.PATTERNS


def _keep_from_masks(masks: np.ndarray) -> np.ndarray:
    """uint32 [rows][words] -> bool [rows][words*32], bit j <-> column 32g+j."""
    bits = (masks[..., None] >> np.arange(32, dtype=np.uint32)) & 1
    return bits.reshape(masks.shape[0], -1).astype(bool)


def _masks_from_subgroup_patterns(pats: np.ndarray, M: int) -> np.ndarray:
    """pats: [rows][32/M] subgroup bit patterns (bit i = column s*M+i) -> word."""
    out = np.zeros(pats.shape[0], dtype=np.uint64)
    for s in range(pats.shape[1]):
        out |= pats[:, s].astype(np.uint64) << np.uint64(s * M)
    return out.astype(np.uint32)


def _nonzero_bf16(rows, K, seed):
    w = to_bits(synth.weights(rows, K, seed=seed))
    # replace the (rare) exact zeros by 2^-6 so every drawn value is nonzero
    w = np.where((w & 0x7FFF) == 0, np.uint16(0x3C80), w)
    return w


def _check_pack_against_construction(expected_masks: np.ndarray, N: int, M: int, seed: int):
    """Build W from known masks, pack with the oracle, compare with the construction."""
    rows = expected_masks.shape[0]
    keep = _keep_from_masks(expected_masks[:, None])
    vals = _nonzero_bf16(rows, 32, seed)
    W = np.where(keep, vals, np.uint16(0))
    masks, values = oracle.pack(W, N, M)
    np.testing.assert_array_equal(masks[:, 0], expected_masks)
    # numpy boolean indexing walks each row in ascending column order
    np.testing.assert_array_equal(values, vals[keep].reshape(rows, 16))
    np.testing.assert_array_equal(oracle.unpack(masks, values, 32), W)
    return W, masks, values


# --- golden facts from the pages ----------------------------------------------

def test_golden_format_facts_metadata_bytes():
    facts = json.load(open(os.path.join(GOLDEN, "format_facts.json")))
    rows, K = 64, 1024
    for N, M in facts["patterns"]["value"]:
        W = to_bits(synth.nm_structured(rows, K, N, M, seed=1))
        masks, values = oracle.pack(W, N, M)
        kept = values.size
        assert kept / (rows * K) == facts["kept_fraction"]["value"]
        bits = masks.nbytes * 8
        assert bits / kept == facts["metadata_bits_per_kept_value"]["value"]
        assert (32 * kept) / bits == facts["reduction_vs_int32_index"]["value"]
        assert (8 * kept) / bits == facts["reduction_vs_uint8_offset"]["value"]
        assert masks.dtype.itemsize * 8 == facts["word_bits"]["value"]
        assert np.all(popcount32(masks) == facts["set_bits_per_word"]["value"])


def test_patterns_have_identical_bytes_per_row():
    """All four 50% patterns store the same bytes per row (ai.info, Main Findings,
    'Near-identical throughput across patterns is expected')."""
    sizes = set()
    for N, M in PATTERNS:
        W = to_bits(synth.nm_structured(8, 4096, N, M, seed=2))
        masks, values = oracle.pack(W, N, M)
        sizes.add((masks.nbytes, values.nbytes))
    assert len(sizes) == 1
    (mb, vb), = sizes
    assert mb == 8 * 4096 // 8 and vb == 8 * 4096  # K/8 mask bytes, K/2 bf16 values


# --- pack / unpack: brute force over masks --------------------------------------

@pytest.mark.slow
def test_pack_2_4_every_word():
    """All 6^8 = 1,679,616 valid 2:4 words of one 32-column group."""
    nibbles = np.array([p for p in range(16) if bin(p).count("1") == 2], dtype=np.uint32)
    assert len(nibbles) == 6
    digits = np.array(list(itertools.product(range(6), repeat=8)), dtype=np.int64)
    pats = nibbles[digits]
    expected = _masks_from_subgroup_patterns(pats, 4)
    assert len(np.unique(expected)) == 6 ** 8
    W, masks, values = _check_pack_against_construction(expected, 2, 4, seed=3)
    # and the product of every one of them against numpy's float64 matmul
    x = to_bits(synth.activations(1, 32, seed=3))
    y, S = oracle.spmv_f64(W, x)
    ref = bits_to_f64(W) @ bits_to_f64(x)[0]
    np.testing.assert_allclose(y[0], ref, rtol=0, atol=1e-12 * max(1.0, S.max()))


def _all_patterns(N, M):
    return np.array([sum(1 << i for i in c) for c in itertools.combinations(range(M), N)],
                    dtype=np.uint32)


@pytest.mark.parametrize("N,M", [(4, 8), (8, 16)])
def test_pack_every_subgroup_pattern(N, M):
    """Every C(M,N) subgroup pattern appears in every subgroup position."""
    pats_all = _all_patterns(N, M)
    rng = np.random.default_rng(4)
    blocks = []
    per_word = 32 // M
    for s in range(per_word):
        p = pats_all[rng.integers(0, len(pats_all), size=(len(pats_all), per_word))]
        p[:, s] = pats_all
        blocks.append(p)
    expected = _masks_from_subgroup_patterns(np.concatenate(blocks), M)
    _check_pack_against_construction(expected, N, M, seed=5)


def test_pack_16_32_random_words():
    rng = np.random.default_rng(6)
    keys = rng.random((100_000, 32))
    ranks = keys.argsort(axis=1).argsort(axis=1)
    keep = ranks < 16
    expected = (keep.astype(np.uint64) << np.arange(32, dtype=np.uint64)).sum(axis=1).astype(np.uint32)
    _check_pack_against_construction(expected, 16, 32, seed=7)


@pytest.mark.parametrize("N,M", PATTERNS)
def test_pack_invariants_and_roundtrip_realistic(N, M):
    rows, K = 96, 1024
    W = to_bits(synth.weights(rows, K, seed=8))
    a = synth.col_norms(K, seed=8).numpy()
    Wp = oracle.select(W, a, N, M)
    masks, values = oracle.pack(Wp, N, M)
    assert np.all(popcount32(masks) == 16)
    for s in range(32 // M):
        sub = (masks >> np.uint32(s * M)) & np.uint32((1 << M) - 1 if M < 32 else 0xFFFFFFFF)
        assert np.all(popcount32(sub) == N)
    back = oracle.unpack(masks, values, K)
    np.testing.assert_array_equal(back, Wp)


def test_pack_rejects_more_than_n():
    W = np.zeros((1, 32), dtype=np.uint16)
    W[0, [0, 1, 2]] = 0x3F80  # three nonzeros in the first 2:4 subgroup
    with pytest.raises(oracle.OracleError) as e:
        oracle.pack(W, 2, 4)
    assert e.value.code == 5


def test_pack_fill_rule_and_signed_zero():
    """Fewer than N nonzeros: the lowest-index zero positions are kept, bit for bit."""
    W = np.zeros((1, 32), dtype=np.uint16)
    W[0, 2] = 0x4000            # 2.0 at column 2; subgroup 0 needs one more
    W[0, 0] = 0x8000            # -0.0 at column 0 counts as zero but is the filler
    W[0, 4:8] = [0, 0, 0, 0]    # subgroup 1 empty -> columns 4, 5
    for s in range(2, 8):
        W[0, 4 * s + 1] = 0x3F80
        W[0, 4 * s + 3] = 0xBF80
    masks, values = oracle.pack(W, 2, 4)
    m = int(masks[0, 0])
    assert m & 0xFF == 0b00110101
    assert list(values[0, :4]) == [0x8000, 0x4000, 0x0000, 0x0000]
    back = oracle.unpack(masks, values, 32)
    # unpack writes +0 at pruned positions and the stored bits at kept ones
    assert back[0, 0] == 0x8000 and back[0, 2] == 0x4000 and back[0, 1] == 0


def test_unpack_rejects_malformed_word():
    masks = np.array([[0x0000FFFF, 0x0000FFFE]], dtype=np.uint32)
    values = np.zeros((1, 32), dtype=np.uint16)
    with pytest.raises(oracle.OracleError) as e:
        oracle.unpack(masks, values, 64)
    assert e.value.code == 7


def test_pack_unsupported_and_shape():
    W = np.zeros((1, 32), dtype=np.uint16)
    with pytest.raises(oracle.OracleError) as e:
        oracle.pack(W, 3, 4)
    assert e.value.code == 4
    with pytest.raises(oracle.OracleError) as e:
        oracle.pack(np.zeros((1, 48), dtype=np.uint16), 2, 4)
    assert e.value.code == 2


def test_bit_order_closed_form():
    """Keeping the first N of every subgroup gives the masks one writes by hand."""
    expected = {(2, 4): 0x33333333, (4, 8): 0x0F0F0F0F, (8, 16): 0x00FF00FF, (16, 32): 0x0000FFFF}
    for (N, M), word in expected.items():
        W = np.zeros((1, 64), dtype=np.uint16)
        for c in range(64):
            if (c % M) < N:
                W[0, c] = 0x3F80 + c  # distinct nonzero values
        masks, values = oracle.pack(W, N, M)
        assert list(masks[0]) == [word, word]
        assert list(values[0]) == [0x3F80 + c for c in range(64) if (c % M) < N]


# --- selection --------------------------------------------------------------------

def _select_by_argsort(W, a, N, M):
    """Library construction: per subgroup, numpy stable argsort of -score."""
    rows, K = W.shape
    score = np.abs(bits_to_f32(W)) * a.astype(np.float32)[None, :]
    grp = score.reshape(rows, K // M, M)
    order = np.argsort(-grp, axis=-1, kind="stable")
    keep = np.zeros_like(grp, dtype=bool)
    np.put_along_axis(keep, order[..., :N], True, axis=-1)
    return np.where(keep.reshape(rows, K), W, np.uint16(0))


@pytest.mark.parametrize("N,M", PATTERNS)
def test_select_matches_stable_argsort(N, M):
    rows, K = 64, 512
    W = to_bits(synth.weights(rows, K, seed=9))
    a = synth.col_norms(K, seed=9).numpy()
    np.testing.assert_array_equal(oracle.select(W, a, N, M), _select_by_argsort(W, a, N, M))


@pytest.mark.parametrize("N,M", PATTERNS)
def test_select_ties_go_to_lower_index(N, M):
    """Coarse values make many equal scores; ties must resolve to the lower column."""
    rows, K = 64, 256
    rng = np.random.default_rng(10)
    W = (np.array([0x3F80, 0xBF80, 0x4000, 0x0000], dtype=np.uint16))[rng.integers(0, 4, (rows, K))]
    a = np.ones(K, dtype=np.float32)
    got = oracle.select(W, a, N, M)
    np.testing.assert_array_equal(got, _select_by_argsort(W, a, N, M))
    # all-equal scores keep exactly the first N of each subgroup
    Weq = np.full((1, 64), 0x3F80, dtype=np.uint16)
    kept = oracle.select(Weq, np.ones(64, np.float32), N, M) != 0
    assert list(np.nonzero(kept[0])[0]) == [c for c in range(64) if c % M < N]


def test_select_uses_activation_norm():
    """Equal |W|: the column with the larger a_j wins (the Wanda score, not |W| alone)."""
    W = np.full((1, 32), 0x3F80, dtype=np.uint16)
    a = np.ones(32, dtype=np.float32)
    a[:4] = [0.5, 2.0, 1.0, 3.0]
    got = oracle.select(W, a, 2, 4)
    assert list(got[0, :4] != 0) == [False, True, False, True]


# --- the fp64 product ---------------------------------------------------------------

@pytest.mark.parametrize("batch", [1, 3, 8])
def test_spmv_matches_numpy_float64(batch):
    rows, K = 257, 4096
    W = to_bits(synth.nm_structured(rows, K, 2, 4, seed=11))
    x = to_bits(synth.activations(batch, K, seed=11))
    y, S = oracle.spmv_f64(W, x)
    W64, x64 = bits_to_f64(W), bits_to_f64(x)
    ref = x64 @ W64.T
    assert np.all(np.abs(y - ref) <= 1e-12 * S)
    np.testing.assert_allclose(S, np.abs(x64[:, None, :] * W64[None, :, :]).sum(-1), rtol=1e-12)


def test_spmv_exact_integer_arithmetic():
    """Dyadic weights and small-integer x: 4*y is an integer that int64 gives exactly."""
    rows, K, batch = 64, 2048, 4
    W = to_bits(synth.nm_structured(rows, K, 4, 8, seed=12, dyadic=True))
    x = to_bits(synth.small_int_activations(batch, K, seed=12))
    y, _ = oracle.spmv_f64(W, x)
    Wi = np.rint(bits_to_f64(W) * 4).astype(np.int64)
    xi = np.rint(bits_to_f64(x)).astype(np.int64)
    np.testing.assert_array_equal(np.rint(y * 4).astype(np.int64), xi @ Wi.T)
    np.testing.assert_array_equal(y * 4, (xi @ Wi.T).astype(np.float64))


def test_spmv_one_hot_columns():
    rows, K = 40, 256
    W = to_bits(synth.nm_structured(rows, K, 8, 16, seed=13))
    for j in (0, 1, 31, 32, 100, K - 1):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, j] = 0x3F80
        y, _ = oracle.spmv_f64(W, x)
        np.testing.assert_array_equal(y[0], bits_to_f64(W)[:, j])


def test_spmv_closed_forms():
    rows, K = 16, 512
    keep = synth.random_nm_keep(rows, K, 16, 32, seed=14).numpy()
    W = np.where(keep, np.uint16(0x3F80), np.uint16(0))
    ones = np.full((1, K), 0x3F80, dtype=np.uint16)
    y, S = oracle.spmv_f64(W, ones)
    assert np.all(y == K / 2) and np.all(S == K / 2)
    y0, S0 = oracle.spmv_f64(W, np.zeros((1, K), dtype=np.uint16))
    assert np.all(y0 == 0) and np.all(S0 == 0)
    # -x gives -y exactly
    xb = to_bits(synth.activations(1, K, seed=14))
    ya, _ = oracle.spmv_f64(W, xb)
    yb, _ = oracle.spmv_f64(W, xb ^ np.uint16(0x8000))
    np.testing.assert_array_equal(ya, -yb)


def test_spmv_nan_propagates_to_its_row_only():
    rows, K = 4, 64
    W = to_bits(synth.nm_structured(rows, K, 2, 4, seed=15))
    c = int(np.nonzero(W[1])[0][0])
    W[1, c] = 0x7FC0  # NaN, kept
    x = to_bits(synth.activations(1, K, seed=15))
    y, _ = oracle.spmv_f64(W, x)
    assert np.isnan(y[0, 1]) and not np.isnan(y[0, [0, 2, 3]]).any()


def test_spmv_nonfinite_x_is_the_dense_product():
    """The oracle is the dense product over the pruned W (IEEE arithmetic):
    an Inf in x_j times a pruned zero gives NaN in every row that prunes
    column j, and rows that keep it get +-Inf. This is why the GPU test of
    non-finite activations builds the format's kept-terms-only expectation
    from the oracle run with that entry zeroed, not from this value."""
    rows, K = 64, 128
    W = to_bits(synth.nm_structured(rows, K, 2, 4, seed=17))
    c = 9
    x = to_bits(synth.activations(1, K, seed=17))
    x[0, c] = 0x7F80  # +Inf
    y, _ = oracle.spmv_f64(W, x)
    keeps = W[:, c] != 0
    assert keeps.any() and (~keeps).any()
    assert np.all(np.isnan(y[0][~keeps]))
    w = bits_to_f64(W[keeps, c])
    np.testing.assert_array_equal(np.sign(y[0][keeps]), np.sign(w))
    assert np.all(np.isinf(y[0][keeps]))


def test_packed_path_equals_dense_path():
    rows, K = 33, 1024
    W = to_bits(synth.nm_structured(rows, K, 16, 32, seed=16))
    x = to_bits(synth.activations(2, K, seed=16))
    masks, values = oracle.pack(W, 16, 32)
    y1, _ = oracle.spmv_packed_f64(masks, values, x, K)
    y2, _ = oracle.spmv_f64(W, x)
    np.testing.assert_array_equal(y1, y2)


def test_empty_shapes():
    W = np.zeros((0, 64), dtype=np.uint16)
    masks, values = oracle.pack(W, 2, 4)
    assert masks.shape == (0, 2) and values.shape == (0, 32)
    y, S = oracle.spmv_f64(W, np.zeros((1, 64), dtype=np.uint16))
    assert y.shape == (1, 0)


# --- SwiGLU epilogue (the step after the gate/up SpMV) -------------------------------------------

def test_swiglu_matches_scipy_expit():
    """silu(g) * u against scipy's logistic function (a library routine), over a wide range."""
    from scipy.special import expit
    rng = np.random.default_rng(0)
    g = np.concatenate([rng.normal(0, 3, 10000), np.linspace(-80, 80, 1601)])
    u = rng.normal(0, 2, g.size)
    h = oracle.swiglu_f64(g, u)
    ref = expit(g) * g * u
    np.testing.assert_allclose(h, ref, rtol=1e-13, atol=1e-300)


def test_swiglu_closed_forms():
    g = np.array([0.0, 1.0, -1.0, 40.0, -40.0, np.log(3.0)])
    h = oracle.swiglu_f64(g, np.ones_like(g))
    e = np.e
    expect = np.array([0.0, e / (e + 1), -1 / (e + 1), 40.0 / (1 + np.exp(-40.0)), -40.0 * np.exp(-40.0) / (1 + np.exp(-40.0)),
                       np.log(3.0) * 0.75])
    np.testing.assert_allclose(h, expect, rtol=1e-14)
    # linear in u, odd-even structure: silu(g) - silu(-g) = g
    g = np.linspace(-10, 10, 101)
    u = np.full_like(g, 2.5)
    np.testing.assert_allclose(oracle.swiglu_f64(g, u), 2.5 * oracle.swiglu_f64(g, np.ones_like(g)), rtol=1e-15)
    np.testing.assert_allclose(oracle.swiglu_f64(g, np.ones_like(g)) - oracle.swiglu_f64(-g, np.ones_like(g)), g,
                               rtol=1e-13, atol=1e-13)
    assert np.isnan(oracle.swiglu_f64(np.array([np.nan]), np.array([1.0]))[0])


def test_pair_rows_layout():
    rng = np.random.default_rng(1)
    rows_h, K = 48, 64
    Wg = rng.integers(0, 65536, (rows_h, K), dtype=np.uint16)
    Wu = rng.integers(0, 65536, (rows_h, K), dtype=np.uint16)
    P = oracle.pair_rows(Wg, Wu)
    assert P.shape == (2 * rows_h, K)
    for r in range(rows_h):
        t, i = divmod(r, 16)
        np.testing.assert_array_equal(P[32 * t + i], Wg[r])
        np.testing.assert_array_equal(P[32 * t + 16 + i], Wu[r])
    with pytest.raises(oracle.OracleError):
        oracle.pair_rows(Wg[:40], Wu[:40])


def test_spmv_swiglu_oracle_composes():
    """The fused oracle equals the plain products followed by the activation."""
    Wg = to_bits(synth.nm_structured(64, 256, 2, 4, seed=3))
    Wu = to_bits(synth.nm_structured(64, 256, 2, 4, seed=4))
    x = to_bits(synth.activations(2, 256, seed=5))
    h, g, u, Sg, Su = oracle.spmv_swiglu_f64(Wg, Wu, x)
    g2 = bits_to_f64(Wg) @ bits_to_f64(x).T
    u2 = bits_to_f64(Wu) @ bits_to_f64(x).T
    np.testing.assert_allclose(g, g2.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(u, u2.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h, g2.T / (1 + np.exp(-g2.T)) * u2.T, rtol=1e-12, atol=1e-15)
