"""Pins for the OBS N:M pruning oracle (oracle/obs.py).

Expected values come from constructions that use neither of the oracle's
update formulas:
  * constrained least squares: fixing columns left to right, the free weights
    of a row are always the minimiser of (w0 - w') H (w0 - w')^T given the fixed
    ones, and the saliency denominator 1/[inv(H[c:, c:])]_00 is the Schur
    complement of the trailing block (solved with numpy.linalg.solve);
  * closed forms: diagonal H (no compensation, saliency w^2 h), N = M (nothing
    removed), the pages' literal update delta_w = -(w_q/[H^-1]_qq) H^-1_{:,q}
    with the full inverse when the removed weight is column 0, and the loss
    increase w_q^2/[H^-1]_qq = 2 L_q of the pages;
  * brute force for H = 2 X X^T (outer products summed token by token).
"""
import numpy as np
import pytest

import synth
from oracle import obs
from tests.bits import to_bits


def _case(rows, K, T, seed, dead=()):
    W = synth.weights(rows, K, seed=seed).float().numpy().astype(np.float64)
    X = to_bits(synth.calibration(T, K, seed=seed, dead=dead))
    return W, obs.hessian_f64(X)


def _lsq_prune(W0, H0, N, M, percdamp):
    """Independent derivation: greedy left-to-right N:M by constrained least squares."""
    H, W = obs.damp(H0, W0, percdamp)  # damping is a stated reading, not under test here
    rows, K = W.shape
    out = np.zeros_like(W)
    keep = np.zeros((rows, K), dtype=bool)
    schur = np.empty(K)
    for c in range(K):
        F = slice(c + 1, K)
        schur[c] = H[c, c] - (H[c, F] @ np.linalg.solve(H[F, F], H[F, c]) if c + 1 < K else 0.0)
    for r in range(rows):
        w0 = W[r]
        fixed = np.zeros(0)
        for j in range(K):
            A, F = slice(0, j), slice(j, K)
            # best free part given the fixed prefix: w_F = w0_F + H_FF^-1 H_FA (w0_A - w_A)
            cur = w0[F] + np.linalg.solve(H[F, F], H[F, A] @ (w0[A] - fixed)) if j else w0.copy()
            if j % M == 0:
                s = cur[:M] ** 2 * schur[j:j + M]
                order = np.argsort(-s, kind="stable")
                keep[r, j + order[:N]] = True
            fixed = np.append(fixed, cur[0] if keep[r, j] else 0.0)
        out[r] = fixed
    return out, keep


@pytest.mark.parametrize("N,M,T,percdamp", [(2, 4, 48, 0.01), (4, 8, 12, 0.05), (1, 4, 40, 0.01),
                                            (3, 8, 64, 0.0)])
def test_matches_constrained_least_squares(N, M, T, percdamp):
    W0, H0 = _case(5, 32, T, seed=N * 10 + M, dead=(3,) if T < 32 else ())
    Wo, ko = obs.obs_prune_f64(W0, H0, N, M, percdamp)
    Wl, kl = _lsq_prune(W0, H0, N, M, percdamp)
    assert np.array_equal(ko, kl)
    assert np.allclose(Wo, Wl, rtol=1e-9, atol=1e-12 * np.abs(W0).max())
    assert np.all(Wo[~ko] == 0.0)
    assert np.all(ko.reshape(5, -1, M).sum(axis=2) == N)


def test_explicit_inverse_form_agrees():
    W0, H0 = _case(7, 48, 96, seed=3)
    Wo, ko = obs.obs_prune_f64(W0, H0, 2, 4)
    We, ke = obs.obs_prune_explicit_f64(W0, H0, 2, 4)
    assert np.array_equal(ko, ke)
    assert np.allclose(Wo, We, rtol=1e-9, atol=1e-14)


def test_diagonal_hessian_is_saliency_masking():
    rng = np.random.default_rng(0)
    W = rng.normal(0, 0.02, (6, 32))
    h = rng.uniform(0.5, 4.0, 32)
    Wo, ko = obs.obs_prune_f64(W, np.diag(h), 4, 8, percdamp=0.0)
    s = (W ** 2 * h).reshape(6, 4, 8)
    thr = np.sort(s, axis=2)[:, :, 4:5]  # 4th largest of 8 (no ties in continuous draws)
    expect = (s >= thr).reshape(6, 32)
    assert np.array_equal(ko, expect)
    assert np.array_equal(Wo, np.where(expect, W, 0.0))


def test_keep_all_leaves_weights():
    W0, H0 = _case(4, 16, 40, seed=5)
    Wo, ko = obs.obs_prune_f64(W0, H0, 4, 4)
    assert ko.all() and np.allclose(Wo, W0, rtol=0, atol=1e-15)


def test_pages_update_and_loss_at_first_column():
    """Remove exactly column 0 (N = M - 1 and w_0 tiny): the result is the pages'
    delta_w with the full inverse, and the loss is w_0^2/[H^-1]_00 = 2 L_0."""
    W0, H0 = _case(1, 4, 32, seed=11)
    W0[0, 0] = 1e-6
    Hd, _ = obs.damp(H0, W0, 0.01)
    Hinv = np.linalg.inv(Hd)
    Wo, ko = obs.obs_prune_f64(W0, H0, 3, 4, 0.01)
    assert ko.tolist() == [[False, True, True, True]]
    expect = W0[0] - W0[0, 0] / Hinv[0, 0] * Hinv[:, 0]
    assert np.allclose(Wo[0], expect, rtol=1e-12, atol=1e-18)
    L0 = W0[0, 0] ** 2 / (2 * Hinv[0, 0])
    assert obs.objective_f64(W0, Wo, Hd) == pytest.approx(2 * L0, rel=1e-9)


def test_compensation_never_worse_than_masking():
    W0, H0 = _case(16, 64, 80, seed=2)
    Hd, Wd = obs.damp(H0, W0, 0.01)
    Wo, ko = obs.obs_prune_f64(W0, H0, 2, 4)
    assert obs.objective_f64(Wd, Wo, Hd) < obs.objective_f64(Wd, np.where(ko, Wd, 0.0), Hd)


def test_dead_column_and_scale_invariance():
    W0, H0 = _case(4, 32, 16, seed=9, dead=(5, 17))
    assert H0[5, 5] == 0 and H0[17, 17] == 0
    Wo, ko = obs.obs_prune_f64(W0, H0, 2, 4)
    assert np.all(Wo[:, [5, 17]] == 0)
    assert np.all(ko.reshape(4, -1, 4).sum(axis=2) == 2)
    # without dead columns the damping is relative to diag H, so scaling H changes nothing
    W0, H0 = _case(4, 32, 48, seed=9)
    Wo, ko = obs.obs_prune_f64(W0, H0, 2, 4)
    W2, k2 = obs.obs_prune_f64(W0, 8.0 * H0, 2, 4)
    assert np.array_equal(ko, k2) and np.allclose(Wo, W2, rtol=1e-9, atol=1e-15)


def test_hessian_is_twice_sum_of_outer_products():
    X = to_bits(synth.calibration(9, 12, seed=4))
    x = (X.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    H = np.zeros((12, 12))
    for t in range(9):
        H += 2.0 * np.outer(x[t], x[t])
    assert np.array_equal(obs.hessian_f64(X), H) or np.allclose(obs.hessian_f64(X), H, rtol=1e-15)


def test_keep_words_bit_order():
    keep = np.zeros((2, 64), dtype=bool)
    keep[0, [0, 31, 33]] = True
    keep[1, 63] = True
    w = obs.keep_words(keep)
    assert w.tolist() == [[0x80000001, 0x2], [0, 0x80000000]]


def test_random_cases_match_least_squares():
    """Property check over random small layers: patterns with M in {2, 4, 8},
    1 <= N <= M, damping 0.001-0.2, token counts below and above K, dead inputs."""
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    @hyp.settings(max_examples=25, deadline=None, derandomize=True)
    @hyp.given(st.sampled_from([2, 4, 8]), st.integers(1, 8), st.integers(1, 3), st.integers(4, 40),
               st.floats(0.001, 0.2), st.integers(0, 10_000), st.booleans())
    def check(M, N, kgroups, T, percdamp, seed, with_dead):
        N = min(N, M)
        K = 8 * kgroups
        dead = (1,) if with_dead else ()
        W0, H0 = _case(3, K, T, seed=seed, dead=dead)
        Wo, ko = obs.obs_prune_f64(W0, H0, N, M, percdamp)
        Wl, kl = _lsq_prune(W0, H0, N, M, percdamp)
        assert np.array_equal(ko, kl)
        assert np.allclose(Wo, Wl, rtol=1e-8, atol=1e-11 * max(np.abs(W0).max(), 1e-30))
        assert np.all(ko.reshape(3, -1, M).sum(axis=2) == N)

    check()
