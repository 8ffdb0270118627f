"""CPU oracle for N:M pruning by the OBS rule (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may use this module; the product library never calls it.

What the pages fix (paper.rainbus.top summary, "前置知识" on the OBS framework
and "方法步骤详情" step 2; ai.info summary, "Methodology in Plain English"
step 1): a linear layer is pruned against the Hessian H = 2 X X^T of its
calibration inputs. Removing weight q costs L_q = w_q^2 / (2 [H^-1]_qq); the
weights that stay are compensated by delta_w = -(w_q / [H^-1]_qq) H^-1_{:,q};
the solver is SparseGPT, run to the target N:M pattern.

Readings taken where the pages stop (SparseGPT's published procedure, restated):

  * Columns are fixed one at a time, left to right. When column j is reached,
    columns < j are final and columns >= j are still free, so "H^-1" in both
    formulas is the inverse of the free block, G_j = inv(H[j:, j:]).
  * N:M choice: at the first column j of each aligned group of M columns, each
    row keeps the N weights c of the group with the largest saliency
    w_c^2 / [G_c]_00 (w_c as compensated so far; G_c because weight c is
    removed when column c is reached; the factor 1/2 of L_q does not change
    the order). Equal saliencies: the lower column is kept.
  * Fixing column j: a removed weight is set to 0 and the free columns of its
    row move by -(w_j / [G_j]_00) [G_j]_{0,:}; a kept weight moves nothing.
  * Damping (the pages give none; SparseGPT's): a column whose H_jj is 0 (an
    input that is always zero) gets H_jj = 1 and its weights 0, then
    lam = percdamp * mean(diag H) is added to the diagonal.

Evaluation: with inv(H) = U^T U (U upper triangular), [G_j]_{0,:} / [G_j]_00
= U[j, j:] / U_jj and [G_j]_00 = U_jj^2, so `obs_prune_f64` needs one
factorisation. `obs_prune_explicit_f64` inverts every trailing block instead;
the tests pin both to a derivation that uses neither formula (constrained
least squares with Schur-complement saliencies) and to closed forms.
"""
from __future__ import annotations

import numpy as np


def damp(H: np.ndarray, W: np.ndarray, percdamp: float):
    """(H + lam I with dead columns fixed, W with their weights zeroed), both float64 copies."""
    H = np.array(H, dtype=np.float64, copy=True)
    W = np.array(W, dtype=np.float64, copy=True)
    dead = np.diag(H) == 0
    H[dead, dead] = 1.0
    W[:, dead] = 0.0
    lam = percdamp * float(np.mean(np.diag(H)))
    H[np.diag_indices_from(H)] += lam
    return H, W


def select_group(scores: np.ndarray, N: int) -> np.ndarray:
    """Per row, True for the N largest scores of the group (equal scores: the lower column)."""
    order = np.argsort(-scores, axis=1, kind="stable")
    keep = np.zeros(scores.shape, dtype=bool)
    np.put_along_axis(keep, order[:, :N], True, axis=1)
    return keep


def _check(W, H, N, M):
    rows, K = np.shape(W)
    if np.shape(H) != (K, K) or K % M or not 1 <= N <= M:
        raise ValueError("bad shape or N:M")


def obs_prune_f64(W, H, N: int, M: int, percdamp: float = 0.01, return_scores: bool = False):
    """OBS N:M pruning, trailing inverses read from the factor U (inv(H) = U^T U).

    W: float [rows][K] dense weights; H: float [K][K]. Returns
    (W_pruned float64 [rows][K], keep bool [rows][K]) and, with
    return_scores, the saliency w_c^2 / [G_c]_00 each weight had when its
    group was chosen (float64 [rows][K])."""
    _check(W, H, N, M)
    H, W = damp(H, W, percdamp)
    rows, K = W.shape
    U = np.linalg.cholesky(np.linalg.inv(H)).T
    keep = np.ones((rows, K), dtype=bool)
    scores = np.zeros((rows, K))
    for j in range(K):
        if j % M == 0:
            s = W[:, j:j + M] ** 2 / np.diag(U)[j:j + M] ** 2
            scores[:, j:j + M] = s
            keep[:, j:j + M] = select_group(s, N)
        err = np.where(keep[:, j], 0.0, W[:, j] / U[j, j])
        W[:, j:] -= np.outer(err, U[j, j:])
        W[~keep[:, j], j] = 0.0  # exactly zero (the update leaves rounding residue)
    return (W, keep, scores) if return_scores else (W, keep)


def obs_prune_explicit_f64(W, H, N: int, M: int, percdamp: float = 0.01):
    """The same rule with G_j = inv(H[j:, j:]) formed for every column. O(K^4): small K only."""
    _check(W, H, N, M)
    H, W = damp(H, W, percdamp)
    rows, K = W.shape
    G = [np.linalg.inv(H[j:, j:]) for j in range(K)]
    keep = np.ones((rows, K), dtype=bool)
    for j in range(K):
        if j % M == 0:
            d = np.array([G[c][0, 0] for c in range(j, j + M)])
            keep[:, j:j + M] = select_group(W[:, j:j + M] ** 2 / d, N)
        err = np.where(keep[:, j], 0.0, W[:, j] / G[j][0, 0])
        W[:, j:] -= np.outer(err, G[j][0, :])
        W[~keep[:, j], j] = 0.0
    return W, keep


def hessian_f64(X_bits: np.ndarray) -> np.ndarray:
    """H = 2 X X^T of the pages, for calibration inputs given token-major: X_bits bf16 [T][K] -> [K][K]."""
    X = (np.asarray(X_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return 2.0 * X.T @ X


def objective_f64(W, W_pruned, H) -> float:
    """Layer reconstruction error sum over rows of (w - w') H (w - w')^T."""
    D = np.asarray(W, dtype=np.float64) - np.asarray(W_pruned, dtype=np.float64)
    return float(np.einsum("ij,jk,ik->", D, np.asarray(H, dtype=np.float64), D))


def keep_words(keep: np.ndarray) -> np.ndarray:
    """keep bool [rows][K] -> uint32 [rows][K/32], bit b of word g = column 32g + b."""
    rows, K = keep.shape
    bits = keep.reshape(rows, K // 32, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)
    return bits.sum(axis=2).astype(np.uint32)
