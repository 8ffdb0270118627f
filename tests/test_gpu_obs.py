"""GPU parity of the OBS N:M pruning (nm_obs_hessian, nm_obs_prune) against
the fp64 oracle in oracle/obs.py.

Both sides get the same inputs: W from the synthetic weights, H computed by
the oracle in fp64 from synthetic calibration inputs and rounded to fp32 (the
oracle then reads those fp32 values exactly).

The N:M choice is decided by floating point on both sides, in different
precision and summation order, so a row may legitimately take another branch
where two saliencies nearly tie. The checks:
  * masks: every row has exactly N kept per M-group; a row whose mask differs
    from the oracle's must differ first at a group whose oracle saliencies at
    the keep/remove boundary lie within TIE_REL of each other, and such rows
    are rare (at most MAX_FLIP_FRAC of the rows);
  * values, in rows whose masks agree: |gpu - oracle| <= VAL_REL * max|W row|;
  * the layer objective sum (w - w') H (w - w')^T of the GPU result is within
    OBJ_REL of the oracle's (over all rows, flipped ones included);
  * the bf16 output is the fp32 output rounded to nearest even, removed
    entries are +0, and nm_pack of it reproduces the keep masks.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import obs
from tests.bits import bits_to_f64, to_bits

pytestmark = pytest.mark.gpu

# fp32 pipeline vs fp64 oracle (the derivation is in the design notes):
TIE_REL = 2e-3        # relative saliency gap below which a flipped choice is accepted
MAX_FLIP_FRAC = 0.05  # at most this fraction of rows may take another branch
VAL_REL = 5e-4        # value tolerance, relative to the row's largest dense weight
OBJ_REL = 2e-3        # layer objective, relative


@pytest.fixture(scope="module")
def nm():
    from sparse_decoding_gb300 import build
    build.build()
    import sparse_decoding_gb300 as nm
    torch.cuda.set_device(0)
    nm.init()
    return nm


def _inputs(rows, K, T, seed, dead=()):
    W = synth.weights(rows, K, seed=seed)
    X = synth.calibration(T, K, seed=seed, dead=dead)
    H32 = obs.hessian_f64(to_bits(X)).astype(np.float32)
    return W, X, H32


def _gpu_prune(nm, W, H32, N, M, percdamp=0.01, sgemm=False):
    Wb, m, wf = nm.obs_prune(W.cuda(), torch.from_numpy(H32).cuda(), N, M, percdamp, sgemm=sgemm, f32=True)
    return to_bits(Wb), m.cpu().numpy().view(np.uint32), wf.cpu().numpy().astype(np.float64)


def _check(W, H32, N, M, gpu, percdamp=0.01, rows_idx=None):
    """Compare a GPU result (bits, masks, f32) with the oracle on the rows rows_idx."""
    Wb, masks, wf = gpu
    W64 = W.float().numpy().astype(np.float64)
    if rows_idx is not None:
        W64, Wb, masks, wf = W64[rows_idx], Wb[rows_idx], masks[rows_idx], wf[rows_idx]
    H64 = H32.astype(np.float64)
    Wo, ko, so = obs.obs_prune_f64(W64, H64, N, M, percdamp, return_scores=True)
    rows, K = W64.shape
    keep = ((masks[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(rows, K).astype(bool)
    assert np.all(keep.reshape(rows, -1, M).sum(axis=2) == N), "not N kept per M-group"
    # output format: removed entries +0, bf16 = rn(f32)
    assert np.all(Wb[~keep] == 0) and np.all(wf[~keep] == 0.0)
    rn = to_bits(torch.from_numpy(wf.astype(np.float32)).to(torch.bfloat16))
    assert np.array_equal(rn, Wb), "bf16 output is not the rounded fp32 output"
    flips = []
    for r in range(rows):
        bad = np.nonzero((keep[r] != ko[r]).reshape(-1, M).any(axis=1))[0]
        if len(bad) == 0:
            tol = VAL_REL * np.abs(W64[r]).max()
            err = np.abs(wf[r] - Wo[r]).max()
            assert err <= tol, f"row {r}: |gpu - oracle| = {err:.3e} > {tol:.3e}"
            continue
        g = bad[0]
        s = np.sort(so[r, g * M:(g + 1) * M])[::-1]
        gap = (s[N - 1] - s[N]) / max(s[N - 1], 1e-300)
        assert gap <= TIE_REL, f"row {r} group {g}: choice differs at a clear gap {gap:.3e}"
        flips.append(r)
    assert len(flips) <= max(2, MAX_FLIP_FRAC * rows), f"{len(flips)} of {rows} rows flipped"
    Hd, Wd = obs.damp(H64, W64, percdamp)
    f_gpu = obs.objective_f64(Wd, wf, Hd)
    f_orc = obs.objective_f64(Wd, Wo, Hd)
    assert f_gpu <= f_orc * (1 + OBJ_REL), (f_gpu, f_orc)
    return len(flips)


@pytest.mark.parametrize("N,M", synth.PATTERNS + ((1, 4), (3, 8), (1, 2)))
def test_prune_matches_oracle(nm, N, M):
    # K = 352: two full 128-column blocks and a ragged 96-column block
    W, X, H32 = _inputs(96, 352, 512, seed=M * 7 + N)
    _check(W, H32, N, M, _gpu_prune(nm, W, H32, N, M))


@pytest.mark.parametrize("sgemm", [False, True])
def test_prune_both_trailing_update_gemms(nm, sgemm):
    W, X, H32 = _inputs(130, 416, 300, seed=5)
    _check(W, H32, 2, 4, _gpu_prune(nm, W, H32, 2, 4, sgemm=sgemm))


def test_prune_singular_hessian_dead_columns_and_damping(nm):
    # fewer tokens than columns (H singular without damping) and two inputs that never fire
    W, X, H32 = _inputs(64, 256, 100, seed=8, dead=(3, 130))
    assert H32[3, 3] == 0 and H32[130, 130] == 0
    for pd in (0.01, 0.1):
        gpu = _gpu_prune(nm, W, H32, 8, 16, percdamp=pd)
        assert np.all(gpu[2][:, [3, 130]] == 0.0)
        _check(W, H32, 8, 16, gpu, percdamp=pd)


def test_prune_single_block_and_tiny_rows(nm):
    for rows, K in ((1, 32), (3, 128), (17, 160)):
        W, X, H32 = _inputs(rows, K, 64, seed=rows)
        _check(W, H32, 2, 4, _gpu_prune(nm, W, H32, 2, 4))


def test_prune_keep_all_is_identity(nm):
    W, X, H32 = _inputs(40, 192, 256, seed=2)
    Wb, masks, wf = _gpu_prune(nm, W, H32, 4, 4)
    assert np.all(masks == 0xFFFFFFFF)
    assert np.array_equal(Wb, to_bits(W))


def test_prune_output_feeds_pack(nm):
    W, X, H32 = _inputs(128, 512, 512, seed=4)
    Wb_t, m, _ = nm.obs_prune(W.cuda(), torch.from_numpy(H32).cuda(), 2, 4)
    pm, pv = nm.pack(Wb_t, 2, 4)
    keep_bits = m.cpu().numpy().view(np.uint32)
    Wb = to_bits(Wb_t)
    # every kept weight here is nonzero (continuous values), so the pack finds the same masks
    keep = ((keep_bits[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(128, 512).astype(bool)
    assert np.all(bits_to_f64(Wb)[keep] != 0)
    assert np.array_equal(pm.cpu().numpy().view(np.uint32), keep_bits)


def test_workspace_pool_is_reused_and_released(nm):
    # the workspace (12 K^2 + 4 rows K + ... bytes, here about 24 MB) stays in
    # the library's pool after a call, gives the same result on reuse, and
    # nm_obs_release_workspace returns it to the device
    W, X, H32 = _inputs(256, 1024, 600, seed=8)
    first = _gpu_prune(nm, W, H32, 2, 4)
    torch.cuda.synchronize()
    free_kept = torch.cuda.mem_get_info()[0]
    second = _gpu_prune(nm, W, H32, 2, 4)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_kept, "a repeated call mapped new memory"
    for a, b in zip(first, second):
        assert np.array_equal(a, b)
    nm.obs_release_workspace()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] - free_kept >= 12 * 1024 * 1024, "the pool kept its memory"
    third = _gpu_prune(nm, W, H32, 2, 4)
    for a, b in zip(first, third):
        assert np.array_equal(a, b)


def test_not_positive_definite_is_reported(nm):
    W = synth.weights(8, 64, seed=1)
    H = -torch.eye(64, dtype=torch.float32)
    with pytest.raises(nm.NmError) as e:
        nm.obs_prune(W.cuda(), H.cuda(), 2, 4)
    assert e.value.status == nm.NM_ERR_NOT_PD
    # the device stays usable
    W2, X, H32 = _inputs(16, 64, 64, seed=3)
    _check(W2, H32, 2, 4, _gpu_prune(nm, W2, H32, 2, 4))


def test_hessian_matches_oracle_and_accumulates(nm):
    T, K = 700, 352
    X = synth.calibration(T, K, seed=6, dead=(7,))
    H64 = obs.hessian_f64(to_bits(X))
    x = bits_to_f64(to_bits(X))
    bound = T * 2.0 ** -23 * 2.0 * (np.abs(x).T @ np.abs(x)) + 1e-30  # recursive-summation bound, any order
    Hg = nm.obs_hessian(X.cuda()).cpu().numpy().astype(np.float64)
    assert np.all(np.abs(Hg - H64) <= bound)
    assert np.array_equal(Hg, Hg.T) or np.all(np.abs(Hg - Hg.T) <= bound)
    assert np.all(Hg[7, :] == 0) and np.all(Hg[:, 7] == 0)
    Xc = X.cuda()
    Ha = nm.obs_hessian(Xc[:300].contiguous())
    nm.obs_hessian(Xc[300:].contiguous(), Ha, accumulate=True)
    assert np.all(np.abs(Ha.cpu().numpy().astype(np.float64) - H64) <= bound)
    Hz = nm.obs_hessian(Xc[:0])
    assert Hz.shape == (K, K) and bool((Hz == 0).all())


@pytest.mark.slow
@pytest.mark.parametrize("rows,K,N,M", [(4096, 4096, 2, 4), (1024, 14336, 16, 32)])
def test_prune_full_size_sampled_rows(nm, rows, K, N, M):
    """Llama-3.1-8B shapes (o_proj; down_proj rows cut to 1024), calibration of
    2048 tokens; the oracle checks 12 sampled rows (rows are independent given H)."""
    W = synth.weights(rows, K, seed=9, device="cuda").cpu()
    X = synth.calibration(2048, K, seed=9)
    H32 = obs.hessian_f64(to_bits(X)).astype(np.float32)
    gpu = _gpu_prune(nm, W, H32, N, M)
    idx = np.random.default_rng(0).choice(rows, 12, replace=False)
    idx.sort()
    _check(W, H32, N, M, gpu, rows_idx=idx)
