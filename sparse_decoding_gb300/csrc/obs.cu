// obs.cu -- N:M pruning by the OBS rule (SparseGPT's column order) on the GPU,
// and the calibration Hessian that feeds it.
//
// The rule (paper.rainbus.top summary, "前置知识" on the OBS framework and
// "方法步骤详情" step 2): with H = 2 X X^T, removing weight q costs
// w_q^2 / (2 [H^-1]_qq) and the surviving weights move by
// -(w_q / [H^-1]_qq) H^-1_{:,q}. Columns are fixed left to right; when column j
// is reached the inverse is that of the still-free block, G_j = inv(H[j:, j:]).
// At the first column of every aligned M-column group each row keeps the N
// weights with the largest w_c^2 / [G_c]_00; a removed weight at column j is
// zeroed and the free columns of its row move by -(w_j / [G_j]_00) [G_j]_{0,:}.
//
// With inv(H) = U^T U (U upper triangular), [G_j]_{0,:} / [G_j]_00 =
// U[j, j:] / U_jj and [G_j]_00 = U_jj^2, so one factor serves every column.
// U comes from the reversed matrix: if J reverses the index order and
// J H J = L L^T (Cholesky), then H = R R^T with R = J L J upper triangular
// and U = R^-1 = J L^-1 J. The sweep needs only U's 128 x 128 diagonal blocks
// (the inverses of L's diagonal blocks); the corrections between blocks are
// carried by R itself: with E the errors (w_j / U_jj for removed weights, 0
// for kept ones) and D = W0 - final weights, D = E U, so E = D R, and what the
// finished blocks owe block b is -(D R)_b U_bb.
//
// Steps of nm_obs_prune, all on the caller's stream:
//   1. obs_diag_kernel: dead columns (H_jj == 0) and the damping
//      lam = percdamp * mean(diag H with dead entries set to 1);
//      obs_reverse_damp_kernel: J (H + lam I) J, dead diagonal entries 1 + lam;
//   2. chol_inv: the Cholesky factorisation L by recursion on halves; the
//      off-diagonal steps are GEMMs, and a 128-wide diagonal block is
//      fac_diag_kernel (one CTA factors it and inverts it). Only the inverses
//      that the recursion itself needs are formed in full;
//   3. obs_reverse_kernel: R = J L J (L's flat array reversed);
//   4. per block (128 columns; a narrower one first), obs_sweep_kernel: one
//      warp per row starts from W0 + P U_bb and walks the block column by
//      column (N:M choice, in-block compensation); it writes the block's final
//      values, keep bits and D;
//   5. the lazy update P += D R, in two levels: the rest of the current
//      1024-column superblock after each block, every later column once per
//      superblock (one GEMM with k up to 1024).
// The GEMMs run on this library's tensor-core GEMM (tc_gemm.cu): fp32
// emulated by three bf16 parts per operand and the six products of order up
// to 2, accumulated in fp32 in tensor memory; the smallest ones (up to 256^3),
// and all of them with NM_OBS_SGEMM, in plain fp32 on the CUDA cores. The
// Hessian is one bf16 pass (its products are exact).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "kernels.h"

namespace nm {
namespace {

constexpr int kObsBlock = 128;   // columns per sweep block
constexpr int kSuper = 1024;     // columns per lazy-update superblock (a multiple of kObsBlock)
constexpr int kSweepWarps = 16;  // rows in flight per CTA
constexpr int kMaxDevices = 64;

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// ---- step 1: dead columns and the damping ----------------------------------

// One CTA. dead[j] = (H_jj == 0); lam = percdamp * mean(H_jj, dead -> 1),
// summed in fp64 in a fixed order (strided partial sums, then a tree).
__global__ void __launch_bounds__(1024) obs_diag_kernel(const float *__restrict__ H, int64_t K, float percdamp,
                                                        unsigned char *__restrict__ dead, float *__restrict__ lam)
{
    __shared__ double part[1024];
    pdl_wait_upstream();
    pdl_launch_dependents();
    double s = 0.0;
    for (int64_t j = threadIdx.x; j < K; j += blockDim.x) {
        float h = H[j * K + j];
        bool d = (h == 0.0f);
        dead[j] = d ? 1 : 0;
        s += d ? 1.0 : (double)h;
    }
    part[threadIdx.x] = s;
    __syncthreads();
    for (int w = 512; w > 0; w >>= 1) {
        if (threadIdx.x < w)
            part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0)
        *lam = (float)((double)percdamp * part[0] / (double)K);
}

// ---- step 2: reversed, damped copy -----------------------------------------

// Hr[p] = H[K*K - 1 - p] (Hr = J H J for the symmetric H); on the diagonal a
// zero entry becomes 1 and lam is added.
__global__ void obs_reverse_damp_kernel(const float *__restrict__ H, int64_t K, const float *__restrict__ lam,
                                        float *__restrict__ Hr)
{
    pdl_wait_upstream();
    pdl_launch_dependents();
    const int64_t n = K * K;
    const float l = *lam;
    for (int64_t p = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; p < n; p += (int64_t)gridDim.x * blockDim.x) {
        float h = H[n - 1 - p];
        if (p / K == p % K)
            h = (h == 0.0f ? 1.0f : h) + l;
        Hr[p] = h;
    }
}

// ---- step 3: the blocked Cholesky of Hr and its inverse ---------------------

constexpr int kFacB = 128;        // factorisation block
constexpr int kFacThreads = 512;  // 4 row groups x 128 columns

// One CTA factors the diagonal block [k0, k0 + kb) of the trailing-updated
// matrix A, L_kk L_kk^T = A_kk, and writes X_kk = L_kk^-1 (lower, zeros above
// the diagonal). L_kk itself is not stored: later steps read only blocks of L
// below the diagonal. A block narrower than 128 is padded with the identity.
//
// Phase 1, the factorisation: thread t = 128 g + r holds row r, columns
// 32 g .. 32 g + 31, of the working block in registers. Each step takes two
// pivots j, j + 1: the two columns are published as they stand (one shared
// store each per thread of group j / 32, double buffered so that one barrier
// per step suffices); every thread applies pivot j to the entries of column
// j + 1 it reads, then the rank-2 update
// a_rc -= a_rj a_cj / a_jj + a'_r(j+1) a'_c(j+1) / a'_(j+1)(j+1) to columns
// c > j + 1. Only entries on or below the diagonal of columns j, j + 1 are
// read, so rows already passed may take meaningless updates; warps whose rows
// are all passed, or lie above their columns, skip the step. Column j of L (a_rj / sqrt(a_jj)) and
// 1 / L_jj go to shared memory. A pivot that is not positive sets *not_pd and
// is replaced by 1.
// Phase 2, the inverse X = L^-1 in 32 x 32 blocks: four warps invert the
// diagonal blocks (forward substitution, lane = column, rows in registers);
// the blocks below follow in three waves, X_ij = -X_ii sum_k L_ik X_kj, as
// 8-row x 32-column tile products in shared memory spread over the warps.
constexpr size_t kFacSmem = (size_t)2 * kFacB * (kFacB + 1) * 4 + 3 * 32 * 33 * 4;

// acc[r] += sum_k A[r][k] B[k][lane] for 8 rows of A and 32 columns of B
// (lane = column); A, B in shared memory with row strides lda, ldb.
__device__ __forceinline__ void tile_mm8(const float *A, int lda, const float *B, int ldb, float (&acc)[8], int lane)
{
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
        const float b = B[k * ldb + lane];
#pragma unroll
        for (int r = 0; r < 8; ++r)
            acc[r] = fmaf(A[r * lda + k], b, acc[r]);
    }
}

__global__ void __launch_bounds__(kFacThreads, 1)
    fac_diag_kernel(const float *__restrict__ A, float *__restrict__ X, int64_t K, int64_t k0, int kb,
                    int *__restrict__ not_pd)
{
    extern __shared__ float Ls[];  // [128][129]: L_kk, row-major, padded; then X and scratch
    __shared__ __align__(16) float colA[2][kFacB];
    __shared__ __align__(16) float colB[2][kFacB];
    __shared__ float rdiag[kFacB];
    constexpr int P = kFacB + 1;
    pdl_wait_upstream();
    pdl_launch_dependents(); // one CTA: the next kernel's CTAs may wait on the free SMs
    {
        const int r = threadIdx.x & (kFacB - 1), g = threadIdx.x >> 7, rw0 = r & ~31;
        float a[32];
        if (r < kb && 32 * g < kb) {
            const float4 *src = reinterpret_cast<const float4 *>(A + (k0 + r) * K + k0 + 32 * g);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 v = src[q];
                a[4 * q] = v.x, a[4 * q + 1] = v.y, a[4 * q + 2] = v.z, a[4 * q + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int m = 0; m < 32; ++m)
                a[m] = (r == 32 * g + m) ? 1.0f : 0.0f;
        }
        bool bad = false;
#pragma unroll 1
        for (int gj = 0; gj < 4; ++gj) {
#pragma unroll
            for (int mp = 0; mp < 16; ++mp) {
                // pivots j and j + 1 together: both columns are published as
                // they stand before step j, and every thread applies step j to
                // the entries of column j + 1 that it needs
                const int mj = 2 * mp, j = 32 * gj + mj, buf = mp & 1;
                if (g == gj) {
                    colA[buf][r] = a[mj];
                    colB[buf][r] = a[mj + 1];
                }
                __syncthreads();
                const float d0 = colA[buf][j];
                const float rs0 = rsqrtf(d0 > 0.0f ? d0 : 1.0f), rd0 = rs0 * rs0;
                const float t = colA[buf][j + 1] * rd0;  // column j+1 -= column j * t
                const float d1 = colB[buf][j + 1] - colA[buf][j + 1] * t;
                bad |= !(d0 > 0.0f) || !(d1 > 0.0f);
                const float rs1 = rsqrtf(d1 > 0.0f ? d1 : 1.0f), rd1 = rs1 * rs1;
                if (g == gj) {
                    const float b1 = a[mj + 1] - a[mj] * t;
                    Ls[r * P + j] = r >= j ? a[mj] * rs0 : 0.0f;
                    Ls[r * P + j + 1] = r >= j + 1 ? b1 * rs1 : 0.0f;
                    if (r == j)
                        rdiag[j] = rs0;
                    if (r == j + 1)
                        rdiag[j + 1] = rs1;
                }
                // warps whose rows lie above their columns hold only the upper
                // triangle, which nothing reads
                if (g >= gj && rw0 + 31 > j && rw0 >= 32 * g) {
                    const float ca = colA[buf][r], cb = colB[buf][r] - ca * t;
                    const float ci0 = ca * rd0, ci1 = cb * rd1;
                    // a_rc -= ci0 xa_c + ci1 (xb_c - t xa_c), regrouped as
                    // (ci0 - ci1 t) xa_c + ci1 xb_c: two FMAs per entry
                    const float e0 = fmaf(-ci1, t, ci0);
#pragma unroll
                    for (int m = 0; m < 32; ++m)
                        if (g > gj || m > mj + 1)
                            a[m] = fmaf(-ci1, colB[buf][32 * g + m], fmaf(-e0, colA[buf][32 * g + m], a[m]));
                }
            }
        }
        if (bad && threadIdx.x == 0)
            atomicOr(not_pd, 1);
    }
    __syncthreads();
    {
        // Phase 2 in 32 x 32 blocks: X_pp = L_pp^-1, then for i > j
        // X_ij = -X_ii sum_{k=j}^{i-1} L_ik X_kj, in waves of i - j = 1, 2, 3.
        float *Xs = Ls + kFacB * P;  // X, row-major, padded
        float *Tb = Xs + kFacB * P;  // three 32 x 33 scratch tiles
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
        if (w < 4) {
            // warp p inverts L_pp; lane c holds column c (rows in registers)
            const int o = 32 * w;
            float x[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
                x[i] = (i == lane) ? 1.0f : 0.0f;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float xk = x[k] * rdiag[o + k];
                x[k] = xk;
#pragma unroll
                for (int i = k + 1; i < 32; ++i)
                    x[i] = fmaf(-Ls[(o + i) * P + o + k], xk, x[i]);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i)
                Xs[(o + i) * P + o + lane] = x[i];
        }
        __syncthreads();
        // warp w works on rows 8 (w & 3) .. + 7 of tile slot w >> 2
        const int slot = w >> 2, r0 = 8 * (w & 3);
        auto T = [&](int s) { return Tb + s * 32 * 33; };
#pragma unroll 1
        for (int d = 1; d <= 3; ++d) {
            const int j = slot, i = slot + d;  // block (i, j) of this wave
            const bool active = i < 4;
            if (active) {
                float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                for (int k = j; k < i; ++k)
                    tile_mm8(Ls + (32 * i + r0) * P + 32 * k, P, Xs + (32 * k) * P + 32 * j, P, acc, lane);
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    T(slot)[(r0 + r) * 33 + lane] = acc[r];
            }
            __syncthreads();
            if (active) {
                float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                tile_mm8(Xs + (32 * i + r0) * P + 32 * i, P, T(slot), 33, acc, lane);
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    Xs[(32 * i + r0 + r) * P + 32 * j + lane] = -acc[r];
            }
            __syncthreads();
        }
        // the blocks on and below the diagonal (X's upper part is zero on entry)
        for (int q = threadIdx.x; q < kFacB * kFacB; q += blockDim.x) {
            const int i = q / kFacB, c = q % kFacB;
            if ((c >> 5) <= (i >> 5) && i < kb && c < kb)
                X[(k0 + i) * K + k0 + c] = Xs[i * P + c];
        }
    }
}

// ---- step 4: R = J L J ----------------------------------------------------------

// With L row-major, R(i, j) = L(K-1-i, K-1-j) = L[K*K - 1 - (i K + j)]: R is
// the flat array of L reversed; H + lam I = R R^T with R upper triangular.
__global__ void obs_reverse_kernel(const float *__restrict__ L, int64_t n, float *__restrict__ R)
{
    pdl_wait_upstream();
    pdl_launch_dependents();
    for (int64_t p = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; p < n; p += (int64_t)gridDim.x * blockDim.x)
        R[p] = L[n - 1 - p];
}

// ---- step 6a: the column sweep of one block ----------------------------------

// Bits 0..7 of x moved to bits 0, 4, 8, ..., 28.
__device__ __forceinline__ uint32_t spread8(uint32_t x)
{
    x &= 0xFFu;
    x = (x | (x << 12)) & 0x000F000Fu;
    x = (x | (x << 6)) & 0x03030303u;
    x = (x | (x << 3)) & 0x11111111u;
    return x;
}

// One block [i1, i1 + bw) of columns, all rows. Shared memory:
// Ub[a][c] = U[i1 + a][i1 + c] = X[K-1-i1-a][K-1-i1-c] (U = J X J; zeros below
// the diagonal and outside the block), rinv[a] = 1 / Ub[a][a] and
// dsq[a] = rinv[a]^2.
// Warp w of CTA c takes rows c * 16 + w, then steps by the grid. Lane l holds
// columns i1 + 4 l + t (t = 0..3), so a row of Ub is one 16-byte load per lane
// and a 2- or 4-column group lies in one lane.
//   start : w = W0 + P U_bb, with W0 the dense weights (dead columns 0) and P
//           the accumulated D R of the blocks to the left (see the host side);
//   sweep : at the first column of each M-group the group ranks its
//           saliencies w^2 / U_cc^2 (equal ones by column) and keeps the N
//           largest; a removed column j sends err = w_j / U_jj and every later
//           column c of the block takes w_c -= err U_jc (kept columns move
//           nothing; the zeros of Ub below the diagonal leave the passed
//           columns as they are);
//   output: the final values (bf16, and fp32 if asked), the keep bits as the
//           decode format's mask words, and D = W0 - final.
template <int M>
__global__ void __launch_bounds__(kSweepWarps * 32, 2) obs_sweep_kernel(
    const __nv_bfloat16 *__restrict__ W, const unsigned char *__restrict__ dead, const float *__restrict__ P,
    const float *__restrict__ X, int64_t rows, int64_t K, int i1, int bw, int N, float *__restrict__ D, int ldD,
    __nv_bfloat16 *__restrict__ Wout, float *__restrict__ Wout_f32, uint32_t *__restrict__ masks)
{
    extern __shared__ float4 smem4[];
    float *Ub = reinterpret_cast<float *>(smem4);
    float *rinv = Ub + kObsBlock * kObsBlock;
    float *dsq = rinv + kObsBlock;
    constexpr int kQuads = kObsBlock / 4;
    pdl_wait_upstream();
    pdl_launch_dependents(); // a single wave (at most two CTAs per SM)
    for (int q = threadIdx.x; q < kObsBlock * kQuads; q += blockDim.x) {
        const int a = q / kQuads, c = (q % kQuads) * 4;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (a < bw && c < bw) {
            // columns K-4-i1-c .. K-1-i1-c of row K-1-i1-a, reversed
            const float4 x = *reinterpret_cast<const float4 *>(X + (K - 1 - i1 - a) * K + (K - 4 - i1 - c));
            v = make_float4(c >= a ? x.w : 0.0f, c + 1 >= a ? x.z : 0.0f, c + 2 >= a ? x.y : 0.0f,
                            c + 3 >= a ? x.x : 0.0f);
        }
        smem4[q] = v;
    }
    __syncthreads();
    for (int a = threadIdx.x; a < kObsBlock; a += blockDim.x) {
        const float ri = a < bw ? 1.0f / Ub[a * kObsBlock + a] : 0.0f;
        rinv[a] = ri;
        dsq[a] = ri * ri;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nq = bw >> 2;
    const bool mine = 4 * lane < bw;  // this lane holds columns of the block
    for (int64_t r = (int64_t)blockIdx.x * kSweepWarps + warp; r < rows; r += (int64_t)gridDim.x * kSweepWarps) {
        const int64_t base = r * K + i1 + 4 * lane;
        float w0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, p[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (mine) {
            const uint2 wb = *reinterpret_cast<const uint2 *>(W + base);
            const uchar4 dd = *reinterpret_cast<const uchar4 *>(dead + i1 + 4 * lane);
            w0[0] = dd.x ? 0.0f : __uint_as_float(wb.x << 16);
            w0[1] = dd.y ? 0.0f : __uint_as_float(wb.x & 0xFFFF0000u);
            w0[2] = dd.z ? 0.0f : __uint_as_float(wb.y << 16);
            w0[3] = dd.w ? 0.0f : __uint_as_float(wb.y & 0xFFFF0000u);
            const float4 pv = *reinterpret_cast<const float4 *>(P + base);
            p[0] = pv.x, p[1] = pv.y, p[2] = pv.z, p[3] = pv.w;
        }
        float w[4] = {w0[0], w0[1], w0[2], w0[3]};
        // w += p U_bb  (row a of Ub holds zeros left of its diagonal)
#pragma unroll 2
        for (int qa = 0; qa < nq; ++qa) {
#pragma unroll
            for (int ta = 0; ta < 4; ++ta) {
                const float pa = __shfl_sync(0xffffffffu, p[ta], qa);
                const float4 u = *reinterpret_cast<const float4 *>(Ub + (4 * qa + ta) * kObsBlock + 4 * lane);
                w[0] = fmaf(pa, u.x, w[0]);
                w[1] = fmaf(pa, u.y, w[1]);
                w[2] = fmaf(pa, u.z, w[2]);
                w[3] = fmaf(pa, u.w, w[3]);
            }
        }
        uint32_t kb = 0;  // this lane's keep bits (bit t = column 4 lane + t)
        uint32_t kq = 0;  // keep bits of the current quad, the same in every lane
#pragma unroll 1
        for (int q = 0; q < nq; ++q) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int j = 4 * q + t;
                if constexpr (M <= 4) {
                    // the group is this quad's lane: every lane ranks its own
                    // values, lane q's ranking is the one that counts
                    if (t % M == 0) {
                        uint32_t bits = 0;
#pragma unroll
                        for (int u = 0; u < M; ++u) {
                            const float su = w[t + u] * w[t + u] * dsq[(4 * lane + t + u) & (kObsBlock - 1)];
                            int rk = 0;
#pragma unroll
                            for (int u2 = 0; u2 < M; ++u2) {
                                const float so = w[t + u2] * w[t + u2] * dsq[(4 * lane + t + u2) & (kObsBlock - 1)];
                                rk += u2 != u && ((so > su) || (so == su && u2 < u));
                            }
                            bits |= rk < N ? 1u << (t + u) : 0u;
                        }
                        if (lane == q)
                            kb |= bits;
                        kq = __shfl_sync(0xffffffffu, kb, q);
                    }
                } else {
                    constexpr int G = M / 4;  // lanes per group
                    if (t == 0) {
                        if ((q & (G - 1)) == 0) {
                            float sc[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                sc[u] = w[u] * w[u] * dsq[(4 * lane + u) & (kObsBlock - 1)];
                            int rk[4] = {0, 0, 0, 0};
#pragma unroll
                            for (int m = 0; m < G; ++m)
#pragma unroll
                                for (int u2 = 0; u2 < 4; ++u2) {
                                    const float o = __shfl_sync(0xffffffffu, sc[u2], q + m);
                                    const int ocol = 4 * (q + m) + u2;
#pragma unroll
                                    for (int u = 0; u < 4; ++u)
                                        rk[u] += (o > sc[u]) || (o == sc[u] && ocol < 4 * lane + u);
                                }
                            if ((lane & ~(G - 1)) == q)
#pragma unroll
                                for (int u = 0; u < 4; ++u)
                                    kb |= rk[u] < N ? 1u << u : 0u;
                        }
                        kq = __shfl_sync(0xffffffffu, kb, q);
                    }
                }
                if (!((kq >> t) & 1u)) {
                    const float err = __shfl_sync(0xffffffffu, w[t], q) * rinv[j];
                    const float4 u = *reinterpret_cast<const float4 *>(Ub + j * kObsBlock + 4 * lane);
                    w[0] = fmaf(-err, u.x, w[0]);
                    w[1] = fmaf(-err, u.y, w[1]);
                    w[2] = fmaf(-err, u.z, w[2]);
                    w[3] = fmaf(-err, u.w, w[3]);
                    if (lane == q)
                        w[t] = 0.0f;
                }
            }
        }
        if (mine) {
            const uint32_t b01 = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(w[0])) |
                                 ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(w[1])) << 16);
            const uint32_t b23 = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(w[2])) |
                                 ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(w[3])) << 16);
            *reinterpret_cast<uint2 *>(Wout + base) = make_uint2(b01, b23);
            if (Wout_f32)
                *reinterpret_cast<float4 *>(Wout_f32 + base) = make_float4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<float4 *>(D + r * ldD + 4 * lane) =
                make_float4(w0[0] - w[0], w0[1] - w[1], w0[2] - w[2], w0[3] - w[3]);
        }
        if (masks) {
            // word g (block columns 32 g .. 32 g + 31): bit 4 i + t from lane 8 g + i, bit t
            const uint32_t k0 = __ballot_sync(0xffffffffu, kb & 1u), k1 = __ballot_sync(0xffffffffu, kb & 2u);
            const uint32_t k2 = __ballot_sync(0xffffffffu, kb & 4u), k3 = __ballot_sync(0xffffffffu, kb & 8u);
            if (lane < (bw >> 5)) {
                const int sh = 8 * lane;
                masks[r * (K / 32) + i1 / 32 + lane] = spread8(k0 >> sh) | (spread8(k1 >> sh) << 1) |
                                                       (spread8(k2 >> sh) << 2) | (spread8(k3 >> sh) << 3);
            }
        }
    }
}

constexpr size_t kSweepSmem = (size_t)kObsBlock * kObsBlock * 4 + 2 * kObsBlock * 4;

struct SweepArgs {
    const __nv_bfloat16 *W;
    const unsigned char *dead;
    const float *P, *X;
    int64_t rows, K;
    int N;
    float *D;
    int ldD;
    __nv_bfloat16 *Wout;
    float *Wout_f32;
    uint32_t *masks;
};

template <int M> cudaError_t launch_sweep(const SweepArgs &a, int i1, int bw, int grid, cudaStream_t st)
{
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(obs_sweep_kernel<M>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSweepSmem);
    });
    if (attr != cudaSuccess)
        return attr;
    return launch_pdl(obs_sweep_kernel<M>, dim3(grid), dim3(kSweepWarps * 32), kSweepSmem, st, a.W, a.dead, a.P, a.X,
                      a.rows, a.K, i1, bw, a.N, a.D, a.ldD, a.Wout, a.Wout_f32, a.masks);
}

cudaError_t sweep(int M, const SweepArgs &a, int i1, int bw, int grid, cudaStream_t st)
{
    switch (M) {
    case 2: return launch_sweep<2>(a, i1, bw, grid, st);
    case 4: return launch_sweep<4>(a, i1, bw, grid, st);
    case 8: return launch_sweep<8>(a, i1, bw, grid, st);
    case 16: return launch_sweep<16>(a, i1, bw, grid, st);
    default: return launch_sweep<32>(a, i1, bw, grid, st);
    }
}

// ---- host side ----------------------------------------------------------------

// Per device: the SM count and this library's workspace pool. The pool keeps
// what it has mapped between calls (release threshold: no limit): taking a
// workspace of several GB from a pool that returns memory at every
// synchronisation maps it afresh on every call. nm_obs_release_workspace
// trims it.
struct ObsDevice {
    int sms = 0;
    cudaMemPool_t pool = nullptr;
};

std::mutex g_obs_mu;  // held for the whole of each call
ObsDevice g_obs[kMaxDevices];

nm_status obs_device(ObsDevice **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return NM_ERR_CUDA;
    ObsDevice &d = g_obs[dev];
    if (!d.sms && cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return NM_ERR_CUDA;
    if (!d.pool) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        if (cudaMemPoolCreate(&p, &props) != cudaSuccess)
            return NM_ERR_CUDA;
        uint64_t keep = ~0ull;
        if (cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
            cudaMemPoolDestroy(p);
            return NM_ERR_CUDA;
        }
        d.pool = p;
    }
    *out = &d;
    return NM_OK;
}

int grid_for(int64_t n, int sms)
{
    int64_t g = (n + 255) / 256, cap = (int64_t)sms * 8;
    return (int)(g < 1 ? 1 : (g < cap ? g : cap));
}

// Stream-ordered workspace from the device's pool, released (to the pool) on
// every return path.
struct Workspace {
    cudaStream_t st;
    cudaMemPool_t pool;
    void *p = nullptr;
    Workspace(cudaStream_t s, cudaMemPool_t mp) : st(s), pool(mp) {}
    Workspace(const Workspace &) = delete;
    Workspace &operator=(const Workspace &) = delete;
    ~Workspace()
    {
        if (p)
            cudaFreeAsync(p, st);
    }
    bool alloc(size_t bytes)
    {
        if (cudaMallocFromPoolAsync(&p, bytes, pool, st) != cudaSuccess) {
            p = nullptr;
            return false;
        }
        return true;
    }
};

size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }

// Row-major fp32 GEMMs on K-strided buffers: on the tensor cores with fp32
// emulated by bf16 parts (wa, wb: the split operands' workspace), or plain
// fp32 on the CUDA cores -- always with NM_OBS_SGEMM, and for products of at
// most kSmallMax multiply-adds (up to 256^3: the leaves of the Cholesky
// recursion), where the small-shape kernel takes 6-10 us against 14-16 us
// for the operand split and the tensor-core launch.
constexpr int64_t kSmallMax = (int64_t)1 << 24;
struct RowGemm {
    bool plain;
    int64_t ld;
    uint16_t *wa, *wb;
    uint32_t *status;
    cudaStream_t st;
    // C (M x N) = alpha * A (M x k, stride lda) * op(B) + beta * C (stride ldc);
    // op(B) = B (k x N) when b_kn, else B^T (B is N x k); `tri`: the
    // structure flags of tc_gemm_f32 (zero or unread parts it may skip)
    bool gemm(int64_t M, int64_t N, int64_t k, float alpha, const float *A, int64_t lda, const float *B, int64_t ldb,
              bool b_kn, float beta, float *C, int64_t ldc, unsigned tri = 0) const
    {
        if (plain)
            return simt_gemm_f32(A, lda, B, ldb, b_kn, M, N, k, C, ldc, alpha, beta, st) == NM_OK;
        if (M * N * k <= kSmallMax)
            return simt_small_f32(A, lda, B, ldb, b_kn, M, N, k, C, ldc, alpha, beta, st) == NM_OK;
        return tc_gemm_f32(A, lda, false, B, ldb, b_kn, M, N, k, C, ldc, alpha, beta, wa, wb, status, st, tri) ==
               NM_OK;
    }
    // C (r x c) = alpha * A (r x k) * B (k x c) + beta * C
    bool ab(int64_t r, int64_t c, int64_t k, float alpha, const float *A, const float *B, float beta, float *C,
            unsigned tri = 0) const
    {
        return gemm(r, c, k, alpha, A, ld, B, ld, true, beta, C, ld, tri);
    }
    // C (r x c) = alpha * A (r x k) * B^T (B is c x k) + beta * C
    bool abt(int64_t r, int64_t c, int64_t k, float alpha, const float *A, const float *B, float beta, float *C,
             unsigned tri = 0) const
    {
        return gemm(r, c, k, alpha, A, ld, B, ld, false, beta, C, ld, tri);
    }
};

// Cholesky factorisation, by recursion on halves of the block range [b0, b1)
// (block b = columns [128 b, 128 b + 128)):
//   [[A11, .], [A21, A22]] = L L^T:
//     L11 and X11 = L11^-1 from A11;  L21 = A21 X11^T;  A22 -= L21 L21^T;
//     L22 from A22;  and, if need_x, X21 = -X22 L21 X11 so that X = L^-1 in full.
// The left half is always inverted in full (its inverse makes L21); below the
// top call only nodes whose own inverse some L21 needs invert in full. A
// single block is fac_diag_kernel, which also writes X_kk = L_kk^-1: the
// diagonal blocks of X are always complete. A (J H J, damped) is destroyed; L
// receives every block below the diagonal (its diagonal blocks are not
// written); X's upper part must be zero on entry. L21 X11 is kept in A's A21
// region, which is no longer read once L21 exists.
bool chol_inv(const RowGemm &G, float *A, float *L, float *X, int64_t K, int64_t b0, int64_t b1, bool need_x,
              int *not_pd, cudaStream_t st)
{
    if (b1 - b0 == 1) {
        const int64_t k0 = b0 * kFacB;
        const int kb = (int)(K - k0 < kFacB ? K - k0 : kFacB);
        static std::once_flag once;
        static cudaError_t attr = cudaSuccess;
        std::call_once(once, [] {
            attr = cudaFuncSetAttribute(fac_diag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFacSmem);
        });
        if (attr != cudaSuccess)
            return false;
        return launch_pdl(fac_diag_kernel, dim3(1), dim3(kFacThreads), kFacSmem, st, (const float *)A, X, K, k0, kb,
                          not_pd) == cudaSuccess;
    }
    const int64_t bm = (b0 + b1) / 2;
    const int64_t lo = b0 * kFacB, mid = bm * kFacB, hi = (b1 * kFacB < K ? b1 * kFacB : K);
    const int64_t h1 = mid - lo, h2 = hi - mid;
    float *A21 = A + mid * K + lo, *L21 = L + mid * K + lo;
    float *X11 = X + lo * K + lo, *X22 = X + mid * K + mid;
    // X11 and X22 are lower triangular, and nothing reads A22 above its
    // diagonal: the GEMMs skip those zeros and that triangle
    if (!chol_inv(G, A, L, X, K, b0, bm, true, not_pd, st) ||
        !G.abt(h2, h1, h1, 1.0f, A21, X11, 0.0f, L21, kTcBLower) ||
        !G.abt(h2, h2, h1, -1.0f, L21, L21, 1.0f, A + mid * K + mid, kTcCLower) ||
        !chol_inv(G, A, L, X, K, bm, b1, need_x, not_pd, st))
        return false;
    if (!need_x)
        return true;
    return G.ab(h2, h1, h1, 1.0f, L21, X11, 0.0f, A21, kTcBUpper) &&
           G.ab(h2, h1, h2, -1.0f, X22, A21, 0.0f, X + mid * K + lo, kTcALower);
}

// The sweep's blocks in column order: the factorisation's blocks reversed, so
// a block narrower than 128 (K % 128 != 0) comes first.
int64_t sweep_bound(int64_t b, int64_t nb, int64_t K)
{
    const int64_t first = K - (int64_t)kObsBlock * (nb - 1);
    return b == 0 ? 0 : (b >= nb ? K : first + (int64_t)kObsBlock * (b - 1));
}

nm_status obs_prune_impl(const void *W, const float *H, int64_t rows, int64_t K, int N, int M, float percdamp,
                         unsigned flags, void *Wout, uint32_t *masks, float *Wout_f32, cudaStream_t st)
{
    ObsDevice *d = nullptr;
    nm_status s = obs_device(&d);
    if (s != NM_OK)
        return s;
    const bool plain = (flags & NM_OBS_SGEMM) != 0;
    const int64_t nb = (K + kFacB - 1) / kFacB;

    // buffers: dead flags, lam, the not-PD flag and the GEMMs' status word,
    // three K x K matrices (A, later R; L; X), D of one superblock, the
    // accumulator P, and the bf16 parts of the two operands of one GEMM (none
    // for plain fp32). The recursion's operands are at most Kh x Kh; the lazy
    // update's are D (rows x superblock) and a part of R (K x superblock).
    const int64_t Kh = ((nb + 1) / 2) * kFacB < K ? ((nb + 1) / 2) * kFacB : K;
    const size_t wa_bytes = plain ? 0 : std::max(tc_operand_bytes(Kh, Kh, true), tc_operand_bytes(rows, kSuper, true));
    const size_t wb_bytes = plain ? 0 : std::max(tc_operand_bytes(Kh, Kh, true), tc_operand_bytes(K, kSuper, true));
    const size_t kk = (size_t)K * K * 4;
    const size_t off_lam = round256((size_t)K), off_flag = off_lam + 256, off_A = off_flag + 256;
    const size_t off_L = off_A + round256(kk), off_X = off_L + round256(kk), off_D = off_X + round256(kk);
    const size_t off_P = off_D + round256((size_t)rows * kSuper * 4);
    const size_t off_WA = off_P + round256((size_t)rows * K * 4), off_WB = off_WA + round256(wa_bytes);
    const size_t total = off_WB + round256(wb_bytes);
    Workspace ws(st, d->pool);
    if (!ws.alloc(total))
        return NM_ERR_CUDA;
    char *base = (char *)ws.p;
    unsigned char *dead = (unsigned char *)base;
    float *lam = (float *)(base + off_lam);
    int *not_pd = (int *)(base + off_flag);
    uint32_t *gemm_status = (uint32_t *)(base + off_flag + 16);
    float *A = (float *)(base + off_A), *L = (float *)(base + off_L), *X = (float *)(base + off_X);
    float *Dbuf = (float *)(base + off_D), *P = (float *)(base + off_P);
    float *R = A;  // R replaces A once the factorisation is done
    const RowGemm G{plain, K, (uint16_t *)(base + off_WA), (uint16_t *)(base + off_WB), gemm_status, st};

    if (cudaMemsetAsync(base + off_flag, 0, 256, st) != cudaSuccess || cudaMemsetAsync(X, 0, kk, st) != cudaSuccess ||
        cudaMemsetAsync(P, 0, (size_t)rows * K * 4, st) != cudaSuccess)
        return NM_ERR_CUDA;
    if (launch_pdl(obs_diag_kernel, dim3(1), dim3(1024), 0, st, H, K, percdamp, dead, lam) != cudaSuccess ||
        launch_pdl(obs_reverse_damp_kernel, dim3(grid_for(K * K, d->sms)), dim3(256), 0, st, H, K, (const float *)lam,
                   A) != cudaSuccess)
        return NM_ERR_CUDA;
    if (!chol_inv(G, A, L, X, K, 0, nb, false, not_pd, st))
        return NM_ERR_CUDA;
    // A pivot that is not positive was replaced by 1, so the rest runs on
    // finite values; the flag is read once everything is queued.
    if (launch_pdl(obs_reverse_kernel, dim3(grid_for(K * K, d->sms)), dim3(256), 0, st, (const float *)L, K * K,
                   R) != cudaSuccess)
        return NM_ERR_CUDA;

    // Sweep the blocks left to right. A block starts from W0 + P U_bb, where P
    // accumulates D R over the finished blocks (D = W0 - final values): with
    // E the errors, W0 - final = E U and U = R^-1, so E = D R, and the
    // corrections the finished blocks owe block b, sum E_c U_cb, equal
    // -(D R)_b U_bb. P is updated lazily in two levels: after each block the
    // rest of its superblock (k = block width), after each superblock every
    // later column (k = superblock width).
    const int64_t want = (rows + kSweepWarps - 1) / kSweepWarps, cap = (int64_t)d->sms * 2;
    const int sweep_grid = (int)(want < cap ? want : cap);
    const SweepArgs sa{(const __nv_bfloat16 *)W, dead, P, X, rows, K, N, Dbuf, kSuper, (__nv_bfloat16 *)Wout,
                       Wout_f32, masks};
    auto update = [&](int64_t c0, int64_t c1, int64_t k0, int64_t kw, const float *Dk) {
        // P[:, c0:c1] += D[:, k0 ...] R[k0:k0+kw, c0:c1]   (D rows have stride kSuper)
        return G.gemm(rows, c1 - c0, kw, 1.0f, Dk, kSuper, R + k0 * K + c0, K, true, 1.0f, P + c0, K);
    };
    constexpr int64_t kPerSuper = kSuper / kObsBlock;
    for (int64_t sb = 0; sb < nb; sb += kPerSuper) {
        const int64_t s1 = sweep_bound(sb, nb, K), s2 = sweep_bound(sb + kPerSuper, nb, K);
        for (int64_t b = sb; b < sb + kPerSuper && b < nb; ++b) {
            const int64_t i1 = sweep_bound(b, nb, K), i2 = sweep_bound(b + 1, nb, K);
            SweepArgs a = sa;
            a.D = Dbuf + (i1 - s1);
            if (sweep(M, a, (int)i1, (int)(i2 - i1), sweep_grid, st) != cudaSuccess)
                return NM_ERR_CUDA;
            if (i2 < s2 && !update(i2, s2, i1, i2 - i1, Dbuf + (i1 - s1)))
                return NM_ERR_CUDA;
        }
        if (s2 < K && !update(s2, K, s1, s2 - s1, Dbuf))
            return NM_ERR_CUDA;
    }
    int host_flag[5] = {0, 0, 0, 0, 0}; // not-PD flag, then (16 bytes on) the GEMMs' status word
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyAsync(host_flag, not_pd, sizeof host_flag, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return NM_ERR_CUDA;
    if (host_flag[4] & (1 << NM_ERR_TIMEOUT))
        return NM_ERR_TIMEOUT;
    return host_flag[0] ? NM_ERR_NOT_PD : NM_OK;
}

}  // namespace
}  // namespace nm

using namespace nm;

extern "C" nm_status nm_obs_hessian(const void *X_bf16, int64_t T, int64_t K, float *H, int accumulate, void *stream)
{
    if (T < 0 || K < 0 || K % 32 != 0 || T > INT32_MAX || K > INT32_MAX)
        return NM_ERR_SHAPE;
    if (K == 0)
        return NM_OK;
    if (!H || (T > 0 && !X_bf16))
        return NM_ERR_INVALID_ARG;
    if (!aligned16(H) || (T > 0 && !aligned16(X_bf16)))
        return NM_ERR_ALIGN;
    cudaStream_t st = (cudaStream_t)stream;
    if (T == 0)
        return accumulate ? NM_OK
                          : (cudaMemsetAsync(H, 0, (size_t)K * K * 4, st) == cudaSuccess ? NM_OK : NM_ERR_CUDA);
    std::lock_guard<std::mutex> lock(g_obs_mu);
    // H[i][j] = 2 sum_t X[t][i] X[t][j]: X^T (bf16 [K][Tp], t contiguous, zero
    // padding to a multiple of 64 tokens) is both operands of one bf16 pass;
    // the products are exact and the sums fp32. H is symmetric: the tiles on
    // and below the diagonal are computed and mirrored. A bounded wait that
    // runs out is reported by nm_device_status.
    uint32_t *status = nullptr;
    nm_status s = library_status_word(&status);
    if (s != NM_OK)
        return s;
    ObsDevice *d = nullptr;
    if ((s = obs_device(&d)) != NM_OK)
        return s;
    const int64_t Tp = (T + 63) / 64 * 64;
    Workspace ws(st, d->pool);
    if (!ws.alloc((size_t)K * Tp * 2))
        return NM_ERR_CUDA;
    uint16_t *Xt = (uint16_t *)ws.p;
    if ((s = tc_transpose_bf16((const uint16_t *)X_bf16, T, K, Xt, Tp, st)) != NM_OK)
        return s;
    return tc_gemm_bf16(Xt, Xt, Tp / 64, 1, H, K, K, K, 2.0f, accumulate ? 1.0f : 0.0f, status, st, kTcCSym);
}

extern "C" nm_status nm_obs_prune(const void *W_bf16, const float *H, int64_t rows, int64_t K, int N, int M,
                                  float percdamp, unsigned flags, void *W_out_bf16, uint32_t *keep_masks,
                                  float *W_out_f32, void *stream)
{
    if (rows < 0 || K < 0 || K % 32 != 0 || rows > INT32_MAX || K > INT32_MAX)
        return NM_ERR_SHAPE;
    if ((M != 2 && M != 4 && M != 8 && M != 16 && M != 32) || N < 1 || N > M)
        return NM_ERR_UNSUPPORTED;
    if (!(percdamp >= 0.0f && percdamp <= 1e30f) || (flags & ~(unsigned)NM_OBS_SGEMM))
        return NM_ERR_INVALID_ARG;
    if (rows == 0 || K == 0)
        return NM_OK;
    if (!W_bf16 || !H || !W_out_bf16)
        return NM_ERR_INVALID_ARG;
    if (!aligned16(W_bf16) || !aligned16(H) || !aligned16(W_out_bf16) || (keep_masks && !aligned16(keep_masks)) ||
        (W_out_f32 && !aligned16(W_out_f32)))
        return NM_ERR_ALIGN;
    cudaStream_t st = (cudaStream_t)stream;
    std::lock_guard<std::mutex> lock(g_obs_mu);
    nm_status s = obs_prune_impl(W_bf16, H, rows, K, N, M, percdamp, flags, W_out_bf16, keep_masks, W_out_f32, st);
    cudaError_t e = cudaStreamSynchronize(st);
    return s != NM_OK ? s : (e == cudaSuccess ? NM_OK : NM_ERR_CUDA);
}

extern "C" nm_status nm_obs_release_workspace(void)
{
    std::lock_guard<std::mutex> lock(g_obs_mu);
    ObsDevice *d = nullptr;
    nm_status s = obs_device(&d);
    if (s != NM_OK)
        return s;
    return cudaMemPoolTrimTo(d->pool, 0) == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}
