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
// J H J = L L^T (Cholesky), then U = J L^-1 J. That is one potrf and one
// trtri, and inv(H) itself is never formed.
//
// Steps of nm_obs_prune, all on the caller's stream:
//   1. obs_diag_kernel: dead columns (H_jj == 0) and the damping
//      lam = percdamp * mean(diag H with dead entries set to 1);
//   2. obs_reverse_damp_kernel: J (H + lam I) J, dead diagonal entries = 1 + lam;
//   3. cuSOLVER potrf (lower) and trtri (lower) on it: L^-1, column-major;
//   4. obs_factor_kernel: U = J L^-1 J written row-major, zeros below the diagonal;
//   5. obs_init_w_kernel: fp32 working copy of W, dead columns zeroed;
//   6. per block of 128 columns [i1, i2):
//        obs_sweep_kernel: one warp per row walks the block column by
//          column (N:M choice, in-block compensation), writes the final
//          values of the block, its keep bits, and the error row
//          E[r][c] = w_c / U_cc (0 where kept);
//        lazy trailing update W[:, i2:] -= E U[i1:i2, i2:] (cuBLAS GEMM; by
//          default fp32 emulated on the bf16 tensor cores, 3 bf16 terms per
//          operand, otherwise plain fp32).
// The blocked order only regroups the same updates: a column receives every
// earlier column's correction before it is read.
#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cusolverDn.h>

#include <mutex>
#include <vector>

#include "nmspmv.h"

namespace nm {
namespace {

constexpr int kObsBlock = 128;   // columns per sweep block
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
    const int64_t n = K * K;
    const float l = *lam;
    for (int64_t p = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; p < n; p += (int64_t)gridDim.x * blockDim.x) {
        float h = H[n - 1 - p];
        if (p / K == p % K)
            h = (h == 0.0f ? 1.0f : h) + l;
        Hr[p] = h;
    }
}

// ---- step 4: U = J L^-1 J, row-major ---------------------------------------

// Linv: column-major, lower triangle valid (element (a, b) at a + b K, a >= b).
// U(i, j) = Linv(K-1-i, K-1-j) = Linv[K*K - 1 - (i + j K)] for j >= i, else 0.
// A 32 x 32 tile goes through shared memory so that both sides are coalesced:
// for a fixed j the source is contiguous in i.
__global__ void __launch_bounds__(256) obs_factor_kernel(const float *__restrict__ Linv, int64_t K,
                                                         float *__restrict__ U)
{
    __shared__ float t[32][33];
    const int64_t n = K * K;
    const int64_t i0 = (int64_t)blockIdx.y * 32, j0 = (int64_t)blockIdx.x * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8 threads
    for (int r = ty; r < 32; r += 8) {  // r: j offset, tx: i offset
        int64_t i = i0 + tx, j = j0 + r;
        t[r][tx] = (i < K && j < K && j >= i) ? Linv[n - 1 - (i + j * K)] : 0.0f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {  // r: i offset, tx: j offset
        int64_t i = i0 + r, j = j0 + tx;
        if (i < K && j < K)
            U[i * K + j] = t[tx][r];
    }
}

// ---- step 5: fp32 working copy ----------------------------------------------

__global__ void obs_init_w_kernel(const __nv_bfloat16 *__restrict__ W, int64_t rows, int64_t K,
                                  const unsigned char *__restrict__ dead, float *__restrict__ Wf)
{
    const int64_t n = rows * K;
    for (int64_t p = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; p < n; p += (int64_t)gridDim.x * blockDim.x)
        Wf[p] = dead[p % K] ? 0.0f : __bfloat162float(W[p]);
}

// ---- step 6a: the column sweep of one block ----------------------------------

// Shared memory: Ub[a][b] = U[i1 + a][i1 + b] for a, b < bw (zeros below the
// diagonal and outside the block) and rinv[a] = 1 / Ub[a][a].
// Warp w of CTA c takes rows c * 16 + w, then steps by the grid. Lane l holds
// columns i1 + 32 s + l (s = 0..3) in w[s]. A kept column moves nothing, so
// only removed columns run the update; the below-diagonal zeros of Ub leave
// the already final columns of the slot unchanged.
template <int M>
__global__ void __launch_bounds__(kSweepWarps * 32) obs_sweep_kernel(
    float *__restrict__ Wf, const float *__restrict__ U, int64_t rows, int64_t K, int i1, int bw, int N,
    float *__restrict__ E, __nv_bfloat16 *__restrict__ Wout, uint32_t *__restrict__ masks)
{
    extern __shared__ float4 smem4[];
    float *Ub = reinterpret_cast<float *>(smem4);
    float *rinv = Ub + kObsBlock * kObsBlock;
    constexpr int kQuads = kObsBlock / 4;
    for (int q = threadIdx.x; q < kObsBlock * kQuads; q += blockDim.x) {
        const int a = q / kQuads, b = (q % kQuads) * 4;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (a < bw && b < bw)
            v = *reinterpret_cast<const float4 *>(U + (int64_t)(i1 + a) * K + i1 + b);
        smem4[q] = v;
    }
    __syncthreads();
    for (int a = threadIdx.x; a < kObsBlock; a += blockDim.x)
        rinv[a] = a < bw ? 1.0f / Ub[a * kObsBlock + a] : 0.0f;
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ns = bw >> 5;
    for (int64_t r = (int64_t)blockIdx.x * kSweepWarps + warp; r < rows; r += (int64_t)gridDim.x * kSweepWarps) {
        float *wrow = Wf + r * K + i1;
        float w[4], e[4];
        uint32_t keep[4];
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            w[s] = s < ns ? wrow[32 * s + lane] : 0.0f;
            e[s] = 0.0f;
            keep[s] = 0u;
        }
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            if (s >= ns)
                break;
#pragma unroll 1
            for (int l = 0; l < 32; ++l) {
                const int i = 32 * s + l;
                if ((l & (M - 1)) == 0) {
                    // N:M choice for the group starting at column i, from the
                    // current values: rank by saliency w^2 / U_cc^2, equal
                    // saliencies ranked by column.
                    const float d = Ub[(32 * s + lane) * kObsBlock + 32 * s + lane];
                    const float sc = w[s] * w[s] / (d * d);
                    const int base = lane & ~(M - 1);
                    int rank = 0;
#pragma unroll
                    for (int t = 0; t < M; ++t) {
                        const float o = __shfl_sync(0xffffffffu, sc, base + t);
                        rank += (o > sc) || (o == sc && base + t < lane);
                    }
                    keep[s] |= __ballot_sync(0xffffffffu, base == l && rank < N);
                }
                if (!((keep[s] >> l) & 1u)) {
                    const float err = __shfl_sync(0xffffffffu, w[s], l) * rinv[i];
                    const float *urow = Ub + i * kObsBlock;
#pragma unroll
                    for (int s2 = s; s2 < 4; ++s2)
                        w[s2] = fmaf(-err, urow[32 * s2 + lane], w[s2]);
                    if (lane == l) {
                        w[s] = 0.0f;
                        e[s] = err;
                    }
                }
            }
        }
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            if (s >= ns)
                break;
            wrow[32 * s + lane] = w[s];
            Wout[r * K + i1 + 32 * s + lane] = __float2bfloat16_rn(w[s]);
            E[r * kObsBlock + 32 * s + lane] = e[s];
            if (masks && lane == 0)
                masks[r * (K / 32) + i1 / 32 + s] = keep[s];
        }
    }
}

constexpr size_t kSweepSmem = (size_t)kObsBlock * kObsBlock * 4 + kObsBlock * 4;

template <int M>
cudaError_t launch_sweep(float *Wf, const float *U, int64_t rows, int64_t K, int i1, int bw, int N, float *E,
                         __nv_bfloat16 *Wout, uint32_t *masks, int grid, cudaStream_t st)
{
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(obs_sweep_kernel<M>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSweepSmem);
    });
    if (attr != cudaSuccess)
        return attr;
    obs_sweep_kernel<M><<<grid, kSweepWarps * 32, kSweepSmem, st>>>(Wf, U, rows, K, i1, bw, N, E, Wout, masks);
    return cudaGetLastError();
}

cudaError_t sweep(int M, float *Wf, const float *U, int64_t rows, int64_t K, int i1, int bw, int N, float *E,
                  __nv_bfloat16 *Wout, uint32_t *masks, int grid, cudaStream_t st)
{
    switch (M) {
    case 2: return launch_sweep<2>(Wf, U, rows, K, i1, bw, N, E, Wout, masks, grid, st);
    case 4: return launch_sweep<4>(Wf, U, rows, K, i1, bw, N, E, Wout, masks, grid, st);
    case 8: return launch_sweep<8>(Wf, U, rows, K, i1, bw, N, E, Wout, masks, grid, st);
    case 16: return launch_sweep<16>(Wf, U, rows, K, i1, bw, N, E, Wout, masks, grid, st);
    default: return launch_sweep<32>(Wf, U, rows, K, i1, bw, N, E, Wout, masks, grid, st);
    }
}

// ---- host side ----------------------------------------------------------------

struct ObsDevice {
    cublasHandle_t blas = nullptr;
    cusolverDnHandle_t solver = nullptr;
    int sms = 0;
};

std::mutex g_obs_mu;  // held for the whole of each call (the handles are shared)
ObsDevice g_obs[kMaxDevices];

nm_status obs_device(ObsDevice **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return NM_ERR_CUDA;
    ObsDevice &d = g_obs[dev];
    if (!d.sms && cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return NM_ERR_CUDA;
    if (!d.blas && cublasCreate(&d.blas) != CUBLAS_STATUS_SUCCESS) {
        d.blas = nullptr;
        return NM_ERR_CUDA;
    }
    if (!d.solver && cusolverDnCreate(&d.solver) != CUSOLVER_STATUS_SUCCESS) {
        d.solver = nullptr;
        return NM_ERR_CUDA;
    }
    *out = &d;
    return NM_OK;
}

int grid_for(int64_t n, int sms)
{
    int64_t g = (n + 255) / 256, cap = (int64_t)sms * 8;
    return (int)(g < 1 ? 1 : (g < cap ? g : cap));
}

// Stream-ordered workspace, released on every return path.
struct Workspace {
    cudaStream_t st;
    void *p = nullptr;
    explicit Workspace(cudaStream_t s) : st(s) {}
    Workspace(const Workspace &) = delete;
    Workspace &operator=(const Workspace &) = delete;
    ~Workspace()
    {
        if (p)
            cudaFreeAsync(p, st);
    }
    bool alloc(size_t bytes)
    {
        if (cudaMallocAsync(&p, bytes, st) != cudaSuccess) {
            p = nullptr;
            return false;
        }
        return true;
    }
};

size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }

nm_status obs_prune_impl(const void *W, const float *H, int64_t rows, int64_t K, int N, int M, float percdamp,
                         unsigned flags, void *Wout, uint32_t *masks, float *Wout_f32, cudaStream_t st)
{
    ObsDevice *d = nullptr;
    nm_status s = obs_device(&d);
    if (s != NM_OK)
        return s;
    if (cublasSetStream(d->blas, st) != CUBLAS_STATUS_SUCCESS ||
        cusolverDnSetStream(d->solver, st) != CUSOLVER_STATUS_SUCCESS)
        return NM_ERR_CUDA;

    // buffers: dead flags, lam, solver info, the factor (in place), U, E, the fp32 working copy
    const size_t kk = (size_t)K * K * 4;
    const size_t off_lam = round256((size_t)K), off_info = off_lam + 256, off_L = off_info + 256;
    const size_t off_U = off_L + round256(kk), off_E = off_U + round256(kk);
    const size_t off_Wf = off_E + round256((size_t)rows * kObsBlock * 4);
    const size_t total = off_Wf + (Wout_f32 ? 0 : round256((size_t)rows * K * 4));
    Workspace ws(st), solver_ws(st);
    if (!ws.alloc(total))
        return NM_ERR_CUDA;
    char *base = (char *)ws.p;
    unsigned char *dead = (unsigned char *)base;
    float *lam = (float *)(base + off_lam);
    int *info = (int *)(base + off_info);
    float *L = (float *)(base + off_L), *U = (float *)(base + off_U), *E = (float *)(base + off_E);
    float *Wf = Wout_f32 ? Wout_f32 : (float *)(base + off_Wf);

    const int n = (int)K;
    int lwork = 0;
    size_t trtri_dev = 0, trtri_host = 0;
    if (cusolverDnSpotrf_bufferSize(d->solver, CUBLAS_FILL_MODE_LOWER, n, L, n, &lwork) != CUSOLVER_STATUS_SUCCESS ||
        cusolverDnXtrtri_bufferSize(d->solver, CUBLAS_FILL_MODE_LOWER, CUBLAS_DIAG_NON_UNIT, K, CUDA_R_32F, L, K,
                                    &trtri_dev, &trtri_host) != CUSOLVER_STATUS_SUCCESS)
        return NM_ERR_CUDA;
    const size_t off_tw = round256((size_t)lwork * 4);
    if (!solver_ws.alloc(off_tw + round256(trtri_dev) + 256))
        return NM_ERR_CUDA;
    float *pw = (float *)solver_ws.p;
    void *tw = (char *)solver_ws.p + off_tw;
    std::vector<char> host_work(trtri_host ? trtri_host : 1);

    if (cudaMemsetAsync(info, 0, 2 * sizeof(int), st) != cudaSuccess)
        return NM_ERR_CUDA;
    obs_diag_kernel<<<1, 1024, 0, st>>>(H, K, percdamp, dead, lam);
    obs_reverse_damp_kernel<<<grid_for(K * K, d->sms), 256, 0, st>>>(H, K, lam, L);
    if (cudaGetLastError() != cudaSuccess)
        return NM_ERR_CUDA;
    if (cusolverDnSpotrf(d->solver, CUBLAS_FILL_MODE_LOWER, n, L, n, pw, lwork, info) != CUSOLVER_STATUS_SUCCESS ||
        cusolverDnXtrtri(d->solver, CUBLAS_FILL_MODE_LOWER, CUBLAS_DIAG_NON_UNIT, K, CUDA_R_32F, L, K, tw, trtri_dev,
                         host_work.data(), trtri_host, info + 1) != CUSOLVER_STATUS_SUCCESS)
        return NM_ERR_CUDA;
    int hinfo[2] = {0, 0};
    if (cudaMemcpyAsync(hinfo, info, sizeof(hinfo), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return NM_ERR_CUDA;
    if (hinfo[0] != 0 || hinfo[1] != 0)
        return NM_ERR_NOT_PD;

    const dim3 tiles((unsigned)((K + 31) / 32), (unsigned)((K + 31) / 32));
    obs_factor_kernel<<<tiles, 256, 0, st>>>(L, K, U);
    obs_init_w_kernel<<<grid_for(rows * K, d->sms), 256, 0, st>>>((const __nv_bfloat16 *)W, rows, K, dead, Wf);
    if (cudaGetLastError() != cudaSuccess)
        return NM_ERR_CUDA;

    const int64_t want = (rows + kSweepWarps - 1) / kSweepWarps, cap = (int64_t)d->sms * 3;
    const int sweep_grid = (int)(want < cap ? want : cap);
    const cublasComputeType_t ct =
        (flags & NM_OBS_SGEMM) ? CUBLAS_COMPUTE_32F : CUBLAS_COMPUTE_32F_EMULATED_16BFX9;
    const float alpha = -1.0f, beta = 1.0f;
    for (int64_t i1 = 0; i1 < K; i1 += kObsBlock) {
        const int bw = (int)(K - i1 < kObsBlock ? K - i1 : kObsBlock);
        const int64_t i2 = i1 + bw;
        if (sweep(M, Wf, U, rows, K, (int)i1, bw, N, E, (__nv_bfloat16 *)Wout, masks, sweep_grid, st) !=
            cudaSuccess)
            return NM_ERR_CUDA;
        if (i2 < K) {
            // column-major view: (W[:, i2:])^T -= (U[i1:i2, i2:])^T E^T
            if (cublasGemmEx(d->blas, CUBLAS_OP_N, CUBLAS_OP_N, (int)(K - i2), (int)rows, bw, &alpha,
                             U + i1 * K + i2, CUDA_R_32F, n, E, CUDA_R_32F, kObsBlock, &beta, Wf + i2, CUDA_R_32F, n,
                             ct, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
                return NM_ERR_CUDA;
        }
    }
    return cudaGetLastError() == cudaSuccess ? NM_OK : NM_ERR_CUDA;
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
    ObsDevice *d = nullptr;
    nm_status s = obs_device(&d);
    if (s != NM_OK)
        return s;
    if (cublasSetStream(d->blas, st) != CUBLAS_STATUS_SUCCESS)
        return NM_ERR_CUDA;
    // column-major view: X is K x T (ld K); H = 2 X X^T is K x K
    const float alpha = 2.0f, beta = accumulate ? 1.0f : 0.0f;
    if (cublasGemmEx(d->blas, CUBLAS_OP_N, CUBLAS_OP_T, (int)K, (int)K, (int)T, &alpha, X_bf16, CUDA_R_16BF, (int)K,
                     X_bf16, CUDA_R_16BF, (int)K, &beta, H, CUDA_R_32F, (int)K, CUBLAS_COMPUTE_32F,
                     CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
        return NM_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? NM_OK : NM_ERR_CUDA;
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
