// gemv.cu -- dense bf16 GEMV, the same-GPU dense reference for the sparse path
// (the pages' 1.00x rows: aitest123.com article, Table 3).
//
// y[b][r] = sum_j W[r][j] x[b][j], fp32 accumulation. One warp per row: lane l
// streams 16-byte chunks l, l+32, ... of the row with L1-bypassing loads (8
// chunks in flight per lane), x comes through the read-only cache, and a
// butterfly shuffle sums the 32 lane partials. Each CTA owns a contiguous
// range of rows, so all SMs get the same number of weight bytes.
#include <algorithm>

#include "kernels.h"

namespace nm {

constexpr int kGemvWarps = 16;
constexpr int kGemvUnroll = 8;

template <int B, bool F32OUT>
__global__ void __launch_bounds__(kGemvWarps * 32)
    gemv_kernel(const uint16_t *__restrict__ W, const uint16_t *__restrict__ x, void *y, int64_t rows,
                int64_t K)
{
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t r0 = rows * blockIdx.x / gridDim.x;
    const int64_t r1 = rows * (blockIdx.x + 1) / gridDim.x;
    const int64_t chunks = K / 8; // 16-byte chunks per row
    bool waited = false;
    for (int64_t row = r0 + warp; row < r1; row += kGemvWarps) {
        const uint16_t *wr = W + row * K;
        float acc[B];
#pragma unroll
        for (int b = 0; b < B; ++b)
            acc[b] = 0.f;
        for (int64_t c0 = 0; c0 < chunks; c0 += 32 * kGemvUnroll) {
            uint4 wv[kGemvUnroll];
#pragma unroll
            for (int u = 0; u < kGemvUnroll; ++u) {
                const int64_t c = c0 + lane + 32 * u;
                wv[u] = c < chunks ? ldg_stream128(wr + 8 * c) : make_uint4(0, 0, 0, 0);
            }
            if (!waited) { // x may be the previous kernel's output; weights are not
                pdl_wait_upstream();
                waited = true;
            }
#pragma unroll
            for (int u = 0; u < kGemvUnroll; ++u) {
                const int64_t c = c0 + lane + 32 * u;
                if (c < chunks) {
                    const float w[8] = {bf16lo_to_f32(wv[u].x), bf16hi_to_f32(wv[u].x), bf16lo_to_f32(wv[u].y),
                                        bf16hi_to_f32(wv[u].y), bf16lo_to_f32(wv[u].z), bf16hi_to_f32(wv[u].z),
                                        bf16lo_to_f32(wv[u].w), bf16hi_to_f32(wv[u].w)};
#pragma unroll
                    for (int b = 0; b < B; ++b) {
                        const uint4 xv = __ldg((const uint4 *)(x + (int64_t)b * K + 8 * c));
                        const float xs[8] = {bf16lo_to_f32(xv.x), bf16hi_to_f32(xv.x), bf16lo_to_f32(xv.y),
                                             bf16hi_to_f32(xv.y), bf16lo_to_f32(xv.z), bf16hi_to_f32(xv.z),
                                             bf16lo_to_f32(xv.w), bf16hi_to_f32(xv.w)};
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            acc[b] = fmaf(w[e], xs[e], acc[b]);
                    }
                }
            }
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                acc[b] += __shfl_xor_sync(0xFFFFFFFFu, acc[b], off);
        }
        if (lane == 0) {
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if (F32OUT)
                    ((float *)y)[(int64_t)b * rows + row] = acc[b];
                else
                    ((uint16_t *)y)[(int64_t)b * rows + row] = f32_to_bf16_rn(acc[b]);
            }
        }
    }
    if (!waited)
        pdl_wait_upstream();
    pdl_launch_dependents();
}

template <int B, bool F32OUT>
static nm_status launch_gemv_b(const void *W, const void *x, void *y, int64_t rows, int64_t K,
                               const LaunchCtx &ctx)
{
    const int64_t per_sm = 1;
    const int64_t blocks =
        std::max<int64_t>(1, std::min<int64_t>((int64_t)ctx.num_sms * per_sm, (rows + kGemvWarps - 1) / kGemvWarps));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kGemvWarps * 32);
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = ctx.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gemv_kernel<B, F32OUT>, (const uint16_t *)W, (const uint16_t *)x, y, rows, K) !=
        cudaSuccess)
        return NM_ERR_CUDA;
    return NM_OK;
}

template <bool F32OUT>
static nm_status gemv_dispatch(const void *W, const void *x, void *y, int64_t rows, int64_t K, int batch,
                               const LaunchCtx &ctx)
{
    switch (batch) {
    case 1: return launch_gemv_b<1, F32OUT>(W, x, y, rows, K, ctx);
    case 2: return launch_gemv_b<2, F32OUT>(W, x, y, rows, K, ctx);
    case 3: return launch_gemv_b<3, F32OUT>(W, x, y, rows, K, ctx);
    case 4: return launch_gemv_b<4, F32OUT>(W, x, y, rows, K, ctx);
    case 5: return launch_gemv_b<5, F32OUT>(W, x, y, rows, K, ctx);
    case 6: return launch_gemv_b<6, F32OUT>(W, x, y, rows, K, ctx);
    case 7: return launch_gemv_b<7, F32OUT>(W, x, y, rows, K, ctx);
    case 8: return launch_gemv_b<8, F32OUT>(W, x, y, rows, K, ctx);
    default: return NM_ERR_UNSUPPORTED;
    }
}

nm_status launch_gemv(const void *W, const void *x, void *y, bool f32out, int64_t rows, int64_t K, int batch,
                      const LaunchCtx &ctx)
{
    return f32out ? gemv_dispatch<true>(W, x, y, rows, K, batch, ctx)
                  : gemv_dispatch<false>(W, x, y, rows, K, batch, ctx);
}

} // namespace nm
