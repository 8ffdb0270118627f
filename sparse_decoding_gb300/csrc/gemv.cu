// gemv.cu -- dense bf16 GEMV, the same-GPU dense reference for the sparse path
// (the pages' 1.00x rows: aitest123.com article, Table 3).
//
// y[b][r] = sum_j W[r][j] x[b][j], fp32 accumulation.
//
// Main kernel (K % 64 == 0): the same stream-K TMA driver as the sparse
// kernel (streamk.cuh), with units of 32 rows x 64 columns (4 KB of W, the
// same bytes per unit as the sparse kernel's values). Lane i owns row i of the
// unit; all lanes read the same x columns, so the x loads are broadcasts. The
// two kernels differ only in the unit arithmetic, so their ratio measures the
// format, not two different pipelines.
//
// Fallback kernel (K % 64 == 32): one warp per row with streaming loads.
#include <string.h>

#include "streamk.cuh"

namespace nm {

constexpr int kGemvWarps = 16;
constexpr int kGemvUnroll = 8;

template <int B, int OUT>
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
                if (OUT)
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

constexpr int kDnCols = 64; // columns per unit

// The dense unit: a 32 x 64 tile of W (128-byte swizzle) and the x slice.
struct DenseUnit {
    static constexpr int kCols = kDnCols;
    static constexpr bool kHasMasks = false;
    static constexpr int kWBytes = kUnitRows * kCols * 2;
    template <int B> static constexpr int stage_bytes() { return (kWBytes + 1023) / 1024 * 1024; }
    template <int B> static constexpr int x_bytes() { return 2 * kCols * B; }
    template <int B> static constexpr uint32_t tx_bytes() { return kWBytes + x_bytes<B>(); }
    template <int B> static constexpr int xf_bytes() { return kCols * BatchPad<B>::value * 4; }

    static __device__ __forceinline__ void issue_weights(uint32_t st, uint32_t bar, int kc, int32_t row0,
                                                         uint64_t pol, const TensorMaps &maps)
    {
        tma_load_2d_hint(st, &maps.w, kc * kCols, row0, bar, pol);
    }

    static constexpr int kSharedBytes = 0;
    struct State {};
    static __device__ __forceinline__ State initial_state() { return State{}; }
    static __device__ __forceinline__ void init_shared(uint8_t *, int, int) {}

    // One lane's row of the tile: 8 chunks of 8 bf16, in column order.
    template <int B> struct Regs {
        uint4 w[8];
    };
    template <int B> static __device__ __forceinline__ void load(const uint8_t *stp, int lane, Regs<B> &r)
    {
        const uint8_t *roww = stp + lane * 128;
        const int sw = lane & 7; // 16-byte chunk c of row r sits at c ^ (r & 7)
#pragma unroll
        for (int c = 0; c < 8; ++c)
            r.w[c] = *(const uint4 *)(roww + ((c ^ sw) << 4));
    }

    template <int B>
    static __device__ __forceinline__ void compute(const Regs<B> &r, const uint8_t *xs, uint8_t *xf, const uint8_t *,
                                                   State &, int lane, float (&acc)[4][B])
    {
        constexpr int BP = BatchPad<B>::value;
        convert_x<B, kCols>(xs, xf, lane);
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 t = r.w[c];
            const uint32_t wp[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float w = (e & 1) ? bf16hi_to_f32(wp[e >> 1]) : bf16lo_to_f32(wp[e >> 1]);
                const float *xa = (const float *)(xf + (8 * c + e) * BP * 4);
                float xs[BP];
                if (BP == 1) {
                    xs[0] = xa[0];
                } else if (BP == 2) {
                    const float2 v = *(const float2 *)xa;
                    xs[0] = v.x;
                    xs[1 % BP] = v.y;
                } else {
#pragma unroll
                    for (int b0 = 0; b0 < BP; b0 += 4) {
                        const float4 v = *(const float4 *)(xa + b0);
                        xs[b0 % BP] = v.x;
                        xs[(b0 + 1) % BP] = v.y;
                        xs[(b0 + 2) % BP] = v.z;
                        xs[(b0 + 3) % BP] = v.w;
                    }
                }
#pragma unroll
                for (int b = 0; b < B; ++b)
                    acc[c & 3][b] = fmaf(w, xs[b % BP], acc[c & 3][b]);
            }
        }
    }
};

template <int B> struct DenseCfg {
    static constexpr int W = B <= 2 ? 8 : B <= 4 ? 6 : 4;
    static constexpr int NBUF = 2;
    static constexpr int MINB = 2;
};

// Tensor maps of one dense linear: W (box 64 x 32 bf16, 128-byte swizzle), x (box 64 x B).
template <int B>
static nm_status encode_dense_maps(const void *W, const void *x, int64_t rows, int64_t K, TensorMaps *maps)
{
    memset(&maps->m, 0, sizeof maps->m);
    nm_status s;
    if ((s = encode_2d(&maps->w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, (uint64_t)K, (uint64_t)rows, (uint64_t)K * 2,
                       kDnCols, kUnitRows, CU_TENSOR_MAP_SWIZZLE_128B)) != NM_OK)
        return s;
    return encode_2d(&maps->x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)B, (uint64_t)K * 2,
                     kDnCols, B, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int B, int OUT>
static nm_status launch_gemv_tma(const void *W, const void *x, void *y, int64_t rows, int64_t K,
                                 const LaunchCtx &ctx)
{
    TensorMaps maps;
    nm_status s = encode_dense_maps<B>(W, x, rows, K, &maps);
    if (s != NM_OK)
        return s;
    const int64_t nrb = (rows + kUnitRows - 1) / kUnitRows, KC = K / kDnCols;
    if constexpr (B <= 2) {
        if (nrb <= ctx.num_sms && KC >= 64 && choose_split(nrb, KC, 16, 1, ctx.num_sms).whole)
            return launch_streamk<DenseUnit, B, 16, 2, 1, OUT>(maps, y, rows, KC, ctx);
    }
    return launch_streamk<DenseUnit, B, DenseCfg<B>::W, DenseCfg<B>::NBUF, DenseCfg<B>::MINB, OUT>(
        maps, y, rows, KC, ctx);
}

template <int B, int OUT>
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
    if (cudaLaunchKernelEx(&cfg, gemv_kernel<B, OUT>, (const uint16_t *)W, (const uint16_t *)x, y, rows, K) !=
        cudaSuccess)
        return NM_ERR_CUDA;
    return NM_OK;
}

template <int OUT>
static nm_status gemv_dispatch(const void *W, const void *x, void *y, int64_t rows, int64_t K, int batch,
                               const LaunchCtx &ctx)
{
    const bool tma = K % kDnCols == 0 && rows <= 0x7FFFFFFF && K <= 0x7FFFFFFF;
#define NM_CASE(BB)                                                                                         \
    case BB:                                                                                                \
        return tma ? launch_gemv_tma<BB, OUT>(W, x, y, rows, K, ctx) : launch_gemv_b<BB, OUT>(W, x, y, rows, K, ctx);
    switch (batch) {
        NM_CASE(1)
        NM_CASE(2)
        NM_CASE(3)
        NM_CASE(4)
        NM_CASE(5)
        NM_CASE(6)
        NM_CASE(7)
        NM_CASE(8)
    default:
        return NM_ERR_UNSUPPORTED;
    }
#undef NM_CASE
}

// ---------------------------------------------------------------------------
// The persistent stack kernel over dense linears
// ---------------------------------------------------------------------------

template <int B>
using DenseStack = StackLauncher<DenseUnit, B, DenseCfg<B>::W, DenseCfg<B>::NBUF, DenseCfg<B>::MINB>;

bool gemv_tma_ok(int64_t rows, int64_t K)
{
    return K > 0 && rows > 0 && K % kDnCols == 0 && rows <= 0x7FFFFFFF && K <= 0x7FFFFFFF;
}

nm_status stack_grid_dense(int batch, int num_sms, int *ctas)
{
    return with_batch(batch, [&](auto bc) { return DenseStack<decltype(bc)::value>::grid(num_sms, ctas); });
}

nm_status stack_encode_dense(const nm_linear &op, int batch, int ctas, StackOp *out)
{
    return with_batch(batch, [&](auto bc) {
        constexpr int B = decltype(bc)::value;
        nm_status s = encode_dense_maps<B>(op.W, op.x, op.rows, op.K, &out->maps);
        if (s == NM_OK)
            DenseStack<B>::split(out, op.y, op.rows, op.K / kDnCols, ctas);
        return s;
    });
}

nm_status stack_launch_dense(const StackOp *ops, int n_ops, int batch, uint32_t *gbar, int ctas,
                             const LaunchCtx &ctx)
{
    return with_batch(batch, [&](auto bc) {
        return DenseStack<decltype(bc)::value>::launch(ops, n_ops, gbar, ctas, ctx);
    });
}

nm_status launch_gemv(const void *W, const void *x, void *y, bool f32out, int64_t rows, int64_t K, int batch,
                      const LaunchCtx &ctx)
{
    return f32out ? gemv_dispatch<kOutF32>(W, x, y, rows, K, batch, ctx)
                  : gemv_dispatch<kOutBf16>(W, x, y, rows, K, batch, ctx);
}

} // namespace nm
