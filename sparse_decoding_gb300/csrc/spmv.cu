// spmv.cu -- bitmask N:M decode SpMV kernels for sm_103a.
//
// y[b][r] = sum_j W[r][j] x[b][j] with W stored as 32-bit masks plus the kept
// bf16 values (SparseDecoding: paper.rainbus.top summary, "核心方法" and
// "方法步骤详情" steps 3-4; ai.info summary, "Methodology in Plain English"
// steps 2-3). Each mask word has exactly 16 set bits, so every word takes the
// same 16 steps: find a set bit (its position is the column of the next kept
// value), clear it, multiply-accumulate. The pages walk from the least
// significant bit; here the walk runs from the most significant bit down,
// which visits the same (column, value) pairs in reverse order with a
// shorter dependency chain (bfind, clear) -- the product is the same sum.
//
// Main kernel (K % 128 == 0): the work is cut into units of 32 rows x 128
// columns (4 mask words per row). Every warp is a stream-K worker that owns a
// contiguous range of units, so all warps of the GPU get the same number of
// weight bytes whatever the shape. Each warp runs its own TMA pipeline: NBUF
// stage buffers in shared memory, each filled by three tensor copies (values
// with 128-byte swizzle, masks, and the unit's 128-column slice of x) that
// complete on one mbarrier. Lane i of the warp owns row i of the unit, so all
// 32 lanes read x inside the same 32-column window: the gathers never
// conflict in shared memory. A row block split between workers is finished
// by whichever worker arrives last (a counter per block in the scratch), which
// adds the partial sums in worker order: the result does not depend on timing.
//
// Fallback kernel (any K % 32 == 0): the same lane-per-row walk with plain
// loads from global memory.
#include <algorithm>
#include <mutex>

#include "kernels.h"

namespace nm {

constexpr int kUnitRows = 32;                        // one row per lane
constexpr int kUnitCols = 128;                       // columns per unit
constexpr int kUnitWords = kUnitCols / 32;           // mask words per row per unit
constexpr int kValBytes = kUnitRows * kUnitCols;     // 32 rows x 64 bf16
constexpr int kMaskBytes = kUnitRows * kUnitWords * 4;
constexpr int kGuardBytes = 64; // read by the walk of a malformed (all-clear) word

template <int B> struct BatchPad {
    static constexpr int value = B == 1 ? 1 : B == 2 ? 2 : B <= 4 ? 4 : 8;
};
template <int B> constexpr int stage_bytes() { return (kValBytes + kMaskBytes + 256 * B + 1023) / 1024 * 1024; }
template <int B> constexpr int xf_bytes() { return kUnitCols * BatchPad<B>::value * 4; }
template <int B, int W, int NBUF> constexpr int tma_smem_bytes()
{
    return 1024 + W * NBUF * stage_bytes<B>() + W * (kGuardBytes + xf_bytes<B>());
}

// Warps per CTA and stage buffers per warp, by batch size.
template <int B> struct TmaCfg {
    static constexpr int W = B <= 2 ? 16 : B <= 4 ? 12 : 8;
    static constexpr int NBUF = 2;
};

struct SpmvParams {
    void *y;      // bf16 or fp32 [batch][rows]
    int64_t rows; // valid rows
    int64_t U;    // units = row_blocks * KC
    int32_t KC;   // units per row block (K / 128)
    int32_t G;    // stream-K workers (warps) with work, G <= U
    Scratch scratch;
};

template <int B, bool F32OUT>
__device__ __forceinline__ void store_y(void *y, int64_t rows, int64_t row, const float (&v)[B])
{
    if (row >= rows)
        return;
#pragma unroll
    for (int b = 0; b < B; ++b) {
        if (F32OUT)
            ((float *)y)[(int64_t)b * rows + row] = v[b];
        else
            ((uint16_t *)y)[(int64_t)b * rows + row] = f32_to_bf16_rn(v[b]);
    }
}

// Worker whose unit range contains unit u (ranges are [U*g/G, U*(g+1)/G)).
__device__ __forceinline__ int64_t owner_of(int64_t u, int64_t U, int64_t G)
{
    return ((u + 1) * G - 1) / U;
}

// Finish row block rb after this worker has covered units [s0, s1) of it.
template <int B, bool F32OUT>
__device__ __forceinline__ void finish_row_block(const SpmvParams &p, int64_t g, int64_t rb0, int64_t rb,
                                                 int64_t s0, int64_t s1, const float (&tot)[B], int lane)
{
    const int64_t KC = p.KC;
    const int64_t row = rb * kUnitRows + lane;
    if (s0 == rb * KC && s1 == (rb + 1) * KC) {
        store_y<B, F32OUT>(p.y, p.rows, row, tot);
        return;
    }
    const int64_t G = p.G, U = p.U;
    const int64_t first = owner_of(rb * KC, U, G);
    const int64_t last = owner_of((rb + 1) * KC - 1, U, G);
    const int slot = (rb == rb0) ? 0 : 1;
    float *mine = p.scratch.partials + ((g * 2 + slot) * 32 + lane) * 8;
#pragma unroll
    for (int b = 0; b < B; ++b)
        mine[b] = tot[b];
    __threadfence();
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0)
        old = atomicAdd(&p.scratch.counters[first], 1u);
    old = __shfl_sync(0xFFFFFFFFu, old, 0);
    if (old != (uint32_t)(last - first))
        return;
    // Last contributor: add every contributor's partial in worker order.
    __threadfence();
    float sum[B];
#pragma unroll
    for (int b = 0; b < B; ++b)
        sum[b] = 0.f;
    for (int64_t c = first; c <= last; ++c) {
        const int64_t c_rb0 = (U * c / G) / KC;
        const int cs = (rb == c_rb0) ? 0 : 1;
        const float *q = p.scratch.partials + ((c * 2 + cs) * 32 + lane) * 8;
#pragma unroll
        for (int b = 0; b < B; ++b)
            sum[b] += ldcg_f32(q + b);
    }
    store_y<B, F32OUT>(p.y, p.rows, row, sum);
    if (lane == 0)
        atomicExch(&p.scratch.counters[first], 0u);
}

// x slice of one unit, bf16 [B][128] -> fp32 [128][BP] in the warp's buffer.
template <int B>
__device__ __forceinline__ void convert_x(const uint8_t *sx, uint8_t *xf, int lane)
{
    constexpr int BP = BatchPad<B>::value;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = lane + 32 * i;
        float f[BP];
#pragma unroll
        for (int b = 0; b < BP; ++b)
            f[b] = (b < B) ? bf16_to_f32(*(const uint16_t *)(sx + b * 256 + c * 2)) : 0.f;
        float *dst = (float *)(xf + c * BP * 4);
        if (BP == 1) {
            dst[0] = f[0];
        } else if (BP == 2) {
            *(float2 *)dst = make_float2(f[0], f[1 % BP]);
        } else {
#pragma unroll
            for (int b = 0; b < BP; b += 4)
                *(float4 *)(dst + b) = make_float4(f[b], f[(b + 1) % BP], f[(b + 2) % BP], f[(b + 3) % BP]);
        }
    }
}

// 16 fixed steps over the 4 mask words of this lane's row in one unit.
template <int B>
__device__ __forceinline__ void walk_unit(const uint8_t *st, const uint8_t *xf, int lane, float (&acc)[4][B])
{
    constexpr int BP = BatchPad<B>::value;
    const uint4 mw = *(const uint4 *)(st + kValBytes + lane * 16);
    uint32_t m[4] = {mw.x, mw.y, mw.z, mw.w};
    uint32_t v[4][8];
    const uint8_t *rowv = st + lane * 128;
    const int sw = lane & 7; // 128-byte swizzle: 16-byte chunk c of row r sits at c ^ (r & 7)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 t = *(const uint4 *)(rowv + (((2 * q + h) ^ sw) << 4));
            v[q][4 * h + 0] = t.x;
            v[q][4 * h + 1] = t.y;
            v[q][4 * h + 2] = t.z;
            v[q][4 * h + 3] = t.w;
        }
    }
#pragma unroll
    for (int step = 0; step < 16; ++step) {
        const int k = 15 - step; // value index of the highest remaining set bit
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int pos = bfind_u32(m[q]); // -1 only for a malformed word
            m[q] &= ~(1u << (pos & 31));
            const float *xa = (const float *)(xf + (q * 32 + pos) * BP * 4);
            const uint32_t pr = v[q][k >> 1];
            const float wv = (k & 1) ? bf16hi_to_f32(pr) : bf16lo_to_f32(pr);
            if (BP == 1) {
                acc[q][0] = fmaf(wv, xa[0], acc[q][0]);
            } else if (BP == 2) {
                const float2 xv = *(const float2 *)xa;
                acc[q][0] = fmaf(wv, xv.x, acc[q][0]);
                if (B > 1)
                    acc[q][1 % B] = fmaf(wv, xv.y, acc[q][1 % B]);
            } else {
#pragma unroll
                for (int b0 = 0; b0 < BP; b0 += 4) {
                    if (b0 < B) {
                        const float4 xv = *(const float4 *)(xa + b0);
                        const float xs[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (b0 + j < B)
                                acc[q][(b0 + j) % B] = fmaf(wv, xs[j], acc[q][(b0 + j) % B]);
                    }
                }
            }
        }
    }
}

template <int B, int W, int NBUF, bool F32OUT>
__global__ void __launch_bounds__(W * 32, 1)
    spmv_tma_kernel(const __grid_constant__ CUtensorMap tm_vals, const __grid_constant__ CUtensorMap tm_masks,
                    const __grid_constant__ CUtensorMap tm_x, const SpmvParams p)
{
    constexpr int SB = stage_bytes<B>();
    constexpr uint32_t TX = kValBytes + kMaskBytes + 256 * B;
    __shared__ __align__(8) uint64_t full_bar[W * NBUF];
    extern __shared__ __align__(1024) uint8_t dsmem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint8_t *const sbase = dsmem + ((1024u - (smem_addr(dsmem) & 1023u)) & 1023u);
    uint8_t *const stage0p = sbase + warp * NBUF * SB;
    uint8_t *const xfp = sbase + W * NBUF * SB + warp * (kGuardBytes + xf_bytes<B>()) + kGuardBytes;
    const uint32_t stage0 = smem_addr(stage0p);
    const uint32_t bar0 = smem_addr(&full_bar[warp * NBUF]);

    const int64_t g = (int64_t)blockIdx.x * W + warp;
    if (g >= p.G) {
        pdl_wait_upstream();
        pdl_launch_dependents();
        return;
    }
    const int64_t ub = p.U * g / p.G;
    const int64_t ue = p.U * (g + 1) / p.G;
    const int n = (int)(ue - ub);
    const int64_t KC = p.KC;
    const int64_t rb0 = ub / KC;
    const int64_t kc0 = ub - rb0 * KC;

    if (lane == 0) {
        for (int i = 0; i < NBUF; ++i)
            mbar_init(bar0 + 8 * i, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // Weights do not depend on the previous kernel: start streaming them now.
    const uint64_t pol = l2_policy_evict_first();
    const int npre = n < NBUF ? n : NBUF;
    if (lane == 0) {
        int64_t rb = rb0, kc = kc0;
        for (int i = 0; i < npre; ++i) {
            const uint32_t st = stage0 + i * SB, bar = bar0 + 8 * i;
            mbar_arrive_expect_tx(bar, TX);
            tma_load_2d_hint(st, &tm_vals, (int32_t)(kc * 64), (int32_t)(rb * kUnitRows), bar, pol);
            tma_load_2d_hint(st + kValBytes, &tm_masks, (int32_t)(kc * kUnitWords), (int32_t)(rb * kUnitRows),
                             bar, pol);
            if (++kc == KC) {
                kc = 0;
                ++rb;
            }
        }
    }
    // x may be the previous kernel's output.
    pdl_wait_upstream();
    if (lane == 0) {
        int64_t kc = kc0;
        for (int i = 0; i < npre; ++i) {
            tma_load_2d(stage0 + i * SB + kValBytes + kMaskBytes, &tm_x, (int32_t)(kc * kUnitCols), 0,
                        bar0 + 8 * i);
            if (++kc == KC)
                kc = 0;
        }
    }
    pdl_launch_dependents();

    float acc[4][B];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int b = 0; b < B; ++b)
            acc[q][b] = 0.f;

    int64_t rb = rb0, kc = kc0;       // unit being consumed
    int64_t prb = rb0, pkc = kc0;     // unit to prefetch next (i + NBUF)
    for (int i = 0; i < npre; ++i) {
        if (++pkc == KC) {
            pkc = 0;
            ++prb;
        }
    }
    int64_t seg0 = ub;
    bool dead = false;
    for (int i = 0; i < n; ++i) {
        const int s = i % NBUF;
        const uint32_t st = stage0 + s * SB, bar = bar0 + 8 * s;
        mbar_wait_bounded(bar, (uint32_t)((i / NBUF) & 1), p.scratch.status, dead);
        const uint8_t *stp = stage0p + s * SB;
        convert_x<B>(stp + kValBytes + kMaskBytes, xfp, lane);
        __syncwarp();
        walk_unit<B>(stp, xfp, lane, acc);
        __syncwarp();
        if (i + NBUF < n) {
            if (lane == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, TX);
                tma_load_2d_hint(st, &tm_vals, (int32_t)(pkc * 64), (int32_t)(prb * kUnitRows), bar, pol);
                tma_load_2d_hint(st + kValBytes, &tm_masks, (int32_t)(pkc * kUnitWords),
                                 (int32_t)(prb * kUnitRows), bar, pol);
                tma_load_2d(st + kValBytes + kMaskBytes, &tm_x, (int32_t)(pkc * kUnitCols), 0, bar);
            }
            if (++pkc == KC) {
                pkc = 0;
                ++prb;
            }
        }
        const int64_t u = ub + i;
        const bool rb_end = (kc + 1 == KC);
        if (rb_end || i == n - 1) {
            float tot[B];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                tot[b] = (acc[0][b] + acc[1][b]) + (acc[2][b] + acc[3][b]);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    acc[q][b] = 0.f;
            }
            finish_row_block<B, F32OUT>(p, g, rb0, rb, seg0, u + 1, tot, lane);
            seg0 = u + 1;
        }
        if (++kc == KC) {
            kc = 0;
            ++rb;
        }
    }
}

// ---------------------------------------------------------------------------
// Fallback: lane-per-row walk with plain global loads (any K % 32 == 0).
// ---------------------------------------------------------------------------
template <int B, bool F32OUT>
__global__ void __launch_bounds__(256)
    spmv_simple_kernel(const uint32_t *__restrict__ masks, const uint16_t *__restrict__ values,
                       const uint16_t *__restrict__ x, void *y, int64_t rows, int64_t K)
{
    pdl_wait_upstream();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    const int64_t nrb = (rows + 31) / 32;
    const int64_t words = K / 32;
    for (int64_t rb = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); rb < nrb; rb += warps) {
        const int64_t row = rb * 32 + lane;
        float acc[B];
#pragma unroll
        for (int b = 0; b < B; ++b)
            acc[b] = 0.f;
        if (row < rows) {
            for (int64_t g = 0; g < words; ++g) {
                uint32_t m = __ldg(masks + row * words + g);
                const uint4 *vp = (const uint4 *)(values + row * (K / 2) + 16 * g);
                const uint4 v0 = __ldg(vp), v1 = __ldg(vp + 1);
                const uint32_t vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                const uint16_t *xg = x + 32 * g;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int pos = (__ffs(m) - 1) & 31; // stays inside the word's columns
                    m &= m - 1;
                    const float wv = (k & 1) ? bf16hi_to_f32(vv[k >> 1]) : bf16lo_to_f32(vv[k >> 1]);
#pragma unroll
                    for (int b = 0; b < B; ++b)
                        acc[b] = fmaf(wv, bf16_to_f32(__ldg(xg + (int64_t)b * K + pos)), acc[b]);
                }
            }
        }
        store_y<B, F32OUT>(y, rows, row, acc);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

SpmvPath spmv_path(int64_t rows, int64_t K)
{
    if (K % kUnitCols == 0 && K > 0 && rows > 0 && rows <= 0x7FFFFFFF && K <= 0x7FFFFFFF)
        return kSpmvTma;
    return kSpmvSimple;
}

static nm_status encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *ptr, uint64_t inner,
                           uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                           CUtensorMapSwizzle swz)
{
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn)
        return NM_ERR_CUDA;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t es[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? NM_OK : NM_ERR_CUDA;
}

template <int B, bool F32OUT>
static nm_status launch_tma(const uint32_t *masks, const void *values, const void *x, void *y, int64_t rows,
                            int64_t K, const LaunchCtx &ctx)
{
    constexpr int W = TmaCfg<B>::W, NBUF = TmaCfg<B>::NBUF;
    constexpr int smem = tma_smem_bytes<B, W, NBUF>();
    auto kern = spmv_tma_kernel<B, W, NBUF, F32OUT>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_err != cudaSuccess)
        return NM_ERR_CUDA;

    CUtensorMap tv, tmk, tx;
    nm_status s;
    if ((s = encode_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, values, (uint64_t)K / 2, (uint64_t)rows,
                       (uint64_t)K, 64, kUnitRows, CU_TENSOR_MAP_SWIZZLE_128B)) != NM_OK)
        return s;
    if ((s = encode_2d(&tmk, CU_TENSOR_MAP_DATA_TYPE_UINT32, masks, (uint64_t)K / 32, (uint64_t)rows,
                       (uint64_t)K / 8, kUnitWords, kUnitRows, CU_TENSOR_MAP_SWIZZLE_NONE)) != NM_OK)
        return s;
    if ((s = encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)B, (uint64_t)K * 2,
                       kUnitCols, B, CU_TENSOR_MAP_SWIZZLE_NONE)) != NM_OK)
        return s;

    SpmvParams p;
    p.y = y;
    p.rows = rows;
    p.KC = (int32_t)(K / kUnitCols);
    p.U = ((rows + kUnitRows - 1) / kUnitRows) * (int64_t)p.KC;
    int64_t ctas = std::min<int64_t>((int64_t)ctx.num_sms, (p.U + W - 1) / W);
    if (ctas < 1)
        ctas = 1;
    p.G = (int32_t)std::min<int64_t>(std::min<int64_t>(ctas * W, p.U), kMaxWorkers);
    ctas = (p.G + W - 1) / W;
    p.scratch = ctx.scratch;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(W * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = ctx.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tv, tmk, tx, p) != cudaSuccess)
        return NM_ERR_CUDA;
    return NM_OK;
}

template <int B, bool F32OUT>
static nm_status launch_simple(const uint32_t *masks, const void *values, const void *x, void *y, int64_t rows,
                               int64_t K, const LaunchCtx &ctx)
{
    const int64_t nrb = (rows + 31) / 32;
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((nrb + 7) / 8, (int64_t)ctx.num_sms * 8));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = ctx.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, spmv_simple_kernel<B, F32OUT>, masks, (const uint16_t *)values,
                           (const uint16_t *)x, y, rows, K) != cudaSuccess)
        return NM_ERR_CUDA;
    return NM_OK;
}

template <bool F32OUT>
static nm_status dispatch(const uint32_t *masks, const void *values, const void *x, void *y, int64_t rows,
                          int64_t K, int batch, const LaunchCtx &ctx)
{
    const bool tma = spmv_path(rows, K) == kSpmvTma;
#define NM_CASE(BB)                                                                                         \
    case BB:                                                                                                \
        return tma ? launch_tma<BB, F32OUT>(masks, values, x, y, rows, K, ctx)                              \
                   : launch_simple<BB, F32OUT>(masks, values, x, y, rows, K, ctx);
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

nm_status launch_spmv(const uint32_t *masks, const void *values, const void *x, void *y, bool f32out,
                      int64_t rows, int64_t K, int batch, const LaunchCtx &ctx)
{
    return f32out ? dispatch<true>(masks, values, x, y, rows, K, batch, ctx)
                  : dispatch<false>(masks, values, x, y, rows, K, batch, ctx);
}

} // namespace nm
