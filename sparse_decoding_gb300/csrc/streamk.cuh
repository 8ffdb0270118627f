// streamk.cuh -- the persistent TMA pipeline and the stream-K split shared by
// the sparse kernel (spmv.cu) and the dense reference (gemv.cu).
//
// Work is a grid of units: a row block is 32 rows (one per lane of a warp)
// and K/cols consecutive units along K. CTA c owns the contiguous unit range
// [U*c/P, U*(c+1)/P) and each of its warps a contiguous sub-range of it, so
// every warp streams the same number of bytes whatever the shape. Each warp
// runs its own pipeline of NBUF stage buffers, filled by TMA tensor copies
// that complete on one mbarrier per stage; the weights of the first stages
// are requested before the kernel waits for the previous kernel (programmatic
// dependent launch), x only after.
//
// A row block split between warps of one CTA is finished by the warp that
// arrives last (a shared-memory counter); one split between CTAs by the CTA
// that arrives last (a counter in the scratch). Partial sums are added in a
// fixed order, so results repeat bit for bit, and nobody waits for anybody.
//
// A unit policy `Pol` supplies the stage layout and the per-unit arithmetic:
//   Pol::kCols            columns per unit
//   Pol::kHasMasks        whether maps.m is used
//   Pol::stage_bytes<B>() bytes of one stage (multiple of 1024)
//   Pol::tx_bytes<B>()    bytes the stage's copies deliver
//   Pol::kXOffset         offset of the x slice in the stage
//   Pol::xf_bytes<B>()    per-warp scratch in shared memory (may be 0)
//   Pol::kSharedBytes     CTA-wide shared memory of the policy (tables)
//   Pol::init_shared(ptr, tid, nthreads)            fills it before the pipeline starts
//   Pol::issue_weights(stage, bar, kc, rb, policy, maps)
//   Pol::consume<B>(stage_ptr, xf_ptr, shared_ptr, state, lane, acc)
//                         accumulates into acc[4][B]; `state` is per warp
#pragma once

#include <algorithm>
#include <mutex>

#include "kernels.h"

namespace nm {

constexpr int kUnitRows = 32;       // one row per lane
constexpr int kGuardBytes = 64;     // guard band before each warp's x buffer
constexpr int kMinUnitsPerCta = 8;  // fewer CTAs than SMs for tiny problems

template <int B> struct BatchPad {
    static constexpr int value = B == 1 ? 1 : B == 2 ? 2 : B <= 4 ? 4 : 8;
};

struct TensorMaps {
    CUtensorMap w;    // values (sparse) or W (dense)
    CUtensorMap m;    // masks (sparse only)
    CUtensorMap x;    // x [batch][K]
};

struct StreamKParams {
    void *y;        // bf16 or fp32 [batch][rows]
    int64_t rows;   // valid rows
    int64_t U;      // units = row_blocks * KC
    int32_t KC;     // units per row block
    int32_t whole;  // CTA ranges in whole row blocks (no row block shared by CTAs)
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

// floor(a * b / c) for non-negative operands, with a 32-bit division when the
// product fits (the common case; 64-bit division is a long software sequence).
__device__ __forceinline__ int64_t muldiv(int64_t a, int64_t b, int64_t c)
{
    const uint64_t prod = (uint64_t)a * (uint64_t)b;
    if (prod <= 0xFFFFFFFFull && (uint64_t)c <= 0xFFFFFFFFull)
        return (int64_t)((uint32_t)prod / (uint32_t)c);
    return (int64_t)(prod / (uint64_t)c);
}

// a / b for non-negative operands, with a 32-bit division when both fit.
__device__ __forceinline__ int64_t div64(int64_t a, int64_t b)
{
    if (((uint64_t)a | (uint64_t)b) <= 0xFFFFFFFFull)
        return (int64_t)((uint32_t)a / (uint32_t)b);
    return a / b;
}

// The CTA's place in the stream-K split.
struct CtaRange {
    int64_t cs, ce; // unit range [cs, ce) of this CTA
    int nw;         // warps with work (min(W, ce - cs))
};

// per-warp partial sums in shared memory: [2 slots][B][32 lanes] fp32
template <int B> constexpr int part_bytes() { return 2 * B * 32 * 4; }

// Row block rb's total over this CTA's part of it is `tot` (lanes = rows).
// Store it, or -- when other CTAs hold parts of rb -- publish it in the scratch;
// the CTA that publishes last adds all parts in CTA order and stores y.
template <int B, bool F32OUT>
__device__ __forceinline__ void finish_across_ctas(const StreamKParams &p, const CtaRange &cr, int64_t rb,
                                                   const float (&tot)[B], int lane)
{
    const int64_t KC = p.KC;
    const int64_t rb_lo = rb * KC, rb_hi = rb_lo + KC;
    const int64_t row = rb * kUnitRows + lane;
    if (rb_lo >= cr.cs && rb_hi <= cr.ce) {
        store_y<B, F32OUT>(p.y, p.rows, row, tot);
        return;
    }
    const int64_t U = p.U, P = gridDim.x;
    const int64_t c = blockIdx.x;
    const int64_t first = div64(((rb_lo + 1) * (P)) - 1, U);
    const int64_t last = div64(((rb_hi) * (P)) - 1, U);
    const int slot = (rb == div64(cr.cs, KC)) ? 0 : 1;
    float *mine = p.scratch.partials + (c * 2 + slot) * (8 * 32) + lane;
#pragma unroll
    for (int b = 0; b < B; ++b)
        mine[b * 32] = tot[b];
    __threadfence();
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0)
        old = atomicAdd(&p.scratch.counters[first], 1u);
    old = __shfl_sync(0xFFFFFFFFu, old, 0);
    if (old != (uint32_t)(last - first))
        return;
    __threadfence();
    float sum[B];
#pragma unroll
    for (int b = 0; b < B; ++b)
        sum[b] = 0.f;
    // Issue the loads of up to 4 contributors at once, then add in CTA order.
    for (int64_t c0 = first; c0 <= last; c0 += 4) {
        float v[4][B];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t cc = c0 + j;
            if (cc <= last) {
                const int cslot = (rb == div64(muldiv(U, cc, P), KC)) ? 0 : 1;
                const float *q = p.scratch.partials + (cc * 2 + cslot) * (8 * 32) + lane;
#pragma unroll
                for (int b = 0; b < B; ++b)
                    v[j][b] = ldcg_f32(q + b * 32);
            } else {
#pragma unroll
                for (int b = 0; b < B; ++b)
                    v[j][b] = 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int b = 0; b < B; ++b)
                sum[b] += v[j][b];
    }
    store_y<B, F32OUT>(p.y, p.rows, row, sum);
    if (lane == 0)
        atomicExch(&p.scratch.counters[first], 0u);
}

// After the CTA's barrier: if this warp holds the last part of row block rb
// inside the CTA and rb is not complete in one warp, add the CTA's parts of
// rb (warp order, shared memory) and finish it across CTAs.
template <int B, bool F32OUT>
__device__ __forceinline__ void finish_in_cta(const StreamKParams &p, const CtaRange &cr, const float *part,
                                              int64_t rb, int64_t s0, int64_t s1, int lane)
{
    const int64_t KC = p.KC;
    const int64_t rb_lo = rb * KC, rb_hi = rb_lo + KC;
    const int64_t lo = rb_lo > cr.cs ? rb_lo : cr.cs;
    const int64_t hi = rb_hi < cr.ce ? rb_hi : cr.ce;
    if (s1 != hi)
        return; // a later warp holds the end of rb's part
    if (s0 == rb_lo && s1 == rb_hi)
        return; // stored directly by the loop
    const int64_t n = cr.ce - cr.cs;
    const int first = (int)div64(((lo - cr.cs + 1) * (cr.nw)) - 1, n);
    const int last = (int)div64(((hi - cr.cs) * (cr.nw)) - 1, n);
    float tot[B];
#pragma unroll
    for (int b = 0; b < B; ++b)
        tot[b] = 0.f;
    for (int w = first; w <= last; ++w) {
        const int64_t w_rb0 = div64(cr.cs + muldiv(n, w, cr.nw), KC);
        const int ws = (rb == w_rb0) ? 0 : 1;
        const float *q = part + ((w * 2 + ws) * B) * 32 + lane;
#pragma unroll
        for (int b = 0; b < B; ++b)
            tot[b] += q[b * 32];
    }
    finish_across_ctas<B, F32OUT>(p, cr, rb, tot, lane);
}

template <class Pol, int B, int W, int NBUF> constexpr int streamk_smem_bytes()
{
    return 1024 + W * NBUF * Pol::template stage_bytes<B>() + W * (kGuardBytes + Pol::template xf_bytes<B>()) +
           W * part_bytes<B>() + W * 4 + 16 + Pol::kSharedBytes;
}

template <class Pol, int B, int W, int NBUF, int MINB, bool F32OUT>
__global__ void __launch_bounds__(W * 32, MINB) streamk_kernel(const __grid_constant__ TensorMaps maps,
                                                                const StreamKParams p)
{
    constexpr int SB = Pol::template stage_bytes<B>();
    constexpr uint32_t TX = Pol::template tx_bytes<B>();
    constexpr int XF = Pol::template xf_bytes<B>();
    __shared__ __align__(8) uint64_t full_bar[W * NBUF];
    extern __shared__ __align__(1024) uint8_t dsmem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint8_t *const sbase = dsmem + ((1024u - (smem_addr(dsmem) & 1023u)) & 1023u);
    uint8_t *const stage0p = sbase + warp * NBUF * SB;
    uint8_t *const xfp = sbase + W * NBUF * SB + warp * (kGuardBytes + XF) + kGuardBytes;
    float *const part = (float *)(sbase + W * NBUF * SB + W * (kGuardBytes + XF));
    uint32_t *const cnt = (uint32_t *)((uint8_t *)part + W * part_bytes<B>());
    // 16-byte aligned policy region (the tables are copied with 16-byte stores)
    uint8_t *const pol_smem = (uint8_t *)(((uintptr_t)(cnt + W) + 15) & ~(uintptr_t)15);
    const uint32_t stage0 = smem_addr(stage0p);
    const uint32_t bar0 = smem_addr(&full_bar[warp * NBUF]);

    CtaRange cr;
    if (p.whole) {
        const int64_t nrb = div64(p.U, p.KC);
        cr.cs = muldiv(nrb, blockIdx.x, gridDim.x) * p.KC;
        cr.ce = muldiv(nrb, blockIdx.x + 1, gridDim.x) * p.KC;
    } else {
        cr.cs = muldiv(p.U, blockIdx.x, gridDim.x);
        cr.ce = muldiv(p.U, blockIdx.x + 1, gridDim.x);
    }
    cr.nw = (int)((cr.ce - cr.cs) < W ? (cr.ce - cr.cs) : W);

    Pol::init_shared(pol_smem, threadIdx.x, W * 32);
    if (lane == 0) {
        for (int i = 0; i < NBUF; ++i)
            mbar_init(bar0 + 8 * i, 1);
        fence_mbar_init();
    }
    if (threadIdx.x == 0) {
        prefetch_tensormap(&maps.w);
        if (Pol::kHasMasks)
            prefetch_tensormap(&maps.m);
        prefetch_tensormap(&maps.x);
    }
    __syncthreads();

    const bool active = warp < cr.nw;
    const int64_t n_cta = cr.ce - cr.cs;
    const int64_t ub = active ? cr.cs + muldiv(n_cta, warp, cr.nw) : 0;
    const int64_t ue = active ? cr.cs + muldiv(n_cta, warp + 1, cr.nw) : 0;
    const int n = (int)(ue - ub);
    const int32_t KC = p.KC;
    const int32_t rb0 = (int32_t)div64(ub, KC);
    const int32_t kc0 = (int32_t)(ub - (int64_t)rb0 * KC);

    // Weights do not depend on the previous kernel: start streaming them now.
    const uint64_t pol = l2_policy_evict_first();
    const int npre = n < NBUF ? n : NBUF;
    if (lane == 0) {
        int32_t rb = rb0, kc = kc0;
        for (int i = 0; i < npre; ++i) {
            mbar_arrive_expect_tx(bar0 + 8 * i, TX);
            Pol::issue_weights(stage0 + i * SB, bar0 + 8 * i, kc, rb * kUnitRows, pol, maps);
            if (++kc == KC) {
                kc = 0;
                ++rb;
            }
        }
    }
    // x may be the previous kernel's output.
    pdl_wait_upstream();
    if (lane == 0) {
        int32_t kc = kc0;
        for (int i = 0; i < npre; ++i) {
            tma_load_2d(stage0 + i * SB + Pol::kXOffset, &maps.x, kc * Pol::kCols, 0, bar0 + 8 * i);
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

    int32_t rb = rb0, kc = kc0;   // unit being consumed
    int32_t prb = rb0, pkc = kc0; // unit to prefetch next (i + NBUF)
    for (int i = 0; i < npre; ++i) {
        if (++pkc == KC) {
            pkc = 0;
            ++prb;
        }
    }
    int32_t seg_kc0 = kc0; // first unit of the current segment, as kc
    bool dead = false;
    typename Pol::State pst = Pol::initial_state();
    for (int i = 0; i < n; ++i) {
        const int s = i % NBUF;
        const uint32_t st = stage0 + s * SB, bar = bar0 + 8 * s;
        mbar_wait_bounded(bar, (uint32_t)((i / NBUF) & 1), p.scratch.status, dead);
        Pol::template consume<B>(stage0p + s * SB, xfp, pol_smem, pst, lane, acc);
        __syncwarp();
        if (i + NBUF < n) {
            if (lane == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, TX);
                Pol::issue_weights(st, bar, pkc, prb * kUnitRows, pol, maps);
                tma_load_2d(st + Pol::kXOffset, &maps.x, pkc * Pol::kCols, 0, bar);
            }
            if (++pkc == KC) {
                pkc = 0;
                ++prb;
            }
        }
        if (kc + 1 == KC || i == n - 1) { // end of a segment (row block or range)
            float tot[B];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                tot[b] = (acc[0][b] + acc[1][b]) + (acc[2][b] + acc[3][b]);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    acc[q][b] = 0.f;
            }
            if (seg_kc0 == 0 && kc + 1 == KC) {
                store_y<B, F32OUT>(p.y, p.rows, (int64_t)rb * kUnitRows + lane, tot); // a whole row block
            } else {
                float *mine = part + ((warp * 2 + (rb == rb0 ? 0 : 1)) * B) * 32 + lane;
#pragma unroll
                for (int b = 0; b < B; ++b)
                    mine[b * 32] = tot[b];
            }
            seg_kc0 = 0;
        }
        if (++kc == KC) {
            kc = 0;
            ++rb;
        }
    }
    __syncthreads(); // every partial of this CTA is in shared memory
    if (n > 0) {
        // the first and the last segment are the only ones that can be partial
        const int64_t rbf = rb0, rbl = div64(ue - 1, KC);
        finish_in_cta<B, F32OUT>(p, cr, part, rbf, ub, rbf == rbl ? ue : (rbf + 1) * (int64_t)KC, lane);
        if (rbl != rbf)
            finish_in_cta<B, F32OUT>(p, cr, part, rbl, rbl * (int64_t)KC, ue, lane);
    }
}

inline nm_status encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *ptr, uint64_t inner,
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

// How a launch splits its row blocks over CTAs.
struct Split {
    int64_t ctas;
    bool whole; // every CTA owns whole row blocks
};

// Whole row blocks per CTA avoid the fix-up between CTAs: at the end of a
// kernel, a row block shared by CTAs costs a chain of dependent L2 round trips
// (publish, count, read back) that delays the kernel's completion -- and with
// it the next kernel -- by several microseconds. Take whole row blocks when
// that keeps the CTAs within ~15% of even work and gives no warp more than
// about three units beyond an even split over all slots (the fix-up costs
// about that much); otherwise split units evenly (stream-K) over all slots.
inline Split choose_split(int64_t nrb, int64_t KC, int W, int minb, int num_sms)
{
    const int64_t slots = (int64_t)num_sms * minb;
    const int64_t U = nrb * KC;
    Split sp;
    sp.ctas = std::min<int64_t>(nrb, slots);
    const int64_t most = (nrb + sp.ctas - 1) / sp.ctas; // row blocks of the busiest CTA
    const bool balanced = most * sp.ctas <= nrb + nrb / 7;
    const int64_t per_warp_whole = (most * KC + W - 1) / W;
    const int64_t per_warp_even = (U + slots * W - 1) / (slots * W);
    sp.whole = balanced && per_warp_whole <= per_warp_even + 3;
    if (!sp.whole)
        sp.ctas = std::max<int64_t>(1, std::min<int64_t>(slots, U / kMinUnitsPerCta));
    sp.ctas = std::min<int64_t>(sp.ctas, kMaxCtas);
    return sp;
}

// Launch the stream-K kernel for a problem of `rows` rows and KC units per row
// block. MINB CTAs of W warps share an SM, so that at a kernel boundary the
// next kernel's CTAs can take the place of this kernel's first finishers and
// start streaming their weights while the rest of this kernel drains.
template <class Pol, int B, int W, int NBUF, int MINB, bool F32OUT>
nm_status launch_streamk(const TensorMaps &maps, void *y, int64_t rows, int64_t KC, const LaunchCtx &ctx)
{
    constexpr int smem = streamk_smem_bytes<Pol, B, W, NBUF>();
    static_assert(MINB * (smem + 1024) <= 232448, "MINB CTAs must fit one SM's shared memory");
    auto kern = streamk_kernel<Pol, B, W, NBUF, MINB, F32OUT>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_err != cudaSuccess)
        return NM_ERR_CUDA;

    StreamKParams p;
    p.y = y;
    p.rows = rows;
    p.KC = (int32_t)KC;
    p.U = ((rows + kUnitRows - 1) / kUnitRows) * KC;
    p.scratch = ctx.scratch;
    const int64_t nrb = (rows + kUnitRows - 1) / kUnitRows;
    const Split sp = choose_split(nrb, KC, W, MINB, ctx.num_sms);
    p.whole = sp.whole ? 1 : 0;
    const int64_t ctas = sp.ctas;

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
    if (cudaLaunchKernelEx(&cfg, kern, maps, p) != cudaSuccess)
        return NM_ERR_CUDA;
    return NM_OK;
}

// x slice of one unit, bf16 [B][cols] in the stage -> fp32 [cols][BP] in the warp's buffer.
template <int B, int COLS>
__device__ __forceinline__ void convert_x(const uint8_t *sx, uint8_t *xf, int lane)
{
    constexpr int BP = BatchPad<B>::value;
#pragma unroll
    for (int i = 0; i < COLS / 32; ++i) {
        const int c = lane + 32 * i;
        float f[BP];
#pragma unroll
        for (int b = 0; b < BP; ++b)
            f[b] = (b < B) ? bf16_to_f32(*(const uint16_t *)(sx + b * (COLS * 2) + c * 2)) : 0.f;
        float *dst = (float *)(xf + c * BP * 4);
        if (BP == 1) {
            dst[0] = f[0];
        } else if (BP == 2) {
            *(float2 *)dst = make_float2(f[0], f[1 % BP]);
        } else {
#pragma unroll
            for (int b = 0; b < BP; b += 4)
                *(float4 *)(dst + b) = make_float4(f[b % BP], f[(b + 1) % BP], f[(b + 2) % BP], f[(b + 3) % BP]);
        }
    }
}

} // namespace nm
