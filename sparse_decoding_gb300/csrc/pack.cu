// pack.cu -- GPU N:M selection (Wanda rule) and bitmask pack.
//
// Selection follows the Wanda N:M rule that the pages name as the alternative
// pruning backend (daiwk.github.io notes, section "核心公式"; ai.info summary,
// Main Findings, "Gains are not specific to the pruning backend"): in every
// aligned M-column subgroup keep the N weights with the largest |W| * a_j.
// Pack follows the bitmask conversion (paper.rainbus.top summary,
// "方法步骤详情" step 3): one 32-bit word per 32 columns, bit j set when
// column j is kept, kept values following in ascending column order.
//
// Every kernel gives one thread one (row, 32-column group). select_pack_kernel
// does both steps in one pass (reads W once, writes masks and values).
#include <algorithm>

#include "kernels.h"

namespace nm {

constexpr int kPackThreads = 256;

__device__ __forceinline__ bool score_gt(float a, float b)
{
    // larger score first; a NaN score is above every number
    const bool na = isnan(a), nb = isnan(b);
    return na ? !nb : (!nb && a > b);
}

// The Wanda N:M keep mask of one 32-column group: h holds its 32 bf16
// weights as 16 pairs (low half first), ap points to its 32 activation norms.
// In every aligned M-subgroup the N entries with the largest fp32 score
// |w| * a_j are kept; larger score first, a NaN score above every number,
// equal scores to the lower column.
template <int M>
__device__ __forceinline__ uint32_t wanda_keep(const uint32_t (&h)[16], const float *ap, int N)
{
    float s[32];
    const float4 *a4 = (const float4 *)ap;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 t = __ldg(a4 + i);
        const float av[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = 4 * i + e;
            const float w = (j & 1) ? bf16hi_to_f32(h[j >> 1]) : bf16lo_to_f32(h[j >> 1]);
            s[j] = __fmul_rn(fabsf(w), av[e]);
        }
    }
    uint32_t keep = 0;
#pragma unroll
    for (int base = 0; base < 32; base += M) {
#pragma unroll
        for (int j = 0; j < M; ++j) {
            int above = 0;
#pragma unroll
            for (int i = 0; i < M; ++i) {
                if (i == j)
                    continue;
                // i outranks j: larger score, or an equal score at a lower column
                const bool o = score_gt(s[base + i], s[base + j]) || (i < j && !score_gt(s[base + j], s[base + i]));
                above += o ? 1 : 0;
            }
            keep |= (above < N ? 1u : 0u) << (base + j);
        }
    }
    return keep;
}

__device__ __forceinline__ void load_group(const uint16_t *W, int64_t row, int64_t K, int64_t g, uint32_t (&h)[16])
{
    const uint4 *wp = (const uint4 *)(W + row * K + 32 * g);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 t = wp[i];
        h[4 * i + 0] = t.x;
        h[4 * i + 1] = t.y;
        h[4 * i + 2] = t.z;
        h[4 * i + 3] = t.w;
    }
}

template <int M>
__global__ void __launch_bounds__(kPackThreads)
    select_kernel(const uint16_t *__restrict__ W, const float *__restrict__ a, int64_t rows, int64_t K, int N,
                  uint16_t *out)
{
    const int64_t words = K / 32;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= rows * words)
        return;
    const int64_t row = idx / words, g = idx - row * words;
    uint32_t h[16];
    load_group(W, row, K, g, h);
    const uint32_t keep = wanda_keep<M>(h, a + 32 * g, N);
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t lo = (keep >> (2 * i)) & 1u ? (h[i] & 0xFFFFu) : 0u;
        const uint32_t hi = (keep >> (2 * i + 1)) & 1u ? (h[i] & 0xFFFF0000u) : 0u;
        o[i] = lo | hi;
    }
    uint4 *op = (uint4 *)(out + row * K + 32 * g);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        op[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

// The 16 kept values of a group in ascending column order, from the group's
// columns staged in the thread's slice of `col`.
__device__ __forceinline__ void gather_kept(uint32_t mask, const uint16_t (*col)[kPackThreads], int tid,
                                            uint32_t (&o)[8])
{
    uint32_t m = mask;
#pragma unroll
    for (int k = 0; k < 16; k += 2) {
        const int p0 = (__ffs(m) - 1) & 31;
        m &= m - 1;
        const int p1 = (__ffs(m) - 1) & 31;
        m &= m - 1;
        o[k >> 1] = (uint32_t)col[p0][tid] | ((uint32_t)col[p1][tid] << 16);
    }
}

// The pack's mask word of a group of 32 bf16 values (16 pairs): per aligned
// M-subgroup its nonzero entries (+0 and -0 are zero; NaN is not), filled up
// to N with the subgroup's lowest-index zero entries; `over` is set when a
// subgroup holds more than N nonzeros.
template <int M>
__device__ __forceinline__ uint32_t pack_mask(const uint32_t (&h)[16], int N, bool &over)
{
    uint32_t nz = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        nz |= ((h[i] & 0x7FFFu) != 0 ? 1u : 0u) << (2 * i);
        nz |= ((h[i] & 0x7FFF0000u) != 0 ? 1u : 0u) << (2 * i + 1);
    }
    const uint32_t lowM = M == 32 ? 0xFFFFFFFFu : ((1u << M) - 1u);
    uint32_t mask = 0;
#pragma unroll
    for (int base = 0; base < 32; base += M) {
        uint32_t sub = (nz >> base) & lowM;
        int cnt = __popc(sub);
        if (cnt > N) {
            over = true;
        } else {
            uint32_t zeros = ~sub & lowM; // fill with the lowest-index zero positions
            while (cnt < N) {
                const uint32_t z = zeros & (0u - zeros);
                sub |= z;
                zeros ^= z;
                ++cnt;
            }
        }
        mask |= sub << base;
    }
    return mask;
}

// Selection and pack in one pass (50% patterns, N = M / 2): the Wanda rule
// picks the kept entries, the others become +0, and the pack's rule (nonzeros,
// filled to N with the lowest-index zeros) makes the mask word of that pruned
// group, exactly as nm_select followed by nm_pack -- without the pruned matrix
// being written and read back. (The mask is the selection's keep mask except
// where a kept weight is zero and outranks a lower-index one, which only a NaN
// or infinite column norm can cause: there the pack's fill rule decides.)
template <int M>
__global__ void __launch_bounds__(kPackThreads)
    select_pack_kernel(const uint16_t *__restrict__ W, const float *__restrict__ a, int64_t rows, int64_t K, int N,
                       uint32_t *masks, uint16_t *values)
{
    __shared__ uint16_t col[32][kPackThreads]; // [column][thread]: private to each thread
    const int64_t words = K / 32;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= rows * words)
        return;
    const int64_t row = idx / words, g = idx - row * words;
    uint32_t h[16];
    load_group(W, row, K, g, h);
    const uint32_t keep = wanda_keep<M>(h, a + 32 * g, N);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t lo = (keep >> (2 * i)) & 1u ? (h[i] & 0xFFFFu) : 0u;
        const uint32_t hi = (keep >> (2 * i + 1)) & 1u ? (h[i] & 0xFFFF0000u) : 0u;
        h[i] = lo | hi;
        col[2 * i][threadIdx.x] = (uint16_t)lo;
        col[2 * i + 1][threadIdx.x] = (uint16_t)(hi >> 16);
    }
    bool over = false; // cannot happen: the selection keeps N per subgroup
    const uint32_t mask = pack_mask<M>(h, N, over);
    uint32_t o[8];
    gather_kept(mask, col, threadIdx.x, o);
    uint4 *vp = (uint4 *)(values + row * (K / 2) + 16 * g);
    vp[0] = make_uint4(o[0], o[1], o[2], o[3]);
    vp[1] = make_uint4(o[4], o[5], o[6], o[7]);
    masks[row * words + g] = mask;
}

template <int M>
__global__ void __launch_bounds__(kPackThreads)
    pack_kernel(const uint16_t *__restrict__ W, int64_t rows, int64_t K, int N, uint32_t *masks, uint16_t *values,
                uint32_t *bad, int pair_off)
{
    __shared__ uint16_t col[32][kPackThreads]; // [column][thread]: private to each thread
    const int64_t words = K / 32;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= rows * words)
        return;
    const int64_t row = idx / words, g = idx - row * words;
    uint32_t h[16];
    load_group(W, row, K, g, h);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        col[2 * i][threadIdx.x] = (uint16_t)(h[i] & 0xFFFFu);
        col[2 * i + 1][threadIdx.x] = (uint16_t)(h[i] >> 16);
    }
    bool over = false;
    const uint32_t mask = pack_mask<M>(h, N, over);
    if (over)
        atomicOr(bad, 1u);
    uint32_t o[8];
    gather_kept(mask, col, threadIdx.x, o);
    // output row: the input row, or its slot in the gate/up pair layout
    const int64_t orow = pair_off < 0 ? row : (row >> 4) * 32 + (row & 15) + pair_off;
    uint4 *vp = (uint4 *)(values + orow * (K / 2) + 16 * g);
    vp[0] = make_uint4(o[0], o[1], o[2], o[3]);
    vp[1] = make_uint4(o[4], o[5], o[6], o[7]);
    masks[orow * words + g] = mask;
}

static int64_t grid_for(int64_t items)
{
    return (items + kPackThreads - 1) / kPackThreads;
}

nm_status launch_select(const void *W, const float *a, int64_t rows, int64_t K, int N, int M, void *out,
                        const LaunchCtx &ctx)
{
    const int64_t items = rows * (K / 32);
    if (items == 0)
        return NM_OK;
    const int64_t grid = grid_for(items);
    if (grid > 0x7FFFFFFF)
        return NM_ERR_SHAPE;
    const dim3 gr((unsigned)grid), bl(kPackThreads);
    const uint16_t *w = (const uint16_t *)W;
    uint16_t *o = (uint16_t *)out;
    switch (M) {
    case 4: select_kernel<4><<<gr, bl, 0, ctx.stream>>>(w, a, rows, K, N, o); break;
    case 8: select_kernel<8><<<gr, bl, 0, ctx.stream>>>(w, a, rows, K, N, o); break;
    case 16: select_kernel<16><<<gr, bl, 0, ctx.stream>>>(w, a, rows, K, N, o); break;
    case 32: select_kernel<32><<<gr, bl, 0, ctx.stream>>>(w, a, rows, K, N, o); break;
    default: return NM_ERR_UNSUPPORTED;
    }
    return cudaGetLastError() == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}

nm_status launch_select_pack(const void *W, const float *a, int64_t rows, int64_t K, int N, int M, uint32_t *masks,
                             void *values, const LaunchCtx &ctx)
{
    const int64_t items = rows * (K / 32);
    if (items == 0)
        return NM_OK;
    const int64_t grid = grid_for(items);
    if (grid > 0x7FFFFFFF)
        return NM_ERR_SHAPE;
    const dim3 gr((unsigned)grid), bl(kPackThreads);
    const uint16_t *w = (const uint16_t *)W;
    uint16_t *v = (uint16_t *)values;
    switch (M) {
    case 4: select_pack_kernel<4><<<gr, bl, 0, ctx.stream>>>(w, a, rows, K, N, masks, v); break;
    case 8: select_pack_kernel<8><<<gr, bl, 0, ctx.stream>>>(w, a, rows, K, N, masks, v); break;
    case 16: select_pack_kernel<16><<<gr, bl, 0, ctx.stream>>>(w, a, rows, K, N, masks, v); break;
    case 32: select_pack_kernel<32><<<gr, bl, 0, ctx.stream>>>(w, a, rows, K, N, masks, v); break;
    default: return NM_ERR_UNSUPPORTED;
    }
    return cudaGetLastError() == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}

nm_status launch_pack(const void *W, int64_t rows, int64_t K, int N, int M, uint32_t *masks, void *values,
                      const LaunchCtx &ctx, int pair_off)
{
    const int64_t items = rows * (K / 32);
    if (items == 0)
        return NM_OK;
    const int64_t grid = grid_for(items);
    if (grid > 0x7FFFFFFF)
        return NM_ERR_SHAPE;
    const dim3 gr((unsigned)grid), bl(kPackThreads);
    const uint16_t *w = (const uint16_t *)W;
    uint16_t *v = (uint16_t *)values;
    uint32_t *bad = ctx.scratch.status + 1;
    switch (M) {
    case 4: pack_kernel<4><<<gr, bl, 0, ctx.stream>>>(w, rows, K, N, masks, v, bad, pair_off); break;
    case 8: pack_kernel<8><<<gr, bl, 0, ctx.stream>>>(w, rows, K, N, masks, v, bad, pair_off); break;
    case 16: pack_kernel<16><<<gr, bl, 0, ctx.stream>>>(w, rows, K, N, masks, v, bad, pair_off); break;
    case 32: pack_kernel<32><<<gr, bl, 0, ctx.stream>>>(w, rows, K, N, masks, v, bad, pair_off); break;
    default: return NM_ERR_UNSUPPORTED;
    }
    return cudaGetLastError() == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}

} // namespace nm
