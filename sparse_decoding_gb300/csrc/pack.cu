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
// Both kernels give one thread one (row, 32-column group).
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
    const uint4 *wp = (const uint4 *)(W + row * K + 32 * g);
    uint32_t h[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 t = wp[i];
        h[4 * i + 0] = t.x;
        h[4 * i + 1] = t.y;
        h[4 * i + 2] = t.z;
        h[4 * i + 3] = t.w;
    }
    float s[32];
    const float4 *ap = (const float4 *)(a + 32 * g);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 t = __ldg(ap + i);
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
    const uint4 *wp = (const uint4 *)(W + row * K + 32 * g);
    uint32_t nz = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 t = wp[i];
        const uint32_t hv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = 8 * i + 2 * e;
            const uint32_t lo = hv[e] & 0xFFFFu, hi = hv[e] >> 16;
            col[j][threadIdx.x] = (uint16_t)lo;
            col[j + 1][threadIdx.x] = (uint16_t)hi;
            nz |= ((lo & 0x7FFFu) != 0 ? 1u : 0u) << j;
            nz |= ((hi & 0x7FFFu) != 0 ? 1u : 0u) << (j + 1);
        }
    }
    const uint32_t lowM = M == 32 ? 0xFFFFFFFFu : ((1u << M) - 1u);
    uint32_t mask = 0;
    bool over = false;
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
    if (over)
        atomicOr(bad, 1u);
    uint32_t m = mask, o[8];
#pragma unroll
    for (int k = 0; k < 16; k += 2) {
        const int p0 = (__ffs(m) - 1) & 31;
        m &= m - 1;
        const int p1 = (__ffs(m) - 1) & 31;
        m &= m - 1;
        o[k >> 1] = (uint32_t)col[p0][threadIdx.x] | ((uint32_t)col[p1][threadIdx.x] << 16);
    }
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
