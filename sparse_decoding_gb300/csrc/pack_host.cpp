// pack_host.cpp -- bitmask conversion on the host (the product's packer).
//
// Same contract as the GPU pack (paper.rainbus.top summary, "方法步骤详情"
// step 3): per row and aligned 32-column group, a 32-bit word with bit j set
// when column j is kept, then the kept bf16 values in ascending column order.
// Nonzero is numeric (+-0 are zero). A subgroup short of N nonzeros is filled
// with its lowest-index zero positions; more than N is NM_ERR_NOT_NM.
#include <stdint.h>
#include <string.h>

#include "nmspmv.h"

static bool nm_pattern_ok(int N, int M)
{
    return (N == 2 && M == 4) || (N == 4 && M == 8) || (N == 8 && M == 16) || (N == 16 && M == 32);
}

extern "C" nm_status nm_pack_host(const uint16_t *W_bf16, int64_t rows, int64_t K, int N, int M, uint32_t *masks,
                                  uint16_t *values)
{
    if (!nm_pattern_ok(N, M))
        return NM_ERR_UNSUPPORTED;
    if (rows < 0 || K < 0 || (K % 32) != 0)
        return NM_ERR_SHAPE;
    if (rows == 0 || K == 0)
        return NM_OK;
    if (!W_bf16 || !masks || !values)
        return NM_ERR_INVALID_ARG;
    const int64_t words = K / 32;
    const uint32_t lowM = M == 32 ? 0xFFFFFFFFu : ((1u << M) - 1u);
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *wr = W_bf16 + r * K;
        for (int64_t g = 0; g < words; ++g) {
            const uint16_t *w = wr + 32 * g;
            uint32_t nz = 0;
            for (int j = 0; j < 32; ++j)
                nz |= (uint32_t)((w[j] & 0x7FFFu) != 0) << j;
            uint32_t mask = 0;
            for (int base = 0; base < 32; base += M) {
                uint32_t sub = (nz >> base) & lowM;
                int cnt = __builtin_popcount(sub);
                if (cnt > N)
                    return NM_ERR_NOT_NM;
                uint32_t zeros = ~sub & lowM;
                for (; cnt < N; ++cnt) {
                    const uint32_t z = zeros & (0u - zeros);
                    sub |= z;
                    zeros ^= z;
                }
                mask |= sub << base;
            }
            masks[r * words + g] = mask;
            uint16_t *v = values + r * (K / 2) + 16 * g;
            uint32_t m = mask;
            for (int k = 0; k < 16; ++k) {
                const int j = __builtin_ctz(m);
                m &= m - 1;
                v[k] = w[j];
            }
        }
    }
    return NM_OK;
}
