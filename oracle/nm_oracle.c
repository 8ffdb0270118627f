/*
 * nm_oracle.c -- CPU oracle for the bitmask N:M decode SpMV.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path never
 * calls it, and it shares no source with the CUDA library.
 *
 * Everything here is the plain definition, written for a reader to check by
 * eye: loops in index order, fp64 accumulation, no blocking or fusion.
 *
 * Source: SparseDecoding, "Decoding-Aware Pruning for Accurate and Efficient
 * LLM Inference", as restated by
 *   - paper.rainbus.top summary, section "方法步骤详情" step 3 (rows are stored
 *     as a compact value array plus 32-bit bitmasks, a set bit marks a kept
 *     weight) and section "核心方法" (exactly 16 set bits per aligned 32-bit
 *     word for 50% N:M with M <= 32; least-significant set bit = next column);
 *   - ai.info summary, "Methodology in Plain English" steps 2-3 (values stored
 *     in increasing column order, one-to-one with the set bits);
 *   - daiwk.github.io notes, section "核心公式" (Wanda N:M rule: score
 *     s_ij = |W_ij| * sqrt(sum_t X_jt^2), keep N per M-column group, no
 *     compensation).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - bit j (LSB = 0) of word g of a row <-> column 32g+j; the k-th set bit
 *     from the LSB <-> values[16g+k];
 *   - M-subgroups are aligned inside the word: columns [32g+sM, 32g+sM+M);
 *   - "nonzero" is numeric: +0 and -0 are zero, NaN and Inf are nonzero;
 *   - a subgroup with fewer than N nonzeros is filled up to N with its
 *     lowest-index zero positions; more than N nonzeros is an error;
 *   - kept values are copied bit for bit; unpack writes +0 elsewhere;
 *   - selection: score in fp32 as |W| * a_j, larger wins, NaN counts as larger
 *     than any number, equal scores go to the lower column index.
 *
 * Status codes (this file's own): 0 ok, 1 bad argument, 2 bad shape,
 * 4 unsupported N:M, 5 more than N nonzeros in a subgroup, 7 malformed mask.
 *
 * Parity pins live in tests/test_oracle_pins.py; no function here is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define OR_OK 0
#define OR_BAD_ARG 1
#define OR_BAD_SHAPE 2
#define OR_UNSUPPORTED 4
#define OR_NOT_NM 5
#define OR_BAD_MASK 7

static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* A bf16 value is numerically zero when all bits but the sign are clear. */
static int bf16_is_zero(uint16_t h)
{
    return (h & 0x7FFFu) == 0;
}

static int pattern_supported(int N, int M)
{
    return (N == 2 && M == 4) || (N == 4 && M == 8) || (N == 8 && M == 16) ||
           (N == 16 && M == 32);
}

static int shape_ok(int64_t rows, int64_t K)
{
    return rows >= 0 && K >= 0 && (K % 32) == 0;
}

/* "s_i outranks s_j": larger score first, NaN above every number. */
static int score_greater(float si, float sj)
{
    if (isnan(si))
        return !isnan(sj);
    if (isnan(sj))
        return 0;
    return si > sj;
}

/*
 * Wanda N:M selection (daiwk.github.io notes, "核心公式"; p4 step 4 lists the
 * Wanda backend as an alternative to SparseGPT). For every row and every
 * aligned M-column subgroup keep the N entries with the largest score
 * s_j = |W_rj| * a_j and zero the rest. Rank of entry j = number of entries
 * in its subgroup that outrank it (larger score, or equal score at a lower
 * column); keep j when its rank is below N.
 */
int oracle_select(const uint16_t *W, const float *a, int64_t rows, int64_t K, int N, int M,
                  uint16_t *W_pruned)
{
    if (!pattern_supported(N, M))
        return OR_UNSUPPORTED;
    if (!shape_ok(rows, K))
        return OR_BAD_SHAPE;
    if ((rows > 0 && K > 0) && (!W || !a || !W_pruned))
        return OR_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *w = W + r * K;
        uint16_t *out = W_pruned + r * K;
        for (int64_t c0 = 0; c0 < K; c0 += M) {
            for (int j = 0; j < M; ++j) {
                float sj = fabsf(bf16_bits_to_float(w[c0 + j])) * a[c0 + j];
                int rank = 0;
                for (int i = 0; i < M; ++i) {
                    if (i == j)
                        continue;
                    float si = fabsf(bf16_bits_to_float(w[c0 + i])) * a[c0 + i];
                    if (score_greater(si, sj) || (!score_greater(sj, si) && i < j))
                        rank++;
                }
                out[c0 + j] = (rank < N) ? w[c0 + j] : (uint16_t)0;
            }
        }
    }
    return OR_OK;
}

/*
 * Bitmask pack (paper.rainbus.top "方法步骤详情" step 3; ai.info "Methodology"
 * step 2). Per row, per aligned 32-column group g: the mask word has bit j set
 * when column 32g+j is kept; the kept values follow in ascending column order
 * at values[row][16g ...]. Every M-subgroup must keep exactly N, so every word
 * has 16 set bits.
 */
int oracle_pack(const uint16_t *W, int64_t rows, int64_t K, int N, int M, uint32_t *masks,
                uint16_t *values)
{
    if (!pattern_supported(N, M))
        return OR_UNSUPPORTED;
    if (!shape_ok(rows, K))
        return OR_BAD_SHAPE;
    if ((rows > 0 && K > 0) && (!W || !masks || !values))
        return OR_BAD_ARG;
    const int64_t words = K / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < words; ++g) {
            const uint16_t *w = W + r * K + 32 * g;
            int keep[32];
            for (int j = 0; j < 32; ++j)
                keep[j] = !bf16_is_zero(w[j]);
            for (int s = 0; s < 32 / M; ++s) {
                int count = 0;
                for (int j = s * M; j < (s + 1) * M; ++j)
                    count += keep[j];
                if (count > N)
                    return OR_NOT_NM;
                for (int j = s * M; j < (s + 1) * M && count < N; ++j) {
                    if (!keep[j]) {
                        keep[j] = 1;
                        count++;
                    }
                }
            }
            uint32_t mask = 0;
            int next = 0;
            uint16_t *v = values + r * (K / 2) + 16 * g;
            for (int j = 0; j < 32; ++j) {
                if (keep[j]) {
                    mask |= (uint32_t)1 << j;
                    v[next++] = w[j];
                }
            }
            masks[r * words + g] = mask;
        }
    }
    return OR_OK;
}

/*
 * Independent decoder of the bitmask format: walk the bits of each word from
 * the least significant upwards; a set bit takes the next stored value, a
 * clear bit is +0. A word without exactly 16 set bits is rejected.
 */
int oracle_unpack(const uint32_t *masks, const uint16_t *values, int64_t rows, int64_t K,
                  uint16_t *W)
{
    if (!shape_ok(rows, K))
        return OR_BAD_SHAPE;
    if ((rows > 0 && K > 0) && (!masks || !values || !W))
        return OR_BAD_ARG;
    const int64_t words = K / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < words; ++g) {
            uint32_t mask = masks[r * words + g];
            int bits = 0;
            for (int j = 0; j < 32; ++j)
                bits += (int)((mask >> j) & 1u);
            if (bits != 16)
                return OR_BAD_MASK;
            const uint16_t *v = values + r * (K / 2) + 16 * g;
            uint16_t *w = W + r * K + 32 * g;
            int next = 0;
            for (int j = 0; j < 32; ++j)
                w[j] = ((mask >> j) & 1u) ? v[next++] : (uint16_t)0;
        }
    }
    return OR_OK;
}

/*
 * The product the sparse kernel must reproduce: y[b][r] = sum_j W[r][j] x[b][j]
 * over the pruned dense W, in fp64, j in index order. Also returns
 * S[b][r] = sum_j |W[r][j] x[b][j]|, the scale of the fp32 tolerance.
 * bf16 x bf16 products are exact in fp64.
 */
int oracle_spmv_f64(const uint16_t *W, const uint16_t *x, int64_t rows, int64_t K, int batch,
                    double *y, double *S)
{
    if (!shape_ok(rows, K) || batch < 1)
        return OR_BAD_SHAPE;
    if (rows > 0 && (!W || !x || !y || !S))
        return OR_BAD_ARG;
    for (int b = 0; b < batch; ++b) {
        for (int64_t r = 0; r < rows; ++r) {
            double acc = 0.0, mag = 0.0;
            for (int64_t j = 0; j < K; ++j) {
                double p = (double)bf16_bits_to_float(W[r * K + j]) *
                           (double)bf16_bits_to_float(x[(int64_t)b * K + j]);
                acc += p;
                mag += fabs(p);
            }
            y[(int64_t)b * rows + r] = acc;
            S[(int64_t)b * rows + r] = mag;
        }
    }
    return OR_OK;
}

/*
 * SwiGLU of an MLP's gate and up products (the step after the SpMV in a
 * decode layer; the pages prune only the linear layers): h = silu(g) * u with
 * silu(g) = g / (1 + e^-g), all in fp64, elementwise over n values.
 */
int oracle_swiglu_f64(const double *g, const double *u, int64_t n, double *h)
{
    if (n < 0)
        return OR_BAD_SHAPE;
    if (n > 0 && (!g || !u || !h))
        return OR_BAD_ARG;
    for (int64_t i = 0; i < n; ++i)
        h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
    return OR_OK;
}

/*
 * The pair layout of a gate/up matrix: row block t (rows 32t .. 32t+31) holds
 * gate rows 16t .. 16t+15, then up rows 16t .. 16t+15. Copies bf16 bits.
 */
int oracle_pair_rows(const uint16_t *Wg, const uint16_t *Wu, int64_t rows_h, int64_t K, uint16_t *out)
{
    if (rows_h < 0 || K < 0 || rows_h % 16 != 0)
        return OR_BAD_SHAPE;
    if (rows_h > 0 && K > 0 && (!Wg || !Wu || !out))
        return OR_BAD_ARG;
    for (int64_t r = 0; r < rows_h; ++r) {
        const int64_t og = (r / 16) * 32 + r % 16, ou = og + 16;
        for (int64_t j = 0; j < K; ++j) {
            out[og * K + j] = Wg[r * K + j];
            out[ou * K + j] = Wu[r * K + j];
        }
    }
    return OR_OK;
}
