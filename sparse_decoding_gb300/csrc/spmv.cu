// spmv.cu -- bitmask N:M decode SpMV kernels for sm_103a.
//
// y[b][r] = sum_j W[r][j] x[b][j] with W stored as 32-bit masks plus the kept
// bf16 values (SparseDecoding: paper.rainbus.top summary, "核心方法" and
// "方法步骤详情" steps 3-4; ai.info summary, "Methodology in Plain English"
// steps 2-3). Each mask word has exactly 16 set bits, so every word takes the
// same 16 steps: find a set bit (its position is the column of the next kept
// value), clear it, multiply-accumulate. The pages walk from the least
// significant bit; here each word is walked from both ends at once (the
// highest remaining set bit gives values 15..8, the lowest values 0..7), two
// independent 8-step dependency chains over the same (column, value) pairs --
// the product is the same sum. Words whose bytes all hold four set bits (2:4,
// 4:8) take their columns from byte tables instead (batch 1 and 2).
//
// Main kernel (K % 128 == 0): the stream-K TMA driver of streamk.cuh with
// units of 32 rows x 128 columns (4 mask words per row). A stage is filled by
// three tensor copies: values (box 64 x 32 bf16, 128-byte swizzle), masks
// (box 4 x 32 u32) and the unit's 128-column slice of x (box 128 x batch).
//
// Lane i of a warp owns row i of the unit, so all 32 lanes read x inside the
// same 32-column window. At batch 1 lane j holds column j of that window in a
// register and the gather is a warp shuffle (at batch 2 the same, the two
// batch rows as one bf16 pair, for byte-regular words); otherwise the window
// is transposed to bf16 [column][batch] in shared memory and the gather is
// one conflict-free shared load per column (all batch rows).
//
// Fallback kernel (any K % 32 == 0): the same lane-per-row walk with plain
// loads from global memory.
#include "streamk.cuh"

namespace nm {

constexpr int kSpCols = 128;                    // columns per unit
constexpr int kSpWords = kSpCols / 32;          // mask words per row per unit
constexpr int kValBytes = kUnitRows * kSpCols;  // 32 rows x 64 bf16
constexpr int kMaskBytes = kUnitRows * kSpWords * 4;

// Load this lane's 4 mask words and 4 x 16 kept values of one unit.
__device__ __forceinline__ void load_row_unit(const uint8_t *st, int lane, uint32_t (&m)[4], uint32_t (&v)[4][8])
{
    const uint4 mw = *(const uint4 *)(st + kValBytes + lane * 16);
    m[0] = mw.x;
    m[1] = mw.y;
    m[2] = mw.z;
    m[3] = mw.w;
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
}

// Batch 1: 16 fixed steps over the 4 words, x gathered by warp shuffle.
// Each word is walked from both ends at once: step j takes the highest
// remaining set bit for value 15-j and the lowest remaining set bit for value
// j. The two walks touch disjoint bits, so they are independent dependency
// chains (the walk is bound by the latency of find-bit -> clear, not by
// issue). Each product is one mixed-precision FMA on the bf16 halves (x is
// shuffled as bf16), into one accumulator per walk; this ran 1.5% faster per
// layer than converting both weights of a step to fp32 for a packed fp32x2
// FMA.
__device__ __forceinline__ void walk_unit_b1(const uint32_t (&m)[4], const uint32_t (&v)[4][8], const uint8_t *sx, int lane,
                                             float (&acc)[4][1])
{
    uint32_t xr[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        xr[q] = *(const uint16_t *)(sx + (32 * q + lane) * 2); // bf16 in the low half
    uint32_t mh[4], ml[4];
    float ah[4], al[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        mh[q] = m[q];
        ml[q] = m[q];
        ah[q] = 0.f;
        al[q] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int ph = bfind_u32(mh[q]); // column of value 15-j (-1 only for a malformed word)
            mh[q] ^= bit_at(ph);
            const uint32_t t = ml[q] - 1u;
            const int pl = bfind_u32(ml[q] ^ t); // column of value j: the lowest set bit
            ml[q] &= t;
            const uint32_t xh = __shfl_sync(0xFFFFFFFFu, xr[q], ph), // lane index taken mod 32
                xl = __shfl_sync(0xFFFFFFFFu, xr[q], pl);
            const int kh = 15 - j, kl = j;
            if (kh & 1)
                ah[q] = fma_bf16<1, 0>(v[q][kh >> 1], xh, ah[q]);
            else
                ah[q] = fma_bf16<0, 0>(v[q][kh >> 1], xh, ah[q]);
            if (kl & 1)
                al[q] = fma_bf16<1, 0>(v[q][kl >> 1], xl, al[q]);
            else
                al[q] = fma_bf16<0, 0>(v[q][kl >> 1], xl, al[q]);
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
        acc[q][0] += ah[q] + al[q];
}

// Byte tables for byte-regular words. When every byte of a mask word has
// exactly four set bits -- always so for 2:4 and 4:8, whose M-subgroups sit
// inside a byte -- the kept values of byte b are values 4b..4b+3 of the word,
// so their columns can be looked up instead of walked: table b maps a byte
// value to four bytes 8b + (position of its k-th set bit), k = 0..3, which are
// directly the shuffle source lanes. A byte without four set bits maps to
// kIrregular (bit 7 of byte 0), which no regular entry has.
constexpr uint32_t kIrregular = 0x80u;
constexpr int kLutBytes = 4 * 256 * 4;

// Each CTA computes the four tables into its shared memory (a few dozen
// instructions per entry, no memory reads): a copy from global memory sat on
// the critical path of a CTA's start whenever HBM was busy with the previous
// kernel's traffic, and every CTA of the grid read the same 4 KB at once.
__device__ __forceinline__ void init_byte_tables(uint32_t *lut, int tid, int nthreads)
{
    for (int i = tid; i < 4 * 256; i += nthreads) {
        const uint32_t b = (uint32_t)i >> 8;
        uint32_t e = (uint32_t)i & 255u;
        uint32_t ent = kIrregular;
        if (__popc(e) == 4) {
            ent = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t j = (uint32_t)(__ffs(e) - 1); // position of the k-th set bit
                e &= e - 1;
                ent |= (8 * b + j) << (8 * k);
            }
        }
        lut[i] = ent;
    }
}

// Batch 1, byte-regular words: looked-up columns, x gathered by warp shuffle
// (a shuffle uses the low 5 bits of its source lane, so the other bytes of a
// table entry need no masking). Returns false, having accumulated nothing, if
// any lane of the warp holds a word that is not byte-regular.
__device__ __forceinline__ bool walk_unit_b1_lut(const uint32_t (&m)[4], const uint32_t (&v)[4][8], const uint8_t *sx,
                                                 const uint32_t *lut, int lane, float (&acc)[4][1])
{
    uint32_t ent[4][4];
    uint32_t flags = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            ent[q][b] = lut[b * 256 + ((m[q] >> (8 * b)) & 0xFFu)];
            flags |= ent[q][b];
        }
    if (!__all_sync(0xFFFFFFFFu, (flags & kIrregular) == 0))
        return false;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        // x stays bf16 (low half); one mixed-precision FMA per product
        const uint32_t xr = *(const uint16_t *)(sx + (32 * q + lane) * 2);
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t e = ent[q][b];
            const uint32_t p0 = v[q][2 * b], p1 = v[q][2 * b + 1];
            a0 = fma_bf16<0, 0>(p0, __shfl_sync(0xFFFFFFFFu, xr, (int)e), a0);
            a1 = fma_bf16<1, 0>(p0, __shfl_sync(0xFFFFFFFFu, xr, (int)(e >> 8)), a1);
            a0 = fma_bf16<0, 0>(p1, __shfl_sync(0xFFFFFFFFu, xr, (int)(e >> 16)), a0);
            a1 = fma_bf16<1, 0>(p1, __shfl_sync(0xFFFFFFFFu, xr, (int)(e >> 24)), a1);
        }
        acc[q][0] += a0 + a1;
    }
    return true;
}

// Batch 2, byte-regular words: the byte tables give each kept value's
// column as a shuffle source lane, as at batch 1. Lane j holds column
// 32 q + j of the unit's x slice for every batch row, as bf16 pairs (rows 2h
// and 2h + 1 in xq[h]), so one shuffle gathers two batch rows and no window
// is transposed. Returns false, having accumulated nothing, if any lane of the
// warp holds a word that is not byte-regular.
template <int B>
__device__ __forceinline__ bool walk_unit_bn_lut(const uint32_t (&m)[4], const uint32_t (&v)[4][8],
                                                 const uint8_t *sx, const uint32_t *lut, int lane,
                                                 float (&acc)[4][B])
{
    constexpr int H = (B + 1) / 2; // registers of bf16 pairs per column
    uint32_t ent[4][4];
    uint32_t flags = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            ent[q][b] = lut[b * 256 + ((m[q] >> (8 * b)) & 0xFFu)];
            flags |= ent[q][b];
        }
    if (!__all_sync(0xFFFFFFFFu, (flags & kIrregular) == 0))
        return false;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t xq[H];
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const uint32_t lo = *(const uint16_t *)(sx + (2 * h) * (kSpCols * 2) + (32 * q + lane) * 2);
            const uint32_t hi =
                2 * h + 1 < B ? *(const uint16_t *)(sx + (2 * h + 1) * (kSpCols * 2) + (32 * q + lane) * 2) : 0u;
            xq[h] = lo | (hi << 16);
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t e = ent[q][b];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t wp = v[q][2 * b + (k >> 1)]; // values 4b + k: pair k / 2, half k % 2
                const int src = (int)(e >> (8 * k));          // a shuffle reads the low 5 bits
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const uint32_t xv = __shfl_sync(0xFFFFFFFFu, xq[h], src);
                    if (k & 1) {
                        acc[q][2 * h] = fma_bf16<1, 0>(wp, xv, acc[q][2 * h]);
                        if (2 * h + 1 < B)
                            acc[q][(2 * h + 1) % B] = fma_bf16<1, 1>(wp, xv, acc[q][(2 * h + 1) % B]);
                    } else {
                        acc[q][2 * h] = fma_bf16<0, 0>(wp, xv, acc[q][2 * h]);
                        if (2 * h + 1 < B)
                            acc[q][(2 * h + 1) % B] = fma_bf16<0, 1>(wp, xv, acc[q][(2 * h + 1) % B]);
                    }
                }
            }
        }
    }
    return true;
}

// x slice of one unit, bf16 [B][128] (as copied) -> bf16 [128][BP] in the
// warp's window: the batch rows of a column side by side, two per 32-bit word.
template <int B>
__device__ __forceinline__ void transpose_x_bf16(const uint8_t *sx, uint8_t *xb, int lane)
{
    constexpr int BP = BatchPad<B>::value;
#pragma unroll
    for (int i = 0; i < kSpCols / 32; ++i) {
        const int c = lane + 32 * i;
        uint32_t h[BP];
#pragma unroll
        for (int b = 0; b < BP; ++b)
            h[b] = (b < B) ? *(const uint16_t *)(sx + b * (kSpCols * 2) + c * 2) : 0u;
        uint8_t *dst = xb + c * BP * 2;
        if (BP == 2) {
            *(uint32_t *)dst = h[0] | (h[1 % BP] << 16);
        } else if (BP == 4) {
            *(uint2 *)dst = make_uint2(h[0] | (h[1 % BP] << 16), h[2 % BP] | (h[3 % BP] << 16));
        } else {
            *(uint4 *)dst = make_uint4(h[0] | (h[1 % BP] << 16), h[2 % BP] | (h[3 % BP] << 16),
                                       h[4 % BP] | (h[5 % BP] << 16), h[6 % BP] | (h[7 % BP] << 16));
        }
    }
}

// acc[b] += w * x[col][b] for the batch rows: w is the WH half of `wp`, x the
// bf16 window row at `xa`; one mixed-precision FMA per product.
template <int B, int WH>
__device__ __forceinline__ void fma_window_bf16(uint32_t wp, const uint8_t *xa, float (&acc)[B])
{
    constexpr int BP = BatchPad<B>::value;
    uint32_t xw[BP / 2];
    if (BP == 2) {
        xw[0] = *(const uint32_t *)xa;
    } else if (BP == 4) {
        const uint2 t = *(const uint2 *)xa;
        xw[0] = t.x;
        xw[1 % (BP / 2)] = t.y;
    } else {
        const uint4 t = *(const uint4 *)xa;
        xw[0] = t.x;
        xw[1 % (BP / 2)] = t.y;
        xw[2 % (BP / 2)] = t.z;
        xw[3 % (BP / 2)] = t.w;
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
        if (b & 1)
            acc[b] = fma_bf16<WH, 1>(wp, xw[b >> 1], acc[b]);
        else
            acc[b] = fma_bf16<WH, 0>(wp, xw[b >> 1], acc[b]);
    }
}

// Batch > 1: the same two-ended walk, x from the bf16 [column][batch] window.
template <int B>
__device__ __forceinline__ void walk_unit_bn(const uint32_t (&m)[4], const uint32_t (&v)[4][8], const uint8_t *xb,
                                             int lane, float (&acc)[4][B])
{
    constexpr int BP = BatchPad<B>::value;
    uint32_t mh[4], ml[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        mh[q] = m[q];
        ml[q] = m[q];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int ph = bfind_u32(mh[q]); // -1 only for a malformed word: reads the guard band
            mh[q] ^= bit_at(ph);
            const uint32_t t = ml[q] - 1u;
            const int pl = bfind_u32(ml[q] ^ t);
            ml[q] &= t;
            constexpr int kh = 15, kl = 0;
            const uint32_t vh = v[q][(kh - j) >> 1], vl = v[q][(kl + j) >> 1];
            const uint8_t *xh = xb + (q * 32 + ph) * BP * 2, *xl = xb + (q * 32 + pl) * BP * 2;
            if (((kh - j) & 1) != 0)
                fma_window_bf16<B, 1>(vh, xh, acc[q]);
            else
                fma_window_bf16<B, 0>(vh, xh, acc[q]);
            if (((kl + j) & 1) != 0)
                fma_window_bf16<B, 1>(vl, xl, acc[q]);
            else
                fma_window_bf16<B, 0>(vl, xl, acc[q]);
        }
    }
}

// The sparse unit: masks + values + x slice per stage.
struct SparseUnit {
    static constexpr int kCols = kSpCols;
    static constexpr bool kHasMasks = true;
    template <int B> static constexpr int stage_bytes() { return (kValBytes + kMaskBytes + 1023) / 1024 * 1024; }
    template <int B> static constexpr int x_bytes() { return 2 * kCols * B; }
    template <int B> static constexpr uint32_t tx_bytes() { return kValBytes + kMaskBytes + x_bytes<B>(); }
    template <int B> static constexpr int xf_bytes() { return B == 1 ? 0 : kCols * BatchPad<B>::value * 2; }

    static __device__ __forceinline__ void issue_weights(uint32_t st, uint32_t bar, int kc, int32_t row0,
                                                         uint64_t pol, const TensorMaps &maps)
    {
        tma_load_2d_hint(st, &maps.w, kc * (kCols / 2), row0, bar, pol);
        tma_load_2d_hint(st + kValBytes, &maps.m, kc * kSpWords, row0, bar, pol);
    }

    static constexpr int kSharedBytes = kLutBytes;
    // Per-warp state: whether to try the byte tables. A warp that meets a
    // unit with an irregular word (8:16, 16:32 data) stops trying.
    struct State {
        bool try_lut;
    };
    static __device__ __forceinline__ State initial_state() { return State{true}; }
    static __device__ __forceinline__ void init_shared(uint8_t *p, int tid, int nthreads)
    {
        init_byte_tables((uint32_t *)p, tid, nthreads);
    }

    // One lane's row of the unit: its 4 mask words and 4 x 16 kept values.
    template <int B> struct Regs {
        uint32_t m[4];
        uint32_t v[4][8];
    };
    template <int B> static __device__ __forceinline__ void load(const uint8_t *stp, int lane, Regs<B> &r)
    {
        load_row_unit(stp, lane, r.m, r.v);
    }

    template <int B>
    static __device__ __forceinline__ void compute(const Regs<B> &r, const uint8_t *xs, uint8_t *xf,
                                                   const uint8_t *ps, State &stt, int lane, float (&acc)[4][B])
    {
        if constexpr (B == 1) {
            if (stt.try_lut) {
                if (walk_unit_b1_lut(r.m, r.v, xs, (const uint32_t *)ps, lane, acc))
                    return;
                stt.try_lut = false;
            }
            walk_unit_b1(r.m, r.v, xs, lane, acc);
        } else {
            // batch 2: byte tables with shuffled x; wider batches need a shuffle
            // per bf16 pair of batch rows per kept value, which costs more than
            // the walk's shared-memory window (batch 4 even, batch 8 -12%)
            if constexpr (B <= 2) {
                if (stt.try_lut) {
                    if (walk_unit_bn_lut<B>(r.m, r.v, xs, (const uint32_t *)ps, lane, acc))
                        return;
                    stt.try_lut = false;
                }
            }
            transpose_x_bf16<B>(xs, xf, lane);
            __syncwarp();
            walk_unit_bn<B>(r.m, r.v, xf, lane, acc);
        }
    }
};

// Warps per CTA by batch size (2 stage buffers per warp, 2 CTAs per SM).
template <int B> struct SparseCfg {
    static constexpr int W = B <= 2 ? 8 : B <= 4 ? 6 : 4;
    static constexpr int NBUF = 2;
    static constexpr int MINB = 2;
};

// ---------------------------------------------------------------------------
// Fallback: lane-per-row walk with plain global loads (any K % 32 == 0).
// ---------------------------------------------------------------------------
template <int B, int OUT>
__global__ void __launch_bounds__(256)
    spmv_simple_kernel(const uint32_t *__restrict__ masks, const uint16_t *__restrict__ values,
                       const uint16_t *__restrict__ x, const StreamKParams out, int64_t K)
{
    const int64_t rows = out.rows;
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
        store_y<B, OUT>(out, row, acc);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

int spmv_max_ctas(int num_sms)
{
    int m = 1; // the 16-warp shape runs one CTA per SM
    m = std::max(m, SparseCfg<1>::MINB);
    m = std::max(m, SparseCfg<2>::MINB);
    m = std::max(m, SparseCfg<4>::MINB);
    m = std::max(m, SparseCfg<8>::MINB);
    return std::min(num_sms * m, kMaxCtas);
}

SpmvPath spmv_path(int64_t rows, int64_t K)
{
    if (K % kSpCols == 0 && K > 0 && rows > 0 && rows <= 0x7FFFFFFF && K <= 0x7FFFFFFF)
        return kSpmvTma;
    return kSpmvSimple;
}

// Tensor maps of one sparse linear: values (box 64 x 32 bf16, 128-byte
// swizzle), masks (box 4 x 32 u32), x (box 128 x B bf16).
template <int B>
static nm_status encode_sparse_maps(const uint32_t *masks, const void *values, const void *x, int64_t rows, int64_t K,
                                    TensorMaps *maps)
{
    nm_status s;
    if ((s = encode_2d(&maps->w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, values, (uint64_t)K / 2, (uint64_t)rows,
                       (uint64_t)K, kSpCols / 2, kUnitRows, CU_TENSOR_MAP_SWIZZLE_128B)) != NM_OK)
        return s;
    if ((s = encode_2d(&maps->m, CU_TENSOR_MAP_DATA_TYPE_UINT32, masks, (uint64_t)K / 32, (uint64_t)rows,
                       (uint64_t)K / 8, kSpWords, kUnitRows, CU_TENSOR_MAP_SWIZZLE_NONE)) != NM_OK)
        return s;
    return encode_2d(&maps->x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)B, (uint64_t)K * 2,
                     kSpCols, B, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int B, int OUT>
static nm_status launch_tma(const uint32_t *masks, const void *values, const void *x, void *y, int64_t rows,
                            int64_t K, const LaunchCtx &ctx)
{
    TensorMaps maps;
    nm_status s = encode_sparse_maps<B>(masks, values, x, rows, K, &maps);
    if (s != NM_OK)
        return s;
    const int64_t nrb = (rows + kUnitRows - 1) / kUnitRows, KC = K / kSpCols;
    if constexpr (B <= 2) {
        // Few, long row blocks (at most one per SM, 64+ units each): one CTA
        // of 16 warps per row block halves each warp's share of it -- unless,
        // at batch 1, CTA pairs can split the row blocks' K instead: that
        // halves the share as well and also puts the SMs to work that whole
        // row blocks would leave idle (down of the 8B stack: 128 row blocks,
        // 152 SMs; -5% per layer).
        const bool pairs = B == 1 && pair_split_ok<SparseCfg<1>::W, SparseCfg<1>::MINB>(nrb, KC, ctx.num_sms);
        if (!pairs && nrb <= ctx.num_sms && KC >= 64 && choose_split(nrb, KC, 16, 1, ctx.num_sms).whole)
            return launch_streamk<SparseUnit, B, 16, 2, 1, OUT>(maps, y, rows, KC, ctx);
    }
    return launch_streamk<SparseUnit, B, SparseCfg<B>::W, SparseCfg<B>::NBUF, SparseCfg<B>::MINB, OUT>(
        maps, y, rows, KC, ctx);
}

template <int B, int OUT>
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
    StreamKParams out = {}; // the output fields only
    out.y = y;
    out.rows = rows;
    out.y_k = ctx.y_k;
    out.y_v = ctx.y_v;
    out.rows_q = ctx.rows_q;
    out.rows_qk = ctx.rows_q + ctx.rows_k;
    if (cudaLaunchKernelEx(&cfg, spmv_simple_kernel<B, OUT>, masks, (const uint16_t *)values,
                           (const uint16_t *)x, out, K) != cudaSuccess)
        return NM_ERR_CUDA;
    return NM_OK;
}

template <int OUT>
static nm_status dispatch(const uint32_t *masks, const void *values, const void *x, void *y, int64_t rows,
                          int64_t K, int batch, const LaunchCtx &ctx)
{
    const bool tma = spmv_path(rows, K) == kSpmvTma;
#define NM_CASE(BB)                                                                                         \
    case BB:                                                                                                \
        return tma ? launch_tma<BB, OUT>(masks, values, x, y, rows, K, ctx)                              \
                   : launch_simple<BB, OUT>(masks, values, x, y, rows, K, ctx);
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
// The persistent stack kernel over sparse linears
// ---------------------------------------------------------------------------

template <int B>
using SparseStack = StackLauncher<SparseUnit, B, SparseCfg<B>::W, SparseCfg<B>::NBUF, SparseCfg<B>::MINB>;

nm_status stack_grid_sparse(int batch, int num_sms, int *ctas)
{
    return with_batch(batch, [&](auto bc) { return SparseStack<decltype(bc)::value>::grid(num_sms, ctas); });
}

nm_status stack_encode_sparse(const nm_linear &op, int batch, int ctas, StackOp *out)
{
    return with_batch(batch, [&](auto bc) {
        constexpr int B = decltype(bc)::value;
        nm_status s = encode_sparse_maps<B>(op.masks, op.values, op.x, op.rows, op.K, &out->maps);
        if (s == NM_OK)
            SparseStack<B>::split(out, op.y, op.rows, op.K / kSpCols, ctas);
        return s;
    });
}

nm_status stack_launch_sparse(const StackOp *ops, int n_ops, int batch, uint32_t *gbar, int ctas,
                              const LaunchCtx &ctx)
{
    return with_batch(batch, [&](auto bc) {
        return SparseStack<decltype(bc)::value>::launch(ops, n_ops, gbar, ctas, ctx);
    });
}

nm_status launch_spmv(const uint32_t *masks, const void *values, const void *x, void *y, int out, int64_t rows,
                      int64_t K, int batch, const LaunchCtx &ctx)
{
    switch (out) {
    case kOutBf16: return dispatch<kOutBf16>(masks, values, x, y, rows, K, batch, ctx);
    case kOutF32: return dispatch<kOutF32>(masks, values, x, y, rows, K, batch, ctx);
    case kOutSwiglu: return dispatch<kOutSwiglu>(masks, values, x, y, rows, K, batch, ctx);
    case kOutQkv: return dispatch<kOutQkv>(masks, values, x, y, rows, K, batch, ctx);
    default: return NM_ERR_INVALID_ARG;
    }
}

} // namespace nm
