// tc_gemm.cu -- the GEMM-shaped steps of the OBS pruning on the 5th-generation
// tensor cores (tcgen05), with the operands staged by TMA and the accumulator
// in tensor memory.
//
//   C = alpha * A * B^T + beta * C     A: bf16 [M][k], B: bf16 [N][k] (rows
//                                      contiguous along k), C: fp32 [M][N]
//
// The kernel is persistent (one CTA per SM) and computes 128 x 128 tiles of
// C in turn: warp 0 (one thread) streams k-slices of A and B into a ring of
// shared-memory stages by TMA; warp 1 (one thread) issues M=128, N=128, K=16
// tcgen05.mma into 128-column fp32 accumulators in tensor memory (four of
// them, see below) and releases each stage with tcgen05.commit; warps 2-5
// read a finished tile's accumulators with tcgen05.ld (one row per thread),
// add them, hand the tensor memory back to the MMA warp, and then write C --
// so the next tile's loads and MMAs overlap the stores.
//
// fp32 products (the Cholesky steps and the lazy update) are emulated with
// bf16 parts: a = a0 + a1 + a2 with a0 = bf16(a), a1 = bf16(a - a0),
// a2 = bf16(a - a0 - a1) (together 24 bits of a's significand), and
//   a b ~ a0 b0 + a0 b1 + a1 b0 + a0 b2 + a1 b1 + a2 b0
// -- every product of order up to 2 -- accumulated in fp32; the dropped terms
// are below 2^-24 |a b|. split_kernel writes the three parts of a fp32 matrix
// side by side per 64-column k-tile ([rows][k-tiles][part][64] bf16, the same
// layout for A and B), so a pipeline stage holds the three part tiles of A
// and of B for a slice of k, and the six products are six groups of MMAs on
// them: every operand byte crosses from L2 to shared memory once. The leading
// products a0 b0 of successive k-tiles take turns in three tensor-memory
// accumulators and the five smaller ones go to a fourth; the four are added
// once at the end, in a fixed order. The tensor cores' accumulation loses
// more than fp32 rounding as k grows (in one accumulator, the mean error at
// k = 2048 was 2.8 times that of fp32 on the CUDA cores); spreading k over
// several accumulators keeps each sum shorter. The Hessian's operand (bf16
// calibration inputs, transposed) has one part: its products are exact, and
// its k-tiles take turns in all four accumulators.
//
// Structure flags skip what is known to be zero or not needed: a triangular
// operand limits each tile's k range, a C whose upper part nobody reads
// skips the tiles above the diagonal, and a symmetric C computes the tiles on
// and below the diagonal and writes each off-diagonal one twice (once
// transposed, which stays coalesced: lanes hold consecutive rows).
//
// Every wait is bounded (about a second); a wait that runs out sets a flag the
// host reads, and the kernel still frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kernels.h"

namespace nm {
namespace {

constexpr int kTcM = 128;        // rows of C per CTA (tensor-memory lanes)
constexpr int kTcN = 128;        // columns of C per CTA (tensor-memory columns)
constexpr int kTcK = 64;         // k per part tile in the operand layout
constexpr int kTcThreads = 192;  // producer, MMA issuer, four epilogue warps
constexpr int kTcAcc = 4;        // 128-column accumulators (all 512 tensor-memory columns)

// A pipeline stage holds NP part tiles of A and NP of B, each KW columns of
// k wide (KW = 64: 128-byte rows, 128-byte swizzle; KW = 32: 64-byte rows,
// 64-byte swizzle), in a ring of S stages.
template <int NP, int KW> struct TcCfg {
    static constexpr int kTile = kTcM * KW * 2;                    // bytes of one part tile
    static constexpr int kStage = 2 * NP * kTile;
    static constexpr int kStages = (192 * 1024) / kStage;          // 2..12
    static constexpr int kSmem = kStages * kStage + 1024;          // + alignment slack
    static constexpr int kSub = kTcK / KW;                         // stages per 64-wide k-tile
    static constexpr int kSlices = KW / 16;                        // K=16 MMAs per part pair and stage
    static constexpr int kSwizzleBytes = KW * 2;
};

// ---- tensor-memory and tensor-core instructions (PTX ISA, tcgen05) ----------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (tensor memory) (+)= A (shared, descriptor) * B (shared, descriptor)^T
__device__ __forceinline__ void tc_mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
                 : "memory");
}
// Arrive on an mbarrier once every tcgen05.mma issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                   "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
                   "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
                   "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with a
// SW-byte swizzle (SW = 128 or 64): rows of SW bytes, 8-row groups 8 SW
// bytes apart (the stride byte offset), start address in 16-byte units,
// descriptor version 1, layout type 2 (128-byte swizzle) or 4 (64-byte). The
// leading byte offset is not used by these layouts. The tile starts on a
// 1024-byte boundary (base offset 0); a k-slice of 16 elements inside it
// starts 32 bytes further per slice.
template <int SW> __device__ __forceinline__ uint64_t smem_desc_sw(uint32_t saddr)
{
    static_assert(SW == 128 || SW == 64, "swizzle width");
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;                     // leading byte offset (unused): 16 bytes
    d |= (uint64_t)((8 * SW) >> 4) << 32;       // stride byte offset: 8 rows
    d |= (uint64_t)1 << 46;                     // descriptor version
    d |= (uint64_t)(SW == 128 ? 2 : 4) << 61;   // swizzle mode
    return d;
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, both K-major,
// M = 128, N = 128.
constexpr uint32_t kIdescBf16 = (1u << 4)               // D format: fp32
                                | (1u << 7)             // A format: bf16
                                | (1u << 10)            // B format: bf16
                                | ((kTcN >> 3) << 17)   // N / 8
                                | ((kTcM >> 4) << 24);  // M / 16

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint32_t *status)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, 1u << NM_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// The products of one k-tile with three parts, leading one first:
// a0 b0, a0 b1, a1 b0, a0 b2, a1 b1, a2 b0 (two bits per product: the part).
constexpr uint32_t kPartA = 0u | (0u << 2) | (1u << 4) | (0u << 6) | (1u << 8) | (2u << 10);
constexpr uint32_t kPartB = 0u | (1u << 2) | (0u << 4) | (2u << 6) | (1u << 8) | (0u << 10);
template <int NP> constexpr int kProducts = NP == 1 ? 1 : 6;

// The accumulator of product q of the tile's u-th 64-wide k-tile. One part:
// the k-tiles take turns in all four. Three: the leading products take turns
// in accumulators 0..2, the other five all go to accumulator 3.
__host__ __device__ constexpr int tc_acc(int u, int q, int np)
{
    return np == 1 ? u % kTcAcc : (q == 0 ? u % (kTcAcc - 1) : kTcAcc - 1);
}
// The accumulators that receive a product when a tile runs n k-tiles.
__device__ __forceinline__ uint32_t tc_used(int n, int np)
{
    if (n <= 0)
        return 0;
    if (np == 1)
        return (1u << (n < kTcAcc ? n : kTcAcc)) - 1;
    return ((1u << (n < kTcAcc - 1 ? n : kTcAcc - 1)) - 1) | (1u << (kTcAcc - 1));
}

struct TcMaps {
    CUtensorMap a;  // bf16 [M][kt * NP * 64], box KW x 128
    CUtensorMap b;  // bf16 [N][kt * NP * 64], box KW x 128
};

// One 32-column slice of a finished tile row: C[row][n0+c ..] = alpha v +
// beta C (v = 0 when the tile had no k range), and with `mirror` also
// C[n0+c+j][row] (the transposed tile; lanes hold consecutive rows, so each
// of those 32 stores is one coalesced 128-byte line).
__device__ __forceinline__ void tc_store32(float *C, int64_t ldc, int row, int col, int M, int N, const float (&v)[32],
                                           float alpha, float beta, bool mirror)
{
    if (row >= M || col >= N)
        return;
    float *dst = C + (int64_t)row * ldc + col;
    const int ncol = N - col < 32 ? N - col : 32; // a multiple of 4
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        if (j < ncol) {
            float4 o = make_float4(alpha * v[j], alpha * v[j + 1], alpha * v[j + 2], alpha * v[j + 3]);
            if (beta != 0.f) {
                const float4 c = *(const float4 *)(dst + j);
                o.x = fmaf(beta, c.x, o.x);
                o.y = fmaf(beta, c.y, o.y);
                o.z = fmaf(beta, c.z, o.z);
                o.w = fmaf(beta, c.w, o.w);
            }
            *(float4 *)(dst + j) = o;
        }
    }
    if (mirror) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j < ncol) {
                float *t = C + (int64_t)(col + j) * ldc + row;
                *t = beta != 0.f ? fmaf(beta, *t, alpha * v[j]) : alpha * v[j];
            }
        }
    }
}

// One tile of C and its 64-wide k-tiles [t_lo, t_lo + nt) (global k =
// k_base + 64 t); nt = 0 for a tile with no k range (C = beta C). Tiles are
// numbered row by row, columns fastest; for a lower or symmetric C only the
// tiles on and below the diagonal are numbered (tile i of row `by` is the
// tile with by (by + 1) / 2 <= i < (by + 1) (by + 2) / 2).
struct TcTile {
    int m0, n0, t_lo, nt;
    bool mirror;
};
__host__ __device__ __forceinline__ bool tc_triangular(uint32_t flags) { return (flags & (kTcCLower | kTcCSym)) != 0; }
__device__ __forceinline__ TcTile tc_tile(int tile, int tiles_n, int ktiles, int64_t k_base, uint32_t flags)
{
    TcTile T;
    int bx, by;
    if (tc_triangular(flags)) {
        by = (int)((sqrtf(8.0f * (float)tile + 1.0f) - 1.0f) * 0.5f);
        while ((int64_t)by * (by + 1) / 2 > tile)
            --by;
        while ((int64_t)(by + 1) * (by + 2) / 2 <= tile)
            ++by;
        bx = tile - (int)((int64_t)by * (by + 1) / 2);
    } else {
        bx = tile % tiles_n;
        by = tile / tiles_n;
    }
    T.n0 = bx * kTcN;
    T.m0 = by * kTcM;
    T.mirror = (flags & kTcCSym) && bx < by;
    int64_t lo = k_base, hi = k_base + (int64_t)ktiles * kTcK;
    if ((flags & kTcALower) && hi > (int64_t)T.m0 + kTcM)
        hi = (int64_t)T.m0 + kTcM;
    if ((flags & kTcBLower) && hi > (int64_t)T.n0 + kTcN)
        hi = (int64_t)T.n0 + kTcN;
    if ((flags & kTcBUpper) && lo < (int64_t)T.n0)
        lo = (int64_t)T.n0;
    T.t_lo = lo < hi ? (int)((lo - k_base) / kTcK) : 0;
    T.nt = lo < hi ? (int)((hi - k_base + kTcK - 1) / kTcK) - T.t_lo : 0;
    return T;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Persistent: each CTA takes tiles blockIdx.x, blockIdx.x + gridDim.x, ...
// Warp 0 (one thread) streams the k-slices of every tile through the stage
// ring, warp 1 (one thread) issues the MMAs, warps 2-5 are the epilogue (warp
// w reads tensor-memory lanes 32 (w % 4) .. + 31). The epilogue copies a
// tile's sums into registers, hands the accumulators back (acc_empty) and
// only then writes C, so the next tile's MMAs, and the loads ahead of them,
// overlap the stores.
template <int NP, int KW>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ TcMaps maps, float *C, int64_t ldc, int M, int N, int ktiles,
                   int64_t k_base, uint32_t flags, float alpha, float beta, uint32_t *err)
{
    using Cfg = TcCfg<NP, KW>;
    constexpr int S = Cfg::kStages;
    __shared__ __align__(8) uint64_t full_bar[S];
    __shared__ __align__(8) uint64_t empty_bar[S];
    __shared__ __align__(8) uint64_t acc_full;   // a tile's MMAs are done
    __shared__ __align__(8) uint64_t acc_empty;  // the epilogue has read a tile's accumulators
    __shared__ uint32_t tmem_base;
    extern __shared__ __align__(1024) uint8_t dsmem[];
    uint8_t *const tiles = dsmem + ((1024u - (smem_addr(dsmem) & 1023u)) & 1023u);
    const uint32_t tiles0 = smem_addr(tiles);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_n = (N + kTcN - 1) / kTcN;
    const int ntiles = tc_triangular(flags) ? tiles_n * (tiles_n + 1) / 2 : tiles_n * ((M + kTcM - 1) / kTcM);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(&full_bar[s]), 1);
            mbar_init(smem_addr(&empty_bar[s]), 1);
        }
        mbar_init(smem_addr(&acc_full), 1);
        mbar_init(smem_addr(&acc_empty), 4); // one arrival per epilogue warp
        fence_mbar_init();
    }
    if (warp == 2)
        tmem_alloc(smem_addr(&tmem_base), kTcAcc * kTcN); // four 128-column fp32 accumulators
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    pdl_wait_upstream(); // the operands and C may be the previous kernels' output
    pdl_launch_dependents();

    // a wait that ran out marks the thread dead: its later waits poll once
    bool dead = false;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (dead)
            return mbar_try_wait(bar, parity);
        if (!wait_bounded(bar, parity, err))
            dead = true;
        return !dead;
    };

    if (warp == 0) {
        if (lane == 0) {
            // producer: the CTA's g-th stage goes to slot g % S once the MMAs of stage g - S released it
            uint32_t g = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                const TcTile T = tc_tile(tile, tiles_n, ktiles, k_base, flags);
                for (int i = 0; i < T.nt * Cfg::kSub; ++i, ++g) {
                    const int s = (int)(g % S);
                    if (g >= (uint32_t)S && !wait(smem_addr(&empty_bar[s]), ((g / S) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_addr(&full_bar[s]);
                    mbar_arrive_expect_tx(fb, Cfg::kStage);
                    const uint32_t sa = tiles0 + s * Cfg::kStage;
                    const int t = T.t_lo + i / Cfg::kSub, x0 = (i % Cfg::kSub) * KW;
#pragma unroll
                    for (int p = 0; p < NP; ++p) {
                        const int x = (t * NP + p) * kTcK + x0;
                        tma_load_2d(sa + p * Cfg::kTile, &maps.a, x, T.m0, fb);
                        tma_load_2d(sa + (NP + p) * Cfg::kTile, &maps.b, x, T.n0, fb);
                    }
                }
            }
            // before leaving, let the copies that may still be in flight land (bounded)
            for (uint32_t i = g > (uint32_t)S ? g - S : 0; i < g; ++i)
                if (!wait(smem_addr(&full_bar[i % S]), (i / S) & 1))
                    break;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // MMA issuer; j counts the tiles that had a k range
            uint32_t g = 0, j = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                const TcTile T = tc_tile(tile, tiles_n, ktiles, k_base, flags);
                if (T.nt == 0)
                    continue;
                if (j > 0 && !wait(smem_addr(&acc_empty), (j - 1) & 1)) // the epilogue has the last tile's sums
                    break;
                tc_fence_after();
                uint32_t touched = 0;
                for (int i = 0; i < T.nt * Cfg::kSub; ++i, ++g) {
                    const int s = (int)(g % S);
                    if (!wait(smem_addr(&full_bar[s]), (g / S) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = tiles0 + s * Cfg::kStage, sb = sa + NP * Cfg::kTile;
                    const int u = i / Cfg::kSub;
#pragma unroll
                    for (int q = 0; q < kProducts<NP>; ++q) {
                        const int pa = (kPartA >> (2 * q)) & 3, pb = (kPartB >> (2 * q)) & 3;
                        const int a = tc_acc(u, q, NP);
                        const uint32_t acc = tmem + (uint32_t)(a * kTcN);
#pragma unroll
                        for (int k = 0; k < Cfg::kSlices; ++k) {
                            const uint64_t ad = smem_desc_sw<Cfg::kSwizzleBytes>(sa + pa * Cfg::kTile + k * 32);
                            const uint64_t bd = smem_desc_sw<Cfg::kSwizzleBytes>(sb + pb * Cfg::kTile + k * 32);
                            tc_mma_bf16(acc, ad, bd, kIdescBf16, ((touched >> a) & 1u) | (k > 0 ? 1u : 0u));
                        }
                        touched |= 1u << a;
                    }
                    tc_commit(smem_addr(&empty_bar[s])); // the stage is free once these MMAs are done
                }
                tc_commit(smem_addr(&acc_full)); // the tile's accumulators are complete once its MMAs are done
                ++j;
            }
        }
    } else {
        // epilogue: warp w handles tensor-memory lanes (rows) 32 (w % 4) .. + 31
        const int qw = warp & 3;
        uint32_t j = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            const TcTile T = tc_tile(tile, tiles_n, ktiles, k_base, flags);
            const int row = T.m0 + qw * 32 + lane;
            if (T.nt == 0) {
                // no k range: C = beta C (nothing to do when beta is 1)
                if (beta != 1.0f) {
                    const float zero[32] = {};
#pragma unroll 1
                    for (int c = 0; c < kTcN; c += 32)
                        tc_store32(C, ldc, row, T.n0 + c, M, N, zero, alpha, beta, T.mirror);
                }
                continue;
            }
            const bool have = wait(smem_addr(&acc_full), j & 1);
            tc_fence_after();
            // the accumulators that received a product, added in index order
            const uint32_t used = tc_used(T.nt, NP);
            float v[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(qw * 32) << 16) + (uint32_t)(c * 32), r);
#pragma unroll 1
                for (int a = 1; a < kTcAcc; ++a) {
                    if (!(used & (1u << a)))
                        continue;
                    uint32_t r2[32];
                    tmem_ld32(tmem + ((uint32_t)(qw * 32) << 16) + (uint32_t)(a * kTcN + c * 32), r2);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(r2[e]));
                }
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    v[c][e] = have ? __uint_as_float(r[e]) : 0.0f;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&acc_empty)); // the MMAs of the next tile may start
            ++j;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tc_store32(C, ldc, row, T.n0 + 32 * c, M, N, v[c], alpha, beta, T.mirror);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2)
        tmem_dealloc(tmem, kTcAcc * kTcN);
}

// ---- operand preparation ------------------------------------------------------

// The bf16 parts of a fp32 value: a0 = bf16(a), a1 = bf16(a - a0),
// a2 = bf16(a - a0 - a1) (each difference exact in fp32).
__device__ __forceinline__ void split3(float a, uint16_t &p0, uint16_t &p1, uint16_t &p2)
{
    p0 = f32_to_bf16_rn(a);
    const float r1 = a - __uint_as_float((uint32_t)p0 << 16);
    p1 = f32_to_bf16_rn(r1);
    const float r2 = r1 - __uint_as_float((uint32_t)p1 << 16);
    p2 = f32_to_bf16_rn(r2);
}

// One operand to split: S fp32 with row stride lds, read as S[r][c] (or,
// transposed, S[c][r]) for rows x k, into out.
struct SplitOp {
    const float *S;
    int64_t lds;
    int rows, trans;
    uint16_t *out;
};

// Out [rows][kt][3][64] bf16: for row r and k-tile t, the three parts of S's
// elements (r, 64 t .. 64 t + 63), zero beyond k. A CTA covers 32 rows x 32
// columns through a shared tile (the transposed read stays coalesced);
// blockIdx.z picks the operand, so both operands of a GEMM split in one
// launch.
__global__ void __launch_bounds__(256) split_kernel(const SplitOp a, const SplitOp b, int k, int kt)
{
    __shared__ float tile[32][33];
    pdl_wait_upstream();
    pdl_launch_dependents();
    const SplitOp &o = blockIdx.z == 0 ? a : b;
    const float *__restrict__ S = o.S;
    const int64_t lds = o.lds;
    const int rows = o.rows, trans = o.trans;
    uint16_t *__restrict__ out = o.out;
    const int64_t op = (int64_t)kt * 3 * kTcK; // out row pitch (elements)
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    if (r0 >= rows)
        return;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5; // 32 x 8
    for (int i = ty; i < 32; i += 8) {
        float v = 0.f;
        if (!trans) {
            const int r = r0 + i, c = c0 + tx;
            if (r < rows && c < k)
                v = S[(int64_t)r * lds + c];
            tile[i][tx] = v;
        } else {
            // element (row r, column c) of the operand is S[c][r]: read S rows c0+i, columns r0+tx
            const int c = c0 + i, r = r0 + tx;
            if (r < rows && c < k)
                v = S[(int64_t)c * lds + r];
            tile[tx][i] = v;
        }
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int r = r0 + i, c = c0 + tx;
        if (r >= rows || c >= kt * kTcK)
            continue;
        uint16_t p0, p1, p2;
        split3(tile[i][tx], p0, p1, p2);
        uint16_t *o = out + (int64_t)r * op + (int64_t)(c / kTcK) * 3 * kTcK + c % kTcK;
        o[0] = p0;
        o[kTcK] = p1;
        o[2 * kTcK] = p2;
    }
}

// Xt [K][Tp] = X^T for bf16 X [T][K], zero in the padding (columns T .. Tp).
__global__ void __launch_bounds__(256)
    transpose_bf16_kernel(const uint16_t *__restrict__ X, int T, int K, uint16_t *__restrict__ Xt, int Tp)
{
    __shared__ uint16_t tile[32][34];
    pdl_wait_upstream();
    pdl_launch_dependents();
    const int t0 = blockIdx.y * 32, k0 = blockIdx.x * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int i = ty; i < 32; i += 8) {
        const int t = t0 + i, kk = k0 + tx;
        tile[i][tx] = (t < T && kk < K) ? X[(int64_t)t * K + kk] : (uint16_t)0;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int kk = k0 + i, t = t0 + tx;
        if (kk < K && t < Tp)
            Xt[(int64_t)kk * Tp + t] = tile[tx][i];
    }
}

template <int KW> nm_status encode_operand(CUtensorMap *map, const uint16_t *ptr, int64_t rows, int64_t pitch)
{
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn)
        return NM_ERR_CUDA;
    const cuuint64_t dims[2] = {(cuuint64_t)pitch, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)pitch * 2};
    const cuuint32_t box[2] = {(cuuint32_t)KW, (cuuint32_t)kTcM};
    const cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, KW == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? NM_OK
               : NM_ERR_CUDA;
}

template <int NP, int KW>
nm_status launch_tc(const uint16_t *A, const uint16_t *B, int64_t kt, float *C, int64_t ldc, int64_t M, int64_t N,
                    int64_t k_base, uint32_t flags, float alpha, float beta, uint32_t *status, cudaStream_t st)
{
    using Cfg = TcCfg<NP, KW>;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(tc_gemm_kernel<NP, KW>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    });
    if (attr != cudaSuccess)
        return NM_ERR_CUDA;
    TcMaps maps;
    nm_status s;
    const int64_t pitch = kt * NP * kTcK;
    if ((s = encode_operand<KW>(&maps.a, A, M, pitch)) != NM_OK ||
        (s = encode_operand<KW>(&maps.b, B, N, pitch)) != NM_OK)
        return s;
    // persistent: one CTA per SM (its shared memory allows no second), or one per tile
    const int64_t tn = (N + kTcN - 1) / kTcN;
    const int64_t ntiles = tc_triangular(flags) ? tn * (tn + 1) / 2 : tn * ((M + kTcM - 1) / kTcM);
    if (ntiles > 0x7FFFFFFF)
        return NM_ERR_SHAPE;
    static int sms[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return NM_ERR_CUDA;
    if (!sms[dev] && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return NM_ERR_CUDA;
    const dim3 grid((unsigned)(ntiles < sms[dev] ? ntiles : sms[dev]));
    return launch_pdl(tc_gemm_kernel<NP, KW>, grid, dim3(kTcThreads), Cfg::kSmem, st, maps, C, ldc, (int)M, (int)N,
                      (int)kt, k_base, flags, alpha, beta, status) == cudaSuccess
               ? NM_OK
               : NM_ERR_CUDA;
}

} // namespace

size_t tc_operand_bytes(int64_t rows, int64_t k, bool emulated)
{
    if (emulated && k > 1024) // tc_gemm_f32 splits one chunk of k at a time
        k = 1024;
    const int64_t kt = (k + kTcK - 1) / kTcK;
    return (size_t)rows * kt * kTcK * (emulated ? 3 : 1) * 2;
}

nm_status tc_gemm_bf16(const uint16_t *A, const uint16_t *B, int64_t kt, int nparts, float *C, int64_t ldc, int64_t M,
                       int64_t N, float alpha, float beta, uint32_t *status, cudaStream_t st, unsigned flags,
                       int64_t k_base)
{
    if (M <= 0 || N <= 0)
        return NM_OK;
    if (kt < 0 || kt * nparts * kTcK > 0x7FFFFFFF || N % 4 != 0 || ldc % 4 != 0 || ((uintptr_t)C & 15u) != 0 ||
        M > 0x7FFFFFFF || N > 0x7FFFFFFF || (nparts != 1 && nparts != 3) ||
        ((flags & (kTcCLower | kTcCSym)) && M != N))
        return NM_ERR_SHAPE;
    return nparts == 1 ? launch_tc<1, 64>(A, B, kt, C, ldc, M, N, k_base, flags, alpha, beta, status, st)
                       : launch_tc<3, 32>(A, B, kt, C, ldc, M, N, k_base, flags, alpha, beta, status, st);
}

// Splits A (rows_a x k) and, unless b_rows is 0, B (b_rows x k) in one launch.
nm_status tc_split2(const float *A, int64_t lda, int64_t a_rows, bool a_trans, uint16_t *a_out, const float *B,
                    int64_t ldb, int64_t b_rows, bool b_trans, uint16_t *b_out, int64_t k, cudaStream_t st)
{
    if (k <= 0 || (a_rows <= 0 && b_rows <= 0))
        return NM_OK;
    if (a_rows > 0x7FFFFFFF || b_rows > 0x7FFFFFFF || k > 0x7FFFFFFF)
        return NM_ERR_SHAPE;
    const int64_t kt = (k + kTcK - 1) / kTcK;
    const int64_t rmax = a_rows > b_rows ? a_rows : b_rows;
    // the padding columns up to kt * 64 are written as zero parts by the kernel (grid covers them)
    const dim3 grid((unsigned)((kt * kTcK + 31) / 32), (unsigned)((rmax + 31) / 32), b_rows > 0 ? 2u : 1u);
    if (grid.y > 65535)
        return NM_ERR_SHAPE;
    const SplitOp a{A, lda, (int)a_rows, a_trans ? 1 : 0, a_out}, b{B, ldb, (int)b_rows, b_trans ? 1 : 0, b_out};
    return launch_pdl(split_kernel, grid, dim3(256), 0, st, a, b, (int)k, (int)kt) == cudaSuccess ? NM_OK
                                                                                                  : NM_ERR_CUDA;
}

nm_status tc_transpose_bf16(const uint16_t *X, int64_t T, int64_t K, uint16_t *Xt, int64_t Tp, cudaStream_t st)
{
    if (T <= 0 || K <= 0)
        return NM_OK;
    const dim3 grid((unsigned)((K + 31) / 32), (unsigned)((Tp + 31) / 32));
    return launch_pdl(transpose_bf16_kernel, grid, dim3(256), 0, st, X, (int)T, (int)K, Xt, (int)Tp) == cudaSuccess
               ? NM_OK
               : NM_ERR_CUDA;
}

// ---- plain fp32 on the CUDA cores (the NM_OBS_SGEMM reference mode) -----------

// C = alpha A op(B) + beta C, fp32: A (M x k) row-major; op(B) = B^T for B
// (N x k) row-major, or B for B (k x N) row-major (b_kn). 64 x 64 outputs per
// CTA, 4 x 4 per thread, k in steps of 16 through shared memory.
__global__ void __launch_bounds__(256)
    simt_gemm_kernel(const float *__restrict__ A, int64_t lda, const float *__restrict__ B, int64_t ldb, int b_kn,
                     int M, int N, int k, float *C, int64_t ldc, float alpha, float beta)
{
    __shared__ float As[16][64 + 4];
    __shared__ float Bs[16][64 + 4];
    pdl_wait_upstream();
    pdl_launch_dependents();
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < k; k0 += 16) {
        for (int i = threadIdx.x; i < 64 * 16; i += 256) {
            const int r = i / 16, kk = i % 16; // A tile: row r, column kk
            As[kk][r] = (m0 + r < M && k0 + kk < k) ? A[(int64_t)(m0 + r) * lda + k0 + kk] : 0.f;
            if (b_kn) {
                const int kr = i / 64, c = i % 64; // B rows are k
                Bs[kr][c] = (n0 + c < N && k0 + kr < k) ? B[(int64_t)(k0 + kr) * ldb + n0 + c] : 0.f;
            } else {
                Bs[kk][r] = (n0 + r < N && k0 + kk < k) ? B[(int64_t)(n0 + r) * ldb + k0 + kk] : 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = As[kk][ty * 4 + i];
                b[i] = Bs[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = m0 + ty * 4 + i;
        if (r >= M)
            continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = n0 + tx * 4 + j;
            if (c < N) {
                float *d = C + (int64_t)r * ldc + c;
                *d = beta != 0.f ? fmaf(beta, *d, alpha * acc[i][j]) : alpha * acc[i][j];
            }
        }
    }
}

// The same product for small shapes (the leaves of the Cholesky recursion,
// where one split launch and one tensor-core launch cost more than the
// arithmetic): 32 x 32 outputs per CTA of 256 threads (four consecutive
// columns each), k in steps of 32 through shared memory, the next step's
// operands loaded into registers while the current one is multiplied.
__global__ void __launch_bounds__(256)
    simt_small_kernel(const float *__restrict__ A, int64_t lda, const float *__restrict__ B, int64_t ldb, int b_kn,
                      int M, int N, int k, float *C, int64_t ldc, float alpha, float beta)
{
    __shared__ float As[32][33];                 // [k][m]
    __shared__ __align__(16) float Bs[32][36];   // [k][n]
    pdl_wait_upstream();
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    const int m0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
    const int r = tid >> 3, c = (tid & 7) * 4;   // this thread's output row and first column
    const int li = tid >> 3, lj = (tid & 7) * 4; // this thread's four elements of each loaded tile
    float ra[4], rb[4];
    auto load = [&](int k0) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int m = m0 + li, kk = k0 + lj + e;
            ra[e] = (m < M && kk < k) ? A[(int64_t)m * lda + kk] : 0.f;
            if (b_kn) {
                const int kr = k0 + li, n = n0 + lj + e; // B is k x N
                rb[e] = (kr < k && n < N) ? B[(int64_t)kr * ldb + n] : 0.f;
            } else {
                const int n = n0 + li; // B is N x k
                rb[e] = (n < N && kk < k) ? B[(int64_t)n * ldb + kk] : 0.f;
            }
        }
    };
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (k > 0)
        load(0);
    for (int k0 = 0; k0 < k; k0 += 32) {
        __syncthreads(); // the previous step's reads of the tiles are done
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            As[lj + e][li] = ra[e];
            if (b_kn)
                Bs[li][lj + e] = rb[e];
            else
                Bs[lj + e][li] = rb[e];
        }
        __syncthreads();
        if (k0 + 32 < k)
            load(k0 + 32);
#pragma unroll 8
        for (int kk = 0; kk < 32; ++kk) {
            const float a = As[kk][r];
            const float4 b = *reinterpret_cast<const float4 *>(&Bs[kk][c]);
            acc[0] = fmaf(a, b.x, acc[0]);
            acc[1] = fmaf(a, b.y, acc[1]);
            acc[2] = fmaf(a, b.z, acc[2]);
            acc[3] = fmaf(a, b.w, acc[3]);
        }
    }
    const int m = m0 + r;
    if (m < M) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int n = n0 + c + e;
            if (n < N) {
                float *d = C + (int64_t)m * ldc + n;
                *d = beta != 0.f ? fmaf(beta, *d, alpha * acc[e]) : alpha * acc[e];
            }
        }
    }
}

nm_status simt_small_f32(const float *A, int64_t lda, const float *B, int64_t ldb, bool b_kn, int64_t M, int64_t N,
                         int64_t k, float *C, int64_t ldc, float alpha, float beta, cudaStream_t st)
{
    if (M <= 0 || N <= 0)
        return NM_OK;
    const dim3 grid((unsigned)((N + 31) / 32), (unsigned)((M + 31) / 32));
    if (grid.y > 65535 || M > 0x7FFFFFFF || N > 0x7FFFFFFF || k > 0x7FFFFFFF)
        return NM_ERR_SHAPE;
    return launch_pdl(simt_small_kernel, grid, dim3(256), 0, st, A, lda, B, ldb, b_kn ? 1 : 0, (int)M, (int)N,
                      (int)(k > 0 ? k : 0), C, ldc, alpha, beta) == cudaSuccess
               ? NM_OK
               : NM_ERR_CUDA;
}

nm_status simt_gemm_f32(const float *A, int64_t lda, const float *B, int64_t ldb, bool b_kn, int64_t M, int64_t N,
                        int64_t k, float *C, int64_t ldc, float alpha, float beta, cudaStream_t st)
{
    if (M <= 0 || N <= 0)
        return NM_OK;
    const dim3 grid((unsigned)((N + 63) / 64), (unsigned)((M + 63) / 64));
    if (grid.y > 65535 || M > 0x7FFFFFFF || N > 0x7FFFFFFF || k > 0x7FFFFFFF)
        return NM_ERR_SHAPE;
    return launch_pdl(simt_gemm_kernel, grid, dim3(256), 0, st, A, lda, B, ldb, b_kn ? 1 : 0, (int)M, (int)N,
                      (int)(k > 0 ? k : 0), C, ldc, alpha, beta) == cudaSuccess
               ? NM_OK
               : NM_ERR_CUDA;
}

// The k range of an emulated fp32 GEMM goes through the tensor cores in chunks
// of kTcChunk, each chunk's result added to C in fp32 (the epilogue's
// alpha acc + beta C with beta = 1): the tensor cores' accumulation loses more
// than fp32 rounding over a long k (a Cholesky of K = 14336, with k up to 7168,
// left more N:M choices off the fp64 oracle's than plain fp32 did).
constexpr int64_t kTcChunk = 1024;

nm_status tc_gemm_f32(const float *A, int64_t lda, bool a_trans, const float *B, int64_t ldb, bool b_trans, int64_t M,
                      int64_t N, int64_t k, float *C, int64_t ldc, float alpha, float beta, uint16_t *work_a,
                      uint16_t *work_b, uint32_t *status, cudaStream_t st, unsigned flags)
{
    if (M <= 0 || N <= 0)
        return NM_OK;
    if (k <= 0) // C = beta C
        return simt_gemm_f32(A, lda, B, ldb, b_trans, M, N, 0, C, ldc, alpha, beta, st);
    // B is A (the product of a matrix with its own transpose): one split serves both
    const bool same = A == B && a_trans == b_trans && lda == ldb && M == N;
    for (int64_t k0 = 0; k0 < k; k0 += kTcChunk) {
        const int64_t kc = k - k0 < kTcChunk ? k - k0 : kTcChunk;
        // a chunk that no tile's k range reaches leaves C as it is (beta is 1 after the first)
        if (k0 > 0 && (((flags & kTcALower) && k0 >= M) || ((flags & kTcBLower) && k0 >= N)))
            break;
        const float *Ak = a_trans ? A + k0 * lda : A + k0;
        const float *Bk = b_trans ? B + k0 * ldb : B + k0;
        nm_status s;
        if ((s = tc_split2(Ak, lda, M, a_trans, work_a, Bk, ldb, same ? 0 : N, b_trans, work_b, kc, st)) != NM_OK)
            return s;
        if ((s = tc_gemm_bf16(work_a, same ? work_a : work_b, (kc + kTcK - 1) / kTcK, 3, C, ldc, M, N, alpha,
                              k0 == 0 ? beta : 1.0f, status, st, flags, k0)) != NM_OK)
            return s;
    }
    return NM_OK;
}

} // namespace nm
