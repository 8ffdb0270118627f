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
// A row block split between warps of one CTA is finished, after the CTA's
// barrier, by the warp that holds its last part (it adds the parts in warp
// order); one split between CTAs by the CTA that arrives last (a counter in
// the scratch). Partial sums are added in a fixed order, so results repeat
// bit for bit.
//
// A unit policy `Pol` supplies the stage layout and the per-unit arithmetic:
//   Pol::kCols            columns per unit
//   Pol::kHasMasks        whether maps.m is used
//   Pol::stage_bytes<B>() bytes of one weight stage (multiple of 1024)
//   Pol::tx_bytes<B>()    bytes one unit's copies deliver (weights + x)
//   Pol::x_bytes<B>()     bytes of one unit's x slice (multiple of 128)
//   Pol::xf_bytes<B>()    per-warp scratch in shared memory (may be 0)
//   Pol::kSharedBytes     CTA-wide shared memory of the policy (tables)
//   Pol::init_shared(ptr, tid, nthreads)            fills it before the pipeline starts
//   Pol::issue_weights(stage, bar, kc, rb, policy, maps)
//   Pol::Regs<B>          the unit's weights as one lane holds them
//   Pol::load<B>(stage_ptr, lane, regs)             stage -> registers
//   Pol::compute<B>(regs, x_ptr, xf_ptr, shared_ptr, state, lane, acc)
//                         accumulates into acc[4][B]; `state` is per warp
//
// A unit's weights are copied from its stage into registers first; the stage
// is then refilled at once, and the arithmetic runs while the refill is in
// flight, so a stage is busy only for the memory round trip, not for the
// round trip plus the arithmetic. The x slices have their own ring of NBUF+1
// slots per warp, so the slice of the unit being computed is not the one the
// refill overwrites.
#pragma once

#include <algorithm>
#include <mutex>
#include <type_traits>

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
    int32_t P;      // CTAs taking part (CTAs from P on have no work)
    int32_t shared_queue; // warps take the CTA's units from a shared counter (see consume_queue)
    int32_t pair_k;       // CTA pairs (clusters of 2) split each row block's K in halves (see queue_finish_pair)
    uint32_t kc_inv;      // ceil(2^32 / KC): n / KC = umulhi(n, kc_inv) for the small n used
    int32_t atomic;       // parts of a shared row block go to y by fp32 atomicAdd (y zeroed before)
    void *y_k;            // kOutQkv: the buffers of rows [rows_q, rows_qk) and [rows_qk, rows)
    void *y_v;
    int64_t rows_q;
    int64_t rows_qk;
    Scratch scratch;
};

// Units a CTA of W warps may take from its shared queue (batch 1): one fp32
// partial per row and unit is kept in shared memory until the CTA's end.
template <int W> constexpr int queue_cap() { return W >= 16 ? 128 : 96; }
template <class Pol, int B, int W, int NBUF> constexpr int queue_bytes()
{
    return B == 1 ? 16 + W * NBUF * 4 + queue_cap<W>() * 32 * 4 + 32 * 4 : 0;
}

// Store row `row` (= 32 * row block + lane; all 32 lanes call this together)
// of the output. kOutSwiglu: the rows come in gate/up pairs -- lanes 0-15 of
// row block t hold gate rows 16t..16t+15, lanes 16-31 the up rows of the same
// indices -- and lane i < 16 stores h[16t + i] = bf16_rn(silu(g) * u) with
// silu(g) = g / (1 + exp(-g)), all in fp32; y is then h [batch][rows / 2].
// kOutQkv: row r goes to the one of three [batch][part rows] buffers whose
// row range holds it (q: [0, rows_q), k: [rows_q, rows_qk), v: the rest).
template <int B, int OUT>
__device__ __forceinline__ void store_y(const StreamKParams &p, int64_t row, const float (&v)[B])
{
    void *const y = p.y;
    const int64_t rows = p.rows;
    if constexpr (OUT == kOutQkv) {
        if (row >= rows)
            return;
        uint16_t *dst;
        int64_t n, r;
        if (row < p.rows_q) {
            dst = (uint16_t *)y;
            n = p.rows_q;
            r = row;
        } else if (row < p.rows_qk) {
            dst = (uint16_t *)p.y_k;
            n = p.rows_qk - p.rows_q;
            r = row - p.rows_q;
        } else {
            dst = (uint16_t *)p.y_v;
            n = rows - p.rows_qk;
            r = row - p.rows_qk;
        }
#pragma unroll
        for (int b = 0; b < B; ++b)
            dst[(int64_t)b * n + r] = f32_to_bf16_rn(v[b]);
        return;
    }
    if constexpr (OUT == kOutSwiglu) {
        const int lane = (int)(row & 31);
        const int64_t hrows = rows >> 1, hr = (row >> 5) * 16 + lane;
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const float u = __shfl_down_sync(0xFFFFFFFFu, v[b], 16);
            const float g = v[b];
            if (lane < 16 && hr < hrows)
                ((uint16_t *)y)[(int64_t)b * hrows + hr] = f32_to_bf16_rn(g / (1.0f + expf(-g)) * u);
        }
        return;
    }
    if (row >= rows)
        return;
#pragma unroll
    for (int b = 0; b < B; ++b) {
        if (OUT == kOutF32)
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
// the CTA that publishes last adds all parts in CTA order and stores y. In the
// atomic variant (fp32 output) each part is added into the zeroed y instead:
// the split reduction with atomicAdd; the order of the adds is not fixed.
template <int B, int OUT>
__device__ __forceinline__ void finish_across_ctas(const StreamKParams &p, const CtaRange &cr, int64_t rb,
                                                   const float (&tot)[B], int lane)
{
    const int64_t KC = p.KC;
    const int64_t rb_lo = rb * KC, rb_hi = rb_lo + KC;
    const int64_t row = rb * kUnitRows + lane;
    if (rb_lo >= cr.cs && rb_hi <= cr.ce) {
        store_y<B, OUT>(p, row, tot);
        return;
    }
    if constexpr (OUT == kOutF32) {
        if (p.atomic) {
            if (row < p.rows) {
#pragma unroll
                for (int b = 0; b < B; ++b)
                    atomicAdd((float *)p.y + (int64_t)b * p.rows + row, tot[b]);
            }
            return;
        }
    }
    const int64_t U = p.U, P = p.P;
    const int64_t c = blockIdx.x;
    const int64_t first = div64(((rb_lo + 1) * (P)) - 1, U);
    const int64_t last = div64(((rb_hi) * (P)) - 1, U);
    const int slot = (rb == div64(cr.cs, KC)) ? 0 : 1;
    if (!NM_IN_BOUNDS(p.scratch.status, c < kMaxCtas && first <= last && last < P && first >= 0))
        return;
    float *mine = p.scratch.partials + (c * 2 + slot) * (8 * 32) + lane;
#pragma unroll
    for (int b = 0; b < B; ++b)
        mine[b * 32] = tot[b];
    // The warp's stores are ordered before lane 0's release; the CTA that
    // counts last acquires every earlier part through the same counter.
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0)
        old = atom_add_acq_rel_gpu(&p.scratch.counters[first], 1u);
    old = __shfl_sync(0xFFFFFFFFu, old, 0);
    if (old != (uint32_t)(last - first))
        return;
    __syncwarp();
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
            if (cc <= last && NM_IN_BOUNDS(p.scratch.status, cc < kMaxCtas)) {
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
    store_y<B, OUT>(p, row, sum);
    if (lane == 0)
        atomicExch(&p.scratch.counters[first], 0u);
}

// After the CTA's barrier: if this warp holds the last part of row block rb
// inside the CTA and rb is not complete in one warp, add the CTA's parts of
// rb (warp order, shared memory) and finish it across CTAs.
template <int B, int OUT>
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
    // Every contributor after the first starts its range inside rb, so rb is
    // its first row block (slot 0); the first contributor's slot is 1 when its
    // range began in an earlier row block. (One division for the whole row
    // block: a division per contributor made this loop cost microseconds.)
    const int slot_first = (cr.cs + muldiv(n, first, cr.nw) < lo) ? 1 : 0;
    float tot[B];
#pragma unroll
    for (int b = 0; b < B; ++b)
        tot[b] = 0.f;
    // Up to four contributors' loads in flight, added in warp order (a missing
    // one adds +0, which leaves the sum unchanged: it never is -0).
    for (int w0 = first; w0 <= last; w0 += 4) {
        float v[4][B];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int w = w0 + j;
            const int ws = w == first ? slot_first : 0;
            const bool in = w <= last && NM_IN_BOUNDS(p.scratch.status, w >= 0 && w < cr.nw);
            const float *q = part + ((w * 2 + ws) * B) * 32 + lane;
#pragma unroll
            for (int b = 0; b < B; ++b)
                v[j][b] = in ? q[b * 32] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int b = 0; b < B; ++b)
                tot[b] += v[j][b];
    }
    finish_across_ctas<B, OUT>(p, cr, rb, tot, lane);
}

// Bytes of one warp's x ring (NBUF + 1 slots).
template <class Pol, int B, int NBUF> constexpr int xring_bytes() { return (NBUF + 1) * Pol::template x_bytes<B>(); }

template <class Pol, int B, int W, int NBUF> constexpr int streamk_smem_bytes()
{
    return 1024 + W * NBUF * Pol::template stage_bytes<B>() + W * xring_bytes<Pol, B, NBUF>() +
           W * (kGuardBytes + Pol::template xf_bytes<B>()) + W * part_bytes<B>() + W * 4 + 16 + Pol::kSharedBytes +
           queue_bytes<Pol, B, W, NBUF>();
}

// Dynamic shared memory of a CTA: per-warp stage buffers (1024-aligned for
// the 128-byte swizzle), per-warp x rings (128-aligned), per-warp fp32 x
// windows, per-warp partial-sum slots, then the policy's CTA-wide region
// (16-byte aligned).
template <class Pol, int B, int W, int NBUF> struct SmemLayout {
    uint8_t *stage0p; // this warp's first stage buffer
    uint8_t *xring;   // this warp's first x slot
    uint8_t *xfp;     // this warp's x window
    float *part;      // partial-sum slots of all warps
    uint8_t *pol;     // the policy's region
    uint8_t *queue;   // the shared queue: counter, per-stage unit numbers, per-unit partials
    __device__ __forceinline__ SmemLayout(uint8_t *dsmem, int warp)
    {
        constexpr int SB = Pol::template stage_bytes<B>();
        constexpr int XR = xring_bytes<Pol, B, NBUF>();
        constexpr int XF = Pol::template xf_bytes<B>();
        static_assert(SB % 1024 == 0 && XR % 128 == 0, "stage and x-slot alignment");
        uint8_t *const sbase = dsmem + ((1024u - (smem_addr(dsmem) & 1023u)) & 1023u);
        stage0p = sbase + warp * NBUF * SB;
        uint8_t *const xbase = sbase + W * NBUF * SB;
        xring = xbase + warp * XR;
        uint8_t *const fbase = xbase + W * XR;
        xfp = fbase + warp * (kGuardBytes + XF) + kGuardBytes;
        part = (float *)(fbase + W * (kGuardBytes + XF));
        // pointer arithmetic only (no integer round trip), so that loads
        // through `pol` stay shared-memory loads
        uint8_t *const after = (uint8_t *)part + W * part_bytes<B>() + W * 4;
        pol = after + ((16u - (smem_addr(after) & 15u)) & 15u);
        queue = pol + Pol::kSharedBytes; // 16-byte aligned: kSharedBytes is a multiple of 16
    }
};

// The CTA's unit range: whole row blocks or an even share of the units.
__device__ __forceinline__ CtaRange cta_range(const StreamKParams &p, int W, int c)
{
    CtaRange cr;
    if (c >= p.P) {
        cr.cs = cr.ce = 0;
        cr.nw = 0;
        return cr;
    }
    if (p.pair_k) { // CTA 2t: the first half of row block t's units, CTA 2t+1 the second
        const int64_t rb = c >> 1, h = p.KC >> 1;
        cr.cs = rb * p.KC + ((c & 1) ? h : 0);
        cr.ce = (c & 1) ? (rb + 1) * p.KC : rb * p.KC + h;
    } else if (p.whole) {
        const int64_t nrb = div64(p.U, p.KC);
        cr.cs = muldiv(nrb, c, p.P) * p.KC;
        cr.ce = muldiv(nrb, c + 1, p.P) * p.KC;
    } else {
        cr.cs = muldiv(p.U, c, p.P);
        cr.ce = muldiv(p.U, c + 1, p.P);
    }
    cr.nw = (int)((cr.ce - cr.cs) < W ? (cr.ce - cr.cs) : W);
    return cr;
}

// A warp's contiguous share of its CTA's range.
struct WarpWork {
    int64_t ub, ue; // units [ub, ue)
    int n;          // ue - ub
    int32_t rb0;    // row block of unit ub
    int32_t kc0;    // position of unit ub in its row block
};

__device__ __forceinline__ WarpWork warp_work(const CtaRange &cr, int32_t KC, int warp)
{
    WarpWork w;
    w.ub = w.ue = 0;
    if (warp < cr.nw) {
        const int64_t n_cta = cr.ce - cr.cs;
        w.ub = cr.cs + muldiv(n_cta, warp, cr.nw);
        w.ue = cr.cs + muldiv(n_cta, warp + 1, cr.nw);
    }
    w.n = (int)(w.ue - w.ub);
    w.rb0 = (int32_t)div64(w.ub, KC);
    w.kc0 = (int32_t)(w.ub - (int64_t)w.rb0 * KC);
    return w;
}

// Lane 0: arm the stages of the warp's first min(n, NBUF) units (all bytes
// of the stage expected) and request their weights. `it` counts the units
// the warp consumed before; unit it + i uses stage (it + i) % NBUF.
template <class Pol, int B, int NBUF>
__device__ __forceinline__ void issue_prologue_weights(const TensorMaps *maps, const WarpWork &w, int32_t KC,
                                                       uint32_t it, uint32_t stage0, uint32_t bar0, uint64_t pol)
{
    constexpr int SB = Pol::template stage_bytes<B>();
    constexpr uint32_t TX = Pol::template tx_bytes<B>();
    const int npre = w.n < NBUF ? w.n : NBUF;
    int32_t rb = w.rb0, kc = w.kc0;
    for (int i = 0; i < npre; ++i) {
        const uint32_t s = (it + i) % NBUF;
        mbar_arrive_expect_tx(bar0 + 8 * s, TX);
        Pol::issue_weights(stage0 + s * SB, bar0 + 8 * s, kc, rb * kUnitRows, pol, *maps);
        if (++kc == KC) {
            kc = 0;
            ++rb;
        }
    }
}

// Lane 0: request the x slices of the same units; unit it + i uses x slot
// (it + i) % (NBUF + 1) and completes on its stage's barrier.
template <class Pol, int B, int NBUF>
__device__ __forceinline__ void issue_prologue_x(const TensorMaps *maps, const WarpWork &w, int32_t KC, uint32_t it,
                                                 uint32_t xr0, uint32_t bar0)
{
    constexpr int XB = Pol::template x_bytes<B>();
    const int npre = w.n < NBUF ? w.n : NBUF;
    int32_t kc = w.kc0;
    for (int i = 0; i < npre; ++i) {
        const uint32_t j = it + i;
        tma_load_2d(xr0 + (j % (NBUF + 1)) * XB, &maps->x, kc * Pol::kCols, 0, bar0 + 8 * (j % NBUF));
        if (++kc == KC)
            kc = 0;
    }
}

// Consume the warp's n units (their first min(n, NBUF) already requested):
// for each, wait for its stage, copy its weights into registers, refill the
// stage with the unit NBUF ahead, then do the arithmetic. A segment (the part
// of a row block in this range) that is a whole row block is stored directly;
// other segments leave their sum in the warp's partial slot (0: the range's
// first row block, 1: its last).
template <class Pol, int B, int W, int NBUF, int OUT>
__device__ __forceinline__ void consume_range(const TensorMaps *maps, const StreamKParams &p, const WarpWork &w,
                                              uint32_t it, uint32_t stage0, const uint8_t *stage0p, uint32_t bar0,
                                              uint32_t xr0, const uint8_t *xringp, uint8_t *xfp,
                                              const uint8_t *pol_smem, float *part, int warp, int lane, uint64_t pol,
                                              typename Pol::State &pst, bool &dead)
{
    constexpr int SB = Pol::template stage_bytes<B>();
    constexpr int XB = Pol::template x_bytes<B>();
    constexpr uint32_t TX = Pol::template tx_bytes<B>();
    float acc[4][B];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int b = 0; b < B; ++b)
            acc[q][b] = 0.f;

    const int32_t KC = p.KC;
    const int n = w.n;
    int32_t rb = w.rb0, kc = w.kc0;   // unit being consumed
    int32_t prb = w.rb0, pkc = w.kc0; // unit to request next (i + NBUF)
    for (int i = 0; i < (n < NBUF ? n : NBUF); ++i) {
        if (++pkc == KC) {
            pkc = 0;
            ++prb;
        }
    }
    int32_t seg_kc0 = w.kc0; // first unit of the current segment, as kc
    for (int i = 0; i < n; ++i) {
        const uint32_t j = it + (uint32_t)i;
        const int s = (int)(j % NBUF);
        const uint32_t st = stage0 + s * SB, bar = bar0 + 8 * s;
        mbar_wait_bounded(bar, (j / NBUF) & 1u, p.scratch.status, dead);
        typename Pol::template Regs<B> r;
        Pol::template load<B>(stage0p + s * SB, lane, r);
        __syncwarp(); // every lane's reads of the stage are done
        if (i + NBUF < n && NM_IN_BOUNDS(p.scratch.status, pkc < KC && (int64_t)prb * kUnitRows < p.rows)) {
            if (lane == 0 && !dead) {
                const uint32_t jn = j + NBUF;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, TX);
                Pol::issue_weights(st, bar, pkc, prb * kUnitRows, pol, *maps);
                tma_load_2d(xr0 + (jn % (NBUF + 1)) * XB, &maps->x, pkc * Pol::kCols, 0, bar);
            }
            if (++pkc == KC) {
                pkc = 0;
                ++prb;
            }
        }
        Pol::template compute<B>(r, xringp + (j % (NBUF + 1)) * XB, xfp, pol_smem, pst, lane, acc);
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
                store_y<B, OUT>(p, (int64_t)rb * kUnitRows + lane, tot); // a whole row block
            } else if (NM_IN_BOUNDS(p.scratch.status, warp < W && (rb == w.rb0 || rb == (int32_t)div64(w.ue - 1, KC)))) {
                float *mine = part + ((warp * 2 + (rb == w.rb0 ? 0 : 1)) * B) * 32 + lane;
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
}

// After the CTA barrier that follows consume_range: finish the warp's first
// and last row block (the only segments that can be partial).
template <int B, int OUT>
__device__ __forceinline__ void finish_warp(const StreamKParams &p, const CtaRange &cr, const float *part,
                                            const WarpWork &w, int lane)
{
    if (w.n <= 0)
        return;
    const int64_t KC = p.KC;
    const int64_t rbf = w.rb0, rbl = div64(w.ue - 1, KC);
    finish_in_cta<B, OUT>(p, cr, part, rbf, w.ub, rbf == rbl ? w.ue : (rbf + 1) * KC, lane);
    if (rbl != rbf)
        finish_in_cta<B, OUT>(p, cr, part, rbl, rbl * KC, w.ue, lane);
}

// Batch 1, a CTA range of at most queue_cap<W>() units: the warps take the
// CTA's units from a shared counter instead of fixed sub-ranges, so that a
// warp whose data comes late does fewer units and the CTA's warps finish
// together. Warp w's first NBUF units are units w*NBUF .. w*NBUF+NBUF-1 (set
// before the CTA barrier, with no counter); the counter starts after them.
// Each unit's sum goes to its own slot; after the CTA barrier every row block
// is added in unit order (queue_finish), so the result does not depend on
// which warp took which unit. The unit held by a stage is recorded next to
// it by lane 0 before the stage's copies are requested.
struct QueueView {
    uint32_t *claim;      // next unit to hand out
    uint32_t *stage_unit; // [W][NBUF]
    float *upart;         // [cap][32]
    float *peer;          // [32]: the other half of the row block (pair_k, rank 0)
};

template <class Pol, int B, int W, int NBUF>
__device__ __forceinline__ QueueView queue_view(uint8_t *q)
{
    QueueView v;
    v.claim = (uint32_t *)q;
    v.stage_unit = (uint32_t *)(q + 16);
    v.upart = (float *)(q + 16 + W * NBUF * 4);
    v.peer = v.upart + queue_cap<W>() * 32;
    return v;
}

// Where the CTA range starts: row block rb_cs, position kc_cs in it.
struct QueueBase {
    int32_t rb_cs;
    uint32_t kc_cs;
};

__device__ __forceinline__ QueueBase queue_base(const StreamKParams &p, int64_t cs)
{
    QueueBase qb;
    qb.rb_cs = (int32_t)div64(cs, p.KC);
    qb.kc_cs = (uint32_t)(cs - (int64_t)qb.rb_cs * p.KC);
    return qb;
}

// Row block and position of unit u of the CTA range.
__device__ __forceinline__ void queue_unit_coords(const StreamKParams &p, QueueBase qb, uint32_t u, int32_t &rb,
                                                  int32_t &kc)
{
    const uint32_t k = qb.kc_cs + u; // < KC + cap
    const uint32_t q = __umulhi(k, p.kc_inv);
    rb = qb.rb_cs + (int32_t)q;
    kc = (int32_t)(k - q * (uint32_t)p.KC);
}

// Lane 0: the first units of this warp, requested before the CTA barrier.
template <class Pol, int B, int NBUF>
__device__ __forceinline__ int queue_prologue(const TensorMaps *maps, const StreamKParams &p, const CtaRange &cr,
                                              QueueView qv, int warp, uint32_t stage0, uint32_t bar0, uint64_t pol)
{
    constexpr int SB = Pol::template stage_bytes<B>();
    constexpr uint32_t TX = Pol::template tx_bytes<B>();
    const uint32_t n = (uint32_t)(cr.ce - cr.cs);
    const QueueBase qb = queue_base(p, cr.cs);
    int npre = 0;
    for (int i = 0; i < NBUF; ++i) {
        const uint32_t u = (uint32_t)(warp * NBUF + i);
        if (u >= n)
            break;
        int32_t rb, kc;
        queue_unit_coords(p, qb, u, rb, kc);
        qv.stage_unit[warp * NBUF + i] = u;
        mbar_arrive_expect_tx(bar0 + 8 * i, TX);
        Pol::issue_weights(stage0 + i * SB, bar0 + 8 * i, kc, rb * kUnitRows, pol, *maps);
        ++npre;
    }
    return npre;
}

// Lane 0: x of the prologue's units.
template <class Pol, int B, int NBUF>
__device__ __forceinline__ void queue_prologue_x(const TensorMaps *maps, const StreamKParams &p, const CtaRange &cr,
                                                 QueueView qv, int warp, int npre, uint32_t xr0, uint32_t bar0)
{
    constexpr int XB = Pol::template x_bytes<B>();
    const QueueBase qb = queue_base(p, cr.cs);
    for (int i = 0; i < npre; ++i) {
        int32_t rb, kc;
        queue_unit_coords(p, qb, qv.stage_unit[warp * NBUF + i], rb, kc);
        tma_load_2d(xr0 + i * XB, &maps->x, kc * Pol::kCols, 0, bar0 + 8 * i);
    }
}

template <class Pol, int B, int W, int NBUF>
__device__ __forceinline__ void consume_queue(const TensorMaps *maps, const StreamKParams &p, const CtaRange &cr,
                                              QueueView qv, int npre, uint32_t stage0, const uint8_t *stage0p,
                                              uint32_t bar0, uint32_t xr0, const uint8_t *xringp, uint8_t *xfp,
                                              const uint8_t *pol_smem, int warp, int lane, uint64_t pol,
                                              typename Pol::State &pst, bool &dead)
{
    constexpr int SB = Pol::template stage_bytes<B>();
    constexpr int XB = Pol::template x_bytes<B>();
    constexpr uint32_t TX = Pol::template tx_bytes<B>();
    const uint32_t n = (uint32_t)(cr.ce - cr.cs);
    const QueueBase qb = queue_base(p, cr.cs);
    int pending = npre; // units requested and not yet consumed
    uint32_t xs = 0;    // x slot of unit j: j % (NBUF + 1)
    for (uint32_t j = 0; pending > 0; ++j) {
        const uint32_t xn = xs == 0 ? NBUF : xs - 1; // x slot of unit j + NBUF
        const int s = (int)(j % NBUF);
        const uint32_t st = stage0 + s * SB, bar = bar0 + 8 * s;
        mbar_wait_bounded(bar, (j / NBUF) & 1u, p.scratch.status, dead);
        const uint32_t u = qv.stage_unit[warp * NBUF + s];
        typename Pol::template Regs<B> r;
        Pol::template load<B>(stage0p + s * SB, lane, r);
        __syncwarp(); // every lane's reads of the stage (and of its unit number) are done
        uint32_t un = 0xFFFFFFFFu;
        if (lane == 0 && !dead) {
            un = atomicAdd(qv.claim, 1u);
            if (un < n && NM_IN_BOUNDS(p.scratch.status, un < (uint32_t)queue_cap<W>())) {
                int32_t rb, kc;
                queue_unit_coords(p, qb, un, rb, kc);
                qv.stage_unit[warp * NBUF + s] = un;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, TX);
                Pol::issue_weights(st, bar, kc, rb * kUnitRows, pol, *maps);
                tma_load_2d(xr0 + xn * XB, &maps->x, kc * Pol::kCols, 0, bar);
            } else {
                un = 0xFFFFFFFFu;
            }
        }
        un = __shfl_sync(0xFFFFFFFFu, un, 0);
        if (un == 0xFFFFFFFFu)
            --pending;
        float acc[4][B];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int b = 0; b < B; ++b)
                acc[q][b] = 0.f;
        Pol::template compute<B>(r, xringp + xs * XB, xfp, pol_smem, pst, lane, acc);
        if (u < n && NM_IN_BOUNDS(p.scratch.status, u < (uint32_t)queue_cap<W>() && xs <= (uint32_t)NBUF))
            qv.upart[u * 32 + lane] = (acc[0][0] + acc[1][0]) + (acc[2][0] + acc[3][0]);
        xs = xs == NBUF ? 0 : xs + 1;
    }
}

// After the CTA barrier: warp w adds the unit sums of the CTA's row blocks
// w, w+W, ... in unit order (four interleaved partial sums, combined in a
// fixed order) and finishes them.
template <int B, int W, int OUT>
__device__ __forceinline__ void queue_finish(const StreamKParams &p, const CtaRange &cr, QueueView qv, int warp,
                                             int lane)
{
    if (cr.ce <= cr.cs)
        return;
    const int64_t KC = p.KC;
    const int64_t rbf = div64(cr.cs, KC), rbl = div64(cr.ce - 1, KC);
    for (int64_t rb = rbf + warp; rb <= rbl; rb += W) {
        const int64_t lo = (rb * KC > cr.cs ? rb * KC : cr.cs) - cr.cs;
        const int64_t hi = ((rb + 1) * KC < cr.ce ? (rb + 1) * KC : cr.ce) - cr.cs;
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
        int64_t u = lo;
        for (; u + 4 <= hi; u += 4) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
                s4[t] += qv.upart[(u + t) * 32 + lane];
        }
        if (u < hi)
            s4[0] += qv.upart[u * 32 + lane];
        if (u + 1 < hi)
            s4[1] += qv.upart[(u + 1) * 32 + lane];
        if (u + 2 < hi)
            s4[2] += qv.upart[(u + 2) * 32 + lane];
        float tot[B];
        tot[0] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        finish_across_ctas<B, OUT>(p, cr, rb, tot, lane);
    }
}

// pair_k (batch 1): the CTA pair of a cluster holds the two halves of one
// row block. Warp 0 of each adds its half's unit sums in unit order; rank 1
// writes its per-row sums into rank 0's shared memory, and after the cluster
// barrier rank 0 adds them to its own (first half + second half) and stores.
template <int B, int W, int OUT>
__device__ __forceinline__ void queue_finish_pair(const StreamKParams &p, const CtaRange &cr, QueueView qv, int warp,
                                                  int lane)
{
    const uint32_t rank = cluster_ctarank();
    float tot = 0.f;
    if (warp == 0 && cr.ce > cr.cs) {
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
        const int64_t n = cr.ce - cr.cs;
        int64_t u = 0;
        for (; u + 4 <= n; u += 4) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
                s4[t] += qv.upart[(u + t) * 32 + lane];
        }
        if (u < n)
            s4[0] += qv.upart[u * 32 + lane];
        if (u + 1 < n)
            s4[1] += qv.upart[(u + 1) * 32 + lane];
        if (u + 2 < n)
            s4[2] += qv.upart[(u + 2) * 32 + lane];
        tot = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        if (rank == 1)
            st_cluster_f32(cluster_map(smem_addr(qv.peer + lane), 0), tot);
    }
    cluster_sync();
    if (warp == 0 && rank == 0 && cr.ce > cr.cs) {
        float v[B];
        v[0] = tot + qv.peer[lane];
        store_y<B, OUT>(p, div64(cr.cs, p.KC) * kUnitRows + lane, v);
    }
}

template <class Pol, int B, int W, int NBUF, int MINB, int OUT>
__global__ void __launch_bounds__(W * 32, MINB) streamk_kernel(const __grid_constant__ TensorMaps maps,
                                                                const StreamKParams p)
{
    __shared__ __align__(8) uint64_t full_bar[W * NBUF];
    extern __shared__ __align__(1024) uint8_t dsmem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const SmemLayout<Pol, B, W, NBUF> sm(dsmem, warp);
    const uint32_t stage0 = smem_addr(sm.stage0p);
    const uint32_t xr0 = smem_addr(sm.xring);
    const uint32_t bar0 = smem_addr(&full_bar[warp * NBUF]);
    const CtaRange cr = cta_range(p, W, blockIdx.x);
    const WarpWork w = warp_work(cr, p.KC, warp);
    const uint64_t pol = l2_policy_evict_first();
    bool dead = false;
    typename Pol::State pst = Pol::initial_state();

    if constexpr (B == 1) {
        if (p.shared_queue) {
            const QueueView qv = queue_view<Pol, B, W, NBUF>(sm.queue);
            int npre = 0;
            if (lane == 0) {
                for (int i = 0; i < NBUF; ++i)
                    mbar_init(bar0 + 8 * i, 1);
                fence_mbar_init();
                npre = queue_prologue<Pol, B, NBUF>(&maps, p, cr, qv, warp, stage0, bar0, pol);
            }
            if (threadIdx.x == 0)
                *qv.claim = (uint32_t)(W * NBUF);
            Pol::init_shared(sm.pol, threadIdx.x, W * 32); // overlaps the first weight copies
            __syncthreads();
            pdl_wait_upstream(); // x may be the previous kernel's output
            if (lane == 0)
                queue_prologue_x<Pol, B, NBUF>(&maps, p, cr, qv, warp, npre, xr0, bar0);
            pdl_launch_dependents();
            npre = __shfl_sync(0xFFFFFFFFu, npre, 0);
            consume_queue<Pol, B, W, NBUF>(&maps, p, cr, qv, npre, stage0, sm.stage0p, bar0, xr0, sm.xring, sm.xfp,
                                           sm.pol, warp, lane, pol, pst, dead);
            __syncthreads(); // every unit sum of this CTA is in shared memory
            if (p.pair_k)
                queue_finish_pair<B, W, OUT>(p, cr, qv, warp, lane);
            else
                queue_finish<B, W, OUT>(p, cr, qv, warp, lane);
            return;
        }
    }

    // Each warp's barriers are its own (initialised, armed and waited on by
    // the warp): the weights of its first stages, which do not depend on the
    // previous kernel, are requested before anything else.
    if (lane == 0) {
        for (int i = 0; i < NBUF; ++i)
            mbar_init(bar0 + 8 * i, 1);
        fence_mbar_init();
        issue_prologue_weights<Pol, B, NBUF>(&maps, w, p.KC, 0, stage0, bar0, pol);
    }
    Pol::init_shared(sm.pol, threadIdx.x, W * 32); // overlaps the first weight copies
    __syncthreads();
    // x may be the previous kernel's output.
    pdl_wait_upstream();
    if (lane == 0)
        issue_prologue_x<Pol, B, NBUF>(&maps, w, p.KC, 0, xr0, bar0);
    pdl_launch_dependents();

    consume_range<Pol, B, W, NBUF, OUT>(&maps, p, w, 0, stage0, sm.stage0p, bar0, xr0, sm.xring, sm.xfp, sm.pol,
                                           sm.part, warp,
                                           lane, pol, pst, dead);
    __syncthreads(); // every partial of this CTA is in shared memory
    finish_warp<B, OUT>(p, cr, sm.part, w, lane);
}

// ---------------------------------------------------------------------------
// The whole decode-token stack as one persistent launch
// ---------------------------------------------------------------------------

// One linear of a stack, as the persistent kernel reads it from global memory.
struct StackOp { // aligned as CUtensorMap requires
    TensorMaps maps;
    void *y;
    int64_t rows;
    int64_t U;
    int32_t KC;
    int32_t whole;
    int32_t P;
    int32_t reserved;
};

__device__ __forceinline__ StreamKParams op_params(const StackOp *op, const Scratch &scratch)
{
    StreamKParams p;
    p.y = op->y;
    p.rows = op->rows;
    p.U = op->U;
    p.KC = op->KC;
    p.whole = op->whole;
    p.P = op->P;
    p.shared_queue = 0; // the persistent kernel splits each op statically
    p.pair_k = 0;
    p.kc_inv = 0;
    p.atomic = 0;
    p.y_k = p.y_v = nullptr;
    p.rows_q = p.rows_qk = 0;
    p.scratch = scratch;
    return p;
}

// Barrier over every CTA of a cooperative launch, by sense reversal on one
// counter: CTA 0 adds 2^31 - (n - 1) and every other CTA adds 1, so the top
// bit flips exactly when the n-th CTA arrives and the low 31 bits return to
// where they were. Whatever the order of arrivals, each barrier adds 2^31 in
// total, so the counter is ready for the next launch as long as every CTA
// arrives at every barrier -- which each does, waits being bounded. A wait
// that runs out records NM_ERR_TIMEOUT and marks the CTA dead: it stops
// requesting data and its later waits return at once.
__device__ __forceinline__ void grid_barrier(uint32_t *ctr, uint32_t *status, bool &dead)
{
    __shared__ uint32_t s_timed_out;
    __syncthreads(); // every write of this CTA before the barrier is done
    if (threadIdx.x == 0) {
        const uint32_t add = blockIdx.x == 0 ? 0x80000000u - (gridDim.x - 1u) : 1u;
        __threadfence();
        const uint32_t old = atomicAdd(ctr, add);
        uint32_t to = 0;
        if (!dead) {
            const uint64_t t0 = globaltimer_ns();
            while (((ld_acquire_gpu(ctr) ^ old) & 0x80000000u) == 0u) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(status, 1u << NM_ERR_TIMEOUT);
                    to = 1;
                    break;
                }
            }
        }
        __threadfence();
        s_timed_out = to;
    }
    __syncthreads();
    if (s_timed_out)
        dead = true;
}

// Runs ops[0..n_ops) in order. Each CTA takes the same place in every op's
// split as the single-launch kernel would give it; between two ops a grid
// barrier stands in for the kernel boundary (x of op l+1 is read only after
// every CTA has stored its part of op l). Before arriving there, each warp
// requests the weights of its first stages of op l+1, which keeps HBM busy
// across the barrier.
template <class Pol, int B, int W, int NBUF, int MINB>
__global__ void __launch_bounds__(W * 32, MINB)
    stack_kernel(const StackOp *__restrict__ ops, const int n_ops, uint32_t *const gbar, const Scratch scratch)
{
    __shared__ __align__(8) uint64_t full_bar[W * NBUF];
    extern __shared__ __align__(1024) uint8_t dsmem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const SmemLayout<Pol, B, W, NBUF> sm(dsmem, warp);
    const uint32_t stage0 = smem_addr(sm.stage0p);
    const uint32_t xr0 = smem_addr(sm.xring);
    const uint32_t bar0 = smem_addr(&full_bar[warp * NBUF]);

    const uint64_t pol = l2_policy_evict_first();
    typename Pol::State pst = Pol::initial_state();
    bool dead = false;
    uint32_t it = 0; // units this warp has consumed so far, over all ops
    StreamKParams p = op_params(&ops[0], scratch);
    CtaRange cr = cta_range(p, W, blockIdx.x);
    WarpWork w = warp_work(cr, p.KC, warp);
    if (lane == 0) {
        for (int i = 0; i < NBUF; ++i)
            mbar_init(bar0 + 8 * i, 1);
        fence_mbar_init();
        issue_prologue_weights<Pol, B, NBUF>(&ops[0].maps, w, p.KC, it, stage0, bar0, pol);
    }
    Pol::init_shared(sm.pol, threadIdx.x, W * 32); // overlaps the first weight copies
    __syncthreads();
    for (int l = 0;; ++l) {
        const TensorMaps *maps = &ops[l].maps;
        const bool more = l + 1 < n_ops;
        const StackOp *next = &ops[more ? l + 1 : l];
        if (threadIdx.x == 0 && more) {
            prefetch_tensormap(&next->maps.w);
            if (Pol::kHasMasks)
                prefetch_tensormap(&next->maps.m);
            prefetch_tensormap(&next->maps.x);
        }
        if (lane == 0 && !dead) {
            fence_proxy_async_global(); // x may hold other CTAs' stores from before the barrier
            issue_prologue_x<Pol, B, NBUF>(maps, w, p.KC, it, xr0, bar0);
        }
        consume_range<Pol, B, W, NBUF, false>(maps, p, w, it, stage0, sm.stage0p, bar0, xr0, sm.xring, sm.xfp, sm.pol,
                                              sm.part,
                                              warp, lane, pol, pst, dead);
        it += (uint32_t)w.n;
        const StreamKParams pn = op_params(next, scratch);
        const CtaRange crn = cta_range(pn, W, blockIdx.x);
        const WarpWork wn = warp_work(crn, pn.KC, warp);
        if (more && lane == 0 && !dead) {
            fence_proxy_async_smem(); // the stages were read by this warp's loads
            issue_prologue_weights<Pol, B, NBUF>(&next->maps, wn, pn.KC, it, stage0, bar0, pol);
        }
        __syncthreads(); // every partial of this CTA is in shared memory
        finish_warp<B, false>(p, cr, sm.part, w, lane);
        if (!more)
            break;
        grid_barrier(gbar, scratch.status, dead);
        p = pn;
        cr = crn;
        w = wn;
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
inline Split choose_split_slots(int64_t nrb, int64_t KC, int W, int64_t slots)
{
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

inline Split choose_split(int64_t nrb, int64_t KC, int W, int minb, int num_sms)
{
    return choose_split_slots(nrb, KC, W, (int64_t)num_sms * minb);
}

// Batch 1: whether CTA pairs (clusters of 2) split each row block's K in
// halves -- few row blocks (at most half the CTA slots) whose halves fit the
// shared unit queue.
template <int W, int MINB> inline bool pair_split_ok(int64_t nrb, int64_t KC, int num_sms)
{
    return MINB == 2 && 2 * nrb <= (int64_t)num_sms * MINB && KC % 2 == 0 && KC / 2 >= 2 &&
           KC / 2 <= queue_cap<W>() && KC < 32768;
}

// Launch the stream-K kernel for a problem of `rows` rows and KC units per row
// block. MINB CTAs of W warps share an SM, so that at a kernel boundary the
// next kernel's CTAs can take the place of this kernel's first finishers and
// start streaming their weights while the rest of this kernel drains.
template <class Pol, int B, int W, int NBUF, int MINB, int OUT>
nm_status launch_streamk(const TensorMaps &maps, void *y, int64_t rows, int64_t KC, const LaunchCtx &ctx)
{
    constexpr int smem = streamk_smem_bytes<Pol, B, W, NBUF>();
    static_assert(MINB * (smem + 1024) <= 232448, "MINB CTAs must fit one SM's shared memory");
    auto kern = streamk_kernel<Pol, B, W, NBUF, MINB, OUT>;
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
    p.y_k = ctx.y_k;
    p.y_v = ctx.y_v;
    p.rows_q = ctx.rows_q;
    p.rows_qk = ctx.rows_q + ctx.rows_k;
    p.U = ((rows + kUnitRows - 1) / kUnitRows) * KC;
    p.scratch = ctx.scratch;
    const int64_t nrb = (rows + kUnitRows - 1) / kUnitRows;
    const Split sp = choose_split(nrb, KC, W, MINB, ctx.num_sms);
    p.whole = sp.whole ? 1 : 0;
    p.P = (int32_t)sp.ctas;
    const int64_t ctas = sp.ctas;
    // the shared queue when every CTA's range fits it (and unit numbers stay small)
    const int64_t most = sp.whole ? ((nrb + ctas - 1) / ctas) * KC : (p.U + ctas - 1) / ctas;
    p.shared_queue = (B == 1 && most <= queue_cap<W>() && KC >= 2 && KC < 32768) ? 1 : 0;
    p.kc_inv = (uint32_t)((((uint64_t)1 << 32) + KC - 1) / KC);
    // Few row blocks (at most half the CTA slots) at batch 1: split each row
    // block's K over a CTA pair, so that each warp's share is half as long.
    const int64_t slots = (int64_t)ctx.num_sms * MINB;
    p.pair_k = (B == 1 && pair_split_ok<W, MINB>(nrb, KC, ctx.num_sms)) ? 1 : 0;
    int64_t grid = ctas;
    if (p.pair_k) {
        p.shared_queue = 1;
        p.whole = 0;
        p.P = (int32_t)(2 * nrb);
        grid = 2 * nrb;
    }
    p.atomic = 0;
    if (OUT == kOutF32 && ctx.splitk_atomic) {
        // Split K over every CTA slot (at least kMinUnitsPerCta units each);
        // the parts of a shared row block meet in y by atomicAdd.
        const int64_t P = std::max<int64_t>(1, std::min<int64_t>(slots, p.U / kMinUnitsPerCta));
        p.atomic = 1;
        p.whole = 0;
        p.pair_k = 0;
        p.P = (int32_t)P;
        grid = P;
        p.shared_queue = (B == 1 && (p.U + P - 1) / P <= queue_cap<W>() && KC >= 2 && KC < 32768) ? 1 : 0;
        if (cudaMemsetAsync(y, 0, (size_t)rows * B * 4, ctx.stream) != cudaSuccess)
            return NM_ERR_CUDA;
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(W * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = ctx.pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension; // CTA pairs (pair_k only)
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pair_k ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, kern, maps, p) != cudaSuccess)
        return NM_ERR_CUDA;
    return NM_OK;
}

// The persistent stack kernel of one configuration: grid size (every CTA
// resident, as a cooperative launch requires), the split of each op over that
// grid, and the launch.
template <class Pol, int B, int W, int NBUF, int MINB> struct StackLauncher {
    static constexpr int kSmem = streamk_smem_bytes<Pol, B, W, NBUF>();
    static_assert(MINB * (kSmem + 1024) <= 232448, "MINB CTAs must fit one SM's shared memory");

    // CTAs of the launch: MINB per SM, fewer if fewer fit.
    static nm_status grid(int num_sms, int *ctas)
    {
        auto kern = stack_kernel<Pol, B, W, NBUF, MINB>;
        static std::once_flag once;
        static cudaError_t attr_err = cudaSuccess;
        std::call_once(once, [&] {
            attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        });
        if (attr_err != cudaSuccess)
            return NM_ERR_CUDA;
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, W * 32, kSmem) != cudaSuccess || occ < 1)
            return NM_ERR_CUDA;
        *ctas = std::min(std::min(occ, MINB) * num_sms, kMaxCtas);
        return NM_OK;
    }

    // Fill op's split fields for a grid of `ctas` CTAs (maps are set by the caller).
    static void split(StackOp *op, void *y, int64_t rows, int64_t KC, int ctas)
    {
        const int64_t nrb = (rows + kUnitRows - 1) / kUnitRows;
        const Split sp = choose_split_slots(nrb, KC, W, ctas);
        op->y = y;
        op->rows = rows;
        op->U = nrb * KC;
        op->KC = (int32_t)KC;
        op->whole = sp.whole ? 1 : 0;
        op->P = (int32_t)std::min<int64_t>(sp.ctas, ctas);
        op->reserved = 0;
    }

    static nm_status launch(const StackOp *ops, int n_ops, uint32_t *gbar, int ctas, const LaunchCtx &ctx)
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)ctas);
        cfg.blockDim = dim3(W * 32);
        cfg.dynamicSmemBytes = kSmem;
        cfg.stream = ctx.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative; // the grid barrier needs every CTA resident
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, stack_kernel<Pol, B, W, NBUF, MINB>, ops, n_ops, gbar, ctx.scratch) !=
            cudaSuccess)
            return NM_ERR_CUDA;
        return NM_OK;
    }
};

// Calls f(std::integral_constant<int, batch>) for batch 1..8.
template <class F> nm_status with_batch(int batch, F &&f)
{
    switch (batch) {
    case 1: return f(std::integral_constant<int, 1>{});
    case 2: return f(std::integral_constant<int, 2>{});
    case 3: return f(std::integral_constant<int, 3>{});
    case 4: return f(std::integral_constant<int, 4>{});
    case 5: return f(std::integral_constant<int, 5>{});
    case 6: return f(std::integral_constant<int, 6>{});
    case 7: return f(std::integral_constant<int, 7>{});
    case 8: return f(std::integral_constant<int, 8>{});
    default: return NM_ERR_UNSUPPORTED;
    }
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
