// api.cu -- the library's C entry points (declared in include/nmspmv.h):
// argument checks, the per-device scratch, and dispatch to the kernels.
#include <mutex>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "kernels.h"
#include "streamk.cuh"

namespace nm {

// An NVTX range over one C entry point (visible in a timeline profiler; a
// no-op when no tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

constexpr int kMaxDevices = 64;

static std::mutex g_mu;
static void *g_scratch[kMaxDevices];
static int g_num_sms[kMaxDevices];

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

static bool pattern_ok(int N, int M)
{
    return (N == 2 && M == 4) || (N == 4 && M == 8) || (N == 8 && M == 16) || (N == 16 && M == 32);
}

// Scratch and SM count of the current device; allocates the scratch on first use.
static nm_status device_ctx(cudaStream_t stream, bool pdl, LaunchCtx *ctx)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return NM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch[dev]) {
        void *p = nullptr;
        if (cudaMalloc(&p, kScratchBytes) != cudaSuccess)
            return NM_ERR_CUDA;
        if (cudaMemset(p, 0, kScratchBytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
            cudaFree(p);
            return NM_ERR_CUDA;
        }
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
            cudaFree(p);
            return NM_ERR_CUDA;
        }
        g_num_sms[dev] = sms;
        g_scratch[dev] = p;
    }
    ctx->stream = stream;
    ctx->pdl = pdl;
    ctx->scratch = scratch_from_base(g_scratch[dev]);
    ctx->num_sms = g_num_sms[dev];
    return NM_OK;
}

nm_status library_status_word(uint32_t **status)
{
    LaunchCtx ctx;
    nm_status s = device_ctx(nullptr, false, &ctx);
    if (s == NM_OK)
        *status = ctx.scratch.status;
    return s;
}

EncodeTiledFn encode_tiled_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    });
    return fn;
}

static nm_status check_spmv_args(const void *masks, const void *values, const void *x, const void *y,
                                 int64_t rows, int64_t K, int batch)
{
    if (rows < 0 || K < 0 || (K % 32) != 0)
        return NM_ERR_SHAPE;
    if (batch < 1 || batch > 8)
        return NM_ERR_UNSUPPORTED;
    if (rows == 0)
        return NM_OK;
    if (!y || (K > 0 && (!masks || !values || !x)))
        return NM_ERR_INVALID_ARG;
    if (!aligned16(y) || (K > 0 && (!aligned16(masks) || !aligned16(values) || !aligned16(x))))
        return NM_ERR_ALIGN;
    return NM_OK;
}

static nm_status check_gemv_args(const void *W, const void *x, const void *y, int64_t rows, int64_t K, int batch)
{
    if (rows < 0 || K < 0 || (K % 32) != 0)
        return NM_ERR_SHAPE;
    if (batch < 1 || batch > 8)
        return NM_ERR_UNSUPPORTED;
    if (rows == 0)
        return NM_OK;
    if (!y || (K > 0 && (!W || !x)))
        return NM_ERR_INVALID_ARG;
    if (!aligned16(y) || (K > 0 && (!aligned16(W) || !aligned16(x))))
        return NM_ERR_ALIGN;
    return NM_OK;
}

// The three output parts of nm_spmv_qkv: row counts and buffers.
static nm_status check_qkv_parts(const void *q, const void *k, const void *v, int64_t rows_q, int64_t rows_k,
                                 int64_t rows_v)
{
    if (rows_q < 0 || rows_k < 0 || rows_v < 0)
        return NM_ERR_SHAPE;
    if ((rows_q > 0 && !q) || (rows_k > 0 && !k) || (rows_v > 0 && !v))
        return NM_ERR_INVALID_ARG;
    if ((rows_q > 0 && !aligned16(q)) || (rows_k > 0 && !aligned16(k)) || (rows_v > 0 && !aligned16(v)))
        return NM_ERR_ALIGN;
    return NM_OK;
}

// One op of a stack: the checks of its call, and its flags.
static nm_status check_stack_op(const nm_linear &o, bool dense, int batch)
{
    if (o.flags & ~(uint32_t)(NM_LINEAR_SWIGLU | NM_LINEAR_QKV))
        return NM_ERR_INVALID_ARG;
    if ((o.flags & NM_LINEAR_SWIGLU) && (o.flags & NM_LINEAR_QKV))
        return NM_ERR_INVALID_ARG;
    if (dense) {
        if (o.flags)
            return NM_ERR_INVALID_ARG;
        return check_gemv_args(o.W, o.x, o.y, o.rows, o.K, batch);
    }
    if ((o.flags & NM_LINEAR_SWIGLU) && o.rows % 32 != 0)
        return NM_ERR_SHAPE;
    if (o.flags & NM_LINEAR_QKV) {
        const int64_t rows_v = o.rows - o.rows_q - o.rows_k;
        nm_status s = check_qkv_parts(o.y, o.y_k, o.y_v, o.rows_q, o.rows_k, rows_v);
        if (s != NM_OK)
            return s;
        if (o.rows == 0)
            return NM_OK;
        if (o.K > 0 && (!o.masks || !o.values || !o.x))
            return NM_ERR_INVALID_ARG;
        if (o.K > 0 && (!aligned16(o.masks) || !aligned16(o.values) || !aligned16(o.x)))
            return NM_ERR_ALIGN;
        return (o.K < 0 || o.K % 32 != 0) ? NM_ERR_SHAPE : (batch < 1 || batch > 8) ? NM_ERR_UNSUPPORTED : NM_OK;
    }
    return check_spmv_args(o.masks, o.values, o.x, o.y, o.rows, o.K, batch);
}

// The output parts of a kOutQkv launch.
struct QkvOut {
    void *y_k = nullptr;
    void *y_v = nullptr;
    int64_t rows_q = 0;
    int64_t rows_k = 0;
};

static nm_status zero_output(void *y, int64_t rows, int batch, size_t elt, cudaStream_t stream)
{
    return cudaMemsetAsync(y, 0, (size_t)rows * batch * elt, stream) == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}

// out: kOutBf16, kOutF32, or kOutSwiglu (rows = gate/up pair rows, y = h [batch][rows / 2]).
static nm_status spmv_impl(const uint32_t *masks, const void *values, const void *x, void *y, int out, int64_t rows,
                           int64_t K, int batch, cudaStream_t stream, bool pdl, bool splitk_atomic = false,
                           const QkvOut *qkv = nullptr)
{
    nm_status s;
    if (out == kOutQkv) { // y is the q part and may be NULL when it has no rows: checked by the caller
        if (rows < 0 || K < 0 || (K % 32) != 0)
            return NM_ERR_SHAPE;
        if (batch < 1 || batch > 8)
            return NM_ERR_UNSUPPORTED;
        if (rows == 0)
            return NM_OK;
        if (K > 0 && (!masks || !values || !x))
            return NM_ERR_INVALID_ARG;
        if (K > 0 && (!aligned16(masks) || !aligned16(values) || !aligned16(x)))
            return NM_ERR_ALIGN;
    } else if ((s = check_spmv_args(masks, values, x, y, rows, K, batch)) != NM_OK || rows == 0) {
        return s;
    }
    if (out == kOutSwiglu && rows % 32 != 0)
        return NM_ERR_SHAPE;
    if (K == 0) {
        if (out == kOutQkv) {
            const int64_t rows_v = rows - qkv->rows_q - qkv->rows_k;
            if ((qkv->rows_q > 0 && (s = zero_output(y, qkv->rows_q, batch, 2, stream)) != NM_OK) ||
                (qkv->rows_k > 0 && (s = zero_output(qkv->y_k, qkv->rows_k, batch, 2, stream)) != NM_OK) ||
                (rows_v > 0 && (s = zero_output(qkv->y_v, rows_v, batch, 2, stream)) != NM_OK))
                return s;
            return NM_OK;
        }
        return out == kOutSwiglu ? zero_output(y, rows / 2, batch, 2, stream)
                                 : zero_output(y, rows, batch, out == kOutF32 ? 4 : 2, stream);
    }
    LaunchCtx ctx;
    if ((s = device_ctx(stream, pdl, &ctx)) != NM_OK)
        return s;
    ctx.splitk_atomic = splitk_atomic;
    if (qkv) {
        ctx.y_k = qkv->y_k;
        ctx.y_v = qkv->y_v;
        ctx.rows_q = qkv->rows_q;
        ctx.rows_k = qkv->rows_k;
    }
    s = launch_spmv(masks, values, x, y, out, rows, K, batch, ctx);
    if (s == NM_OK && cudaGetLastError() != cudaSuccess)
        s = NM_ERR_CUDA;
    return s;
}

// Pack Wa (Wb == NULL), or the gate/up pair Wa, Wb (rows rows each) into the pair layout.
static nm_status pack_impl(const void *Wa, const void *Wb, int64_t rows, int64_t K, int N, int M, uint32_t *masks,
                           void *values_bf16, void *stream)
{
    if (!pattern_ok(N, M))
        return NM_ERR_UNSUPPORTED;
    if (rows < 0 || K < 0 || (K % 32) != 0)
        return NM_ERR_SHAPE;
    if (rows == 0 || K == 0)
        return NM_OK;
    if (!Wa || !masks || !values_bf16)
        return NM_ERR_INVALID_ARG;
    if (!aligned16(Wa) || (Wb && !aligned16(Wb)) || !aligned16(masks) || !aligned16(values_bf16))
        return NM_ERR_ALIGN;
    LaunchCtx ctx;
    nm_status s = device_ctx((cudaStream_t)stream, false, &ctx);
    if (s != NM_OK)
        return s;
    // One pack at a time per process: the error flag lives in the shared scratch.
    static std::mutex pack_mu;
    std::lock_guard<std::mutex> lock(pack_mu);
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(ctx.scratch.status + 1, 0, sizeof(uint32_t), st) != cudaSuccess)
        return NM_ERR_CUDA;
    if ((s = launch_pack(Wa, rows, K, N, M, masks, values_bf16, ctx, Wb ? 0 : -1)) != NM_OK)
        return s;
    if (Wb && (s = launch_pack(Wb, rows, K, N, M, masks, values_bf16, ctx, 16)) != NM_OK)
        return s;
    uint32_t bad = 0;
    if (cudaMemcpyAsync(&bad, ctx.scratch.status + 1, sizeof bad, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return NM_ERR_CUDA;
    return bad ? NM_ERR_NOT_NM : NM_OK;
}

static nm_status gemv_impl(const void *W, const void *x, void *y, bool f32out, int64_t rows, int64_t K, int batch,
                           cudaStream_t stream, bool pdl)
{
    nm_status s = check_gemv_args(W, x, y, rows, K, batch);
    if (s != NM_OK || rows == 0)
        return s;
    if (K == 0)
        return zero_output(y, rows, batch, f32out ? 4 : 2, stream);
    LaunchCtx ctx;
    if ((s = device_ctx(stream, pdl, &ctx)) != NM_OK)
        return s;
    s = launch_gemv(W, x, y, f32out, rows, K, batch, ctx);
    if (s == NM_OK && cudaGetLastError() != cudaSuccess)
        s = NM_ERR_CUDA;
    return s;
}

} // namespace nm

using namespace nm;

// A prepared decode-token stack (opaque in the C ABI).
struct nm_stack_plan {
    int dev = 0;
    int batch = 1;
    bool dense = false;
    int n_ops = 0;
    bool persistent = false;  // one launch of the stack kernel; otherwise chained launches
    int ctas = 0;             // grid of the persistent launch
    void *dmem = nullptr;     // StackOp[n_ops], then the grid-barrier counter
    StackOp *ops_dev = nullptr;
    uint32_t *gbar = nullptr;
    std::vector<nm_linear> ops; // host copy for the chained path
    cudaGraphExec_t exec = nullptr; // the chained launches, captured once
};

// Capture the plan's chained launches (PDL edges included) into a graph on a
// private stream. On any failure the plan keeps launching directly.
static void capture_chain(nm_stack_plan *pl)
{
    cudaStream_t cs = nullptr;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    cudaGraph_t g = nullptr;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
        nm_status s = pl->dense ? dense_gemv_stack(pl->ops.data(), pl->n_ops, pl->batch, cs)
                                : nm_spmv_stack(pl->ops.data(), pl->n_ops, pl->batch, cs);
        if (cudaStreamEndCapture(cs, &g) != cudaSuccess || s != NM_OK) {
            if (g)
                cudaGraphDestroy(g);
            g = nullptr;
        }
    }
    if (g && cudaGraphInstantiate(&pl->exec, g, 0) != cudaSuccess)
        pl->exec = nullptr;
    if (g)
        cudaGraphDestroy(g);
    cudaStreamDestroy(cs);
    cudaGetLastError(); // a failed capture leaves no error behind
}

extern "C" {

int nm_abi_version(void) { return 4; }

const char *nm_status_str(int status)
{
    switch (status) {
    case NM_OK: return "ok";
    case NM_ERR_INVALID_ARG: return "invalid argument";
    case NM_ERR_SHAPE: return "bad shape (sizes must be >= 0 and K a multiple of 32)";
    case NM_ERR_ALIGN: return "pointer not 16-byte aligned";
    case NM_ERR_UNSUPPORTED: return "unsupported N:M pattern or batch size";
    case NM_ERR_NOT_NM: return "an M-subgroup holds more than N nonzeros";
    case NM_ERR_CUDA: return "CUDA error";
    case NM_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
    case NM_ERR_NOT_PD: return "the damped Hessian is not positive definite";
    case NM_ERR_BOUNDS: return "a kernel skipped an access outside its buffer (bounds-checking build)";
    default: return "unknown status";
    }
}

nm_status nm_select(const void *W_bf16, const float *a, int64_t rows, int64_t K, int N, int M, void *W_pruned,
                    void *stream)
{
    NvtxRange nvtx_("nm_select");
    if (!pattern_ok(N, M))
        return NM_ERR_UNSUPPORTED;
    if (rows < 0 || K < 0 || (K % 32) != 0)
        return NM_ERR_SHAPE;
    if (rows == 0 || K == 0)
        return NM_OK;
    if (!W_bf16 || !a || !W_pruned)
        return NM_ERR_INVALID_ARG;
    if (!aligned16(W_bf16) || !aligned16(a) || !aligned16(W_pruned))
        return NM_ERR_ALIGN;
    LaunchCtx ctx;
    nm_status s = device_ctx((cudaStream_t)stream, false, &ctx);
    if (s != NM_OK)
        return s;
    return launch_select(W_bf16, a, rows, K, N, M, W_pruned, ctx);
}

nm_status nm_select_pack(const void *W_bf16, const float *a, int64_t rows, int64_t K, int N, int M, uint32_t *masks,
                         void *values_bf16, void *stream)
{
    NvtxRange nvtx_("nm_select_pack");
    if (!pattern_ok(N, M))
        return NM_ERR_UNSUPPORTED;
    if (rows < 0 || K < 0 || (K % 32) != 0)
        return NM_ERR_SHAPE;
    if (rows == 0 || K == 0)
        return NM_OK;
    if (!W_bf16 || !a || !masks || !values_bf16)
        return NM_ERR_INVALID_ARG;
    if (!aligned16(W_bf16) || !aligned16(a) || !aligned16(masks) || !aligned16(values_bf16))
        return NM_ERR_ALIGN;
    LaunchCtx ctx;
    nm_status s = device_ctx((cudaStream_t)stream, false, &ctx);
    if (s != NM_OK)
        return s;
    return launch_select_pack(W_bf16, a, rows, K, N, M, masks, values_bf16, ctx);
}

nm_status nm_pack(const void *W_bf16, int64_t rows, int64_t K, int N, int M, uint32_t *masks, void *values_bf16,
                  void *stream)
{
    NvtxRange nvtx_("nm_pack");
    return pack_impl(W_bf16, nullptr, rows, K, N, M, masks, values_bf16, stream);
}

nm_status nm_pack_swiglu(const void *W_gate_bf16, const void *W_up_bf16, int64_t rows_h, int64_t K, int N, int M,
                         uint32_t *masks, void *values_bf16, void *stream)
{
    NvtxRange nvtx_("nm_pack_swiglu");
    if (rows_h % 16 != 0)
        return NM_ERR_SHAPE;
    if (rows_h > 0 && K > 0 && !W_up_bf16)
        return NM_ERR_INVALID_ARG;
    return pack_impl(W_gate_bf16, W_up_bf16, rows_h, K, N, M, masks, values_bf16, stream);
}

nm_status nm_spmv_swiglu(const uint32_t *masks, const void *values_bf16, const void *x_bf16, void *h_bf16,
                         int64_t rows_h, int64_t K, int batch, void *stream)
{
    NvtxRange nvtx_("nm_spmv_swiglu");
    if (rows_h < 0 || rows_h % 16 != 0)
        return NM_ERR_SHAPE;
    return spmv_impl(masks, values_bf16, x_bf16, h_bf16, kOutSwiglu, 2 * rows_h, K, batch, (cudaStream_t)stream,
                     false);
}

nm_status nm_spmv(const uint32_t *masks, const void *values_bf16, const void *x_bf16, void *y_bf16, int64_t rows,
                  int64_t K, int batch, void *stream)
{
    NvtxRange nvtx_("nm_spmv");
    return spmv_impl(masks, values_bf16, x_bf16, y_bf16, kOutBf16, rows, K, batch, (cudaStream_t)stream, false);
}

nm_status nm_spmv_f32out(const uint32_t *masks, const void *values_bf16, const void *x_bf16, float *y_f32,
                         int64_t rows, int64_t K, int batch, void *stream)
{
    NvtxRange nvtx_("nm_spmv_f32out");
    return spmv_impl(masks, values_bf16, x_bf16, y_f32, kOutF32, rows, K, batch, (cudaStream_t)stream, false);
}

nm_status nm_spmv_qkv(const uint32_t *masks, const void *values_bf16, const void *x_bf16, void *q_bf16, void *k_bf16,
                      void *v_bf16, int64_t rows_q, int64_t rows_k, int64_t rows_v, int64_t K, int batch, void *stream)
{
    NvtxRange nvtx_("nm_spmv_qkv");
    nm_status s = check_qkv_parts(q_bf16, k_bf16, v_bf16, rows_q, rows_k, rows_v);
    if (s != NM_OK)
        return s;
    QkvOut qo;
    qo.y_k = k_bf16;
    qo.y_v = v_bf16;
    qo.rows_q = rows_q;
    qo.rows_k = rows_k;
    return spmv_impl(masks, values_bf16, x_bf16, q_bf16, kOutQkv, rows_q + rows_k + rows_v, K, batch,
                     (cudaStream_t)stream, false, false, &qo);
}

nm_status nm_spmv_f32out_atomic(const uint32_t *masks, const void *values_bf16, const void *x_bf16, float *y_f32,
                                int64_t rows, int64_t K, int batch, void *stream)
{
    NvtxRange nvtx_("nm_spmv_f32out_atomic");
    return spmv_impl(masks, values_bf16, x_bf16, y_f32, kOutF32, rows, K, batch, (cudaStream_t)stream, false, true);
}

nm_status dense_gemv(const void *W_bf16, const void *x_bf16, void *y_bf16, int64_t rows, int64_t K, int batch,
                     void *stream)
{
    NvtxRange nvtx_("dense_gemv");
    return gemv_impl(W_bf16, x_bf16, y_bf16, false, rows, K, batch, (cudaStream_t)stream, false);
}

nm_status dense_gemv_f32out(const void *W_bf16, const void *x_bf16, float *y_f32, int64_t rows, int64_t K,
                            int batch, void *stream)
{
    NvtxRange nvtx_("dense_gemv_f32out");
    return gemv_impl(W_bf16, x_bf16, y_f32, true, rows, K, batch, (cudaStream_t)stream, false);
}

nm_status nm_spmv_stack(const nm_linear *ops, int n_ops, int batch, void *stream)
{
    NvtxRange nvtx_("nm_spmv_stack");
    if (n_ops < 0 || (n_ops > 0 && !ops))
        return NM_ERR_INVALID_ARG;
    for (int i = 0; i < n_ops; ++i) {
        nm_status s = check_stack_op(ops[i], false, batch);
        if (s != NM_OK)
            return s;
    }
    for (int i = 0; i < n_ops; ++i) {
        const nm_linear &o = ops[i];
        QkvOut qo;
        qo.y_k = o.y_k;
        qo.y_v = o.y_v;
        qo.rows_q = o.rows_q;
        qo.rows_k = o.rows_k;
        const int out = (o.flags & NM_LINEAR_SWIGLU) ? kOutSwiglu : (o.flags & NM_LINEAR_QKV) ? kOutQkv : kOutBf16;
        nm_status s = spmv_impl(o.masks, o.values, o.x, o.y, out, o.rows, o.K, batch, (cudaStream_t)stream, true, false,
                                out == kOutQkv ? &qo : nullptr);
        if (s != NM_OK)
            return s;
    }
    return NM_OK;
}

nm_status dense_gemv_stack(const nm_linear *ops, int n_ops, int batch, void *stream)
{
    NvtxRange nvtx_("dense_gemv_stack");
    if (n_ops < 0 || (n_ops > 0 && !ops))
        return NM_ERR_INVALID_ARG;
    for (int i = 0; i < n_ops; ++i) {
        nm_status s = check_stack_op(ops[i], true, batch);
        if (s != NM_OK)
            return s;
    }
    for (int i = 0; i < n_ops; ++i) {
        nm_status s = gemv_impl(ops[i].W, ops[i].x, ops[i].y, false, ops[i].rows, ops[i].K, batch,
                                (cudaStream_t)stream, true);
        if (s != NM_OK)
            return s;
    }
    return NM_OK;
}

nm_status nm_stack_plan_create(const nm_linear *ops, int n_ops, int batch, unsigned flags, nm_stack_plan **plan)
{
    NvtxRange nvtx_("nm_stack_plan_create");
    if (!plan || n_ops < 0 || (n_ops > 0 && !ops) || (flags & ~(NM_STACK_DENSE | NM_STACK_PERSISTENT)))
        return NM_ERR_INVALID_ARG;
    const bool dense = (flags & NM_STACK_DENSE) != 0;
    bool fits = n_ops > 0 && (flags & NM_STACK_PERSISTENT);
    for (int i = 0; i < n_ops; ++i) {
        const nm_linear &o = ops[i];
        nm_status s = check_stack_op(o, dense, batch);
        if (s != NM_OK)
            return s;
        // the persistent kernel stores plain bf16 y only
        fits = fits && o.flags == 0 &&
               (dense ? gemv_tma_ok(o.rows, o.K) : (o.rows > 0 && o.K > 0 && spmv_path(o.rows, o.K) == kSpmvTma));
    }
    if (n_ops == 0 && (batch < 1 || batch > 8))
        return NM_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    nm_status s = device_ctx(nullptr, false, &ctx);
    if (s != NM_OK)
        return s;
    nm_stack_plan *pl = new (std::nothrow) nm_stack_plan;
    if (!pl)
        return NM_ERR_CUDA;
    if (cudaGetDevice(&pl->dev) != cudaSuccess) {
        delete pl;
        return NM_ERR_CUDA;
    }
    pl->batch = batch;
    pl->dense = dense;
    pl->n_ops = n_ops;
    pl->ops.assign(ops, ops + n_ops);
    pl->persistent = fits;
    if (fits) {
        s = dense ? stack_grid_dense(batch, ctx.num_sms, &pl->ctas) : stack_grid_sparse(batch, ctx.num_sms, &pl->ctas);
        std::vector<StackOp> host(n_ops);
        for (int i = 0; i < n_ops && s == NM_OK; ++i)
            s = dense ? stack_encode_dense(ops[i], batch, pl->ctas, &host[i])
                      : stack_encode_sparse(ops[i], batch, pl->ctas, &host[i]);
        const size_t desc_bytes = ((sizeof(StackOp) * n_ops + 255) / 256) * 256;
        if (s == NM_OK && cudaMalloc(&pl->dmem, desc_bytes + 256) != cudaSuccess) {
            pl->dmem = nullptr;
            s = NM_ERR_CUDA;
        }
        if (s == NM_OK) {
            pl->ops_dev = (StackOp *)pl->dmem;
            pl->gbar = (uint32_t *)((char *)pl->dmem + desc_bytes);
            if (cudaMemcpy(pl->ops_dev, host.data(), sizeof(StackOp) * n_ops, cudaMemcpyHostToDevice) != cudaSuccess ||
                cudaMemset(pl->gbar, 0, 256) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
                s = NM_ERR_CUDA;
        }
        if (s != NM_OK) {
            if (pl->dmem)
                cudaFree(pl->dmem);
            delete pl;
            return s;
        }
    }
    if (!fits && n_ops > 0)
        capture_chain(pl);
    *plan = pl;
    return NM_OK;
}

nm_status nm_stack_plan_run(const nm_stack_plan *plan, void *stream)
{
    NvtxRange nvtx_("nm_stack_plan_run");
    if (!plan)
        return NM_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return NM_ERR_CUDA;
    if (dev != plan->dev)
        return NM_ERR_INVALID_ARG;
    if (!plan->persistent) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (plan->exec && cudaStreamIsCapturing((cudaStream_t)stream, &cap) == cudaSuccess &&
            cap == cudaStreamCaptureStatusNone)
            return cudaGraphLaunch(plan->exec, (cudaStream_t)stream) == cudaSuccess ? NM_OK : NM_ERR_CUDA;
        cudaGetLastError();
        return plan->dense ? dense_gemv_stack(plan->ops.data(), plan->n_ops, plan->batch, stream)
                           : nm_spmv_stack(plan->ops.data(), plan->n_ops, plan->batch, stream);
    }
    LaunchCtx ctx;
    nm_status s = device_ctx((cudaStream_t)stream, false, &ctx);
    if (s != NM_OK)
        return s;
    s = plan->dense ? stack_launch_dense(plan->ops_dev, plan->n_ops, plan->batch, plan->gbar, plan->ctas, ctx)
                    : stack_launch_sparse(plan->ops_dev, plan->n_ops, plan->batch, plan->gbar, plan->ctas, ctx);
    if (s == NM_OK && cudaGetLastError() != cudaSuccess)
        s = NM_ERR_CUDA;
    return s;
}

nm_status nm_stack_plan_destroy(nm_stack_plan *plan)
{
    NvtxRange nvtx_("nm_stack_plan_destroy");
    if (!plan)
        return NM_OK;
    nm_status s = NM_OK;
    if (plan->exec) {
        int cur = -1;
        cudaGetDevice(&cur);
        cudaSetDevice(plan->dev);
        if (cudaDeviceSynchronize() != cudaSuccess || cudaGraphExecDestroy(plan->exec) != cudaSuccess)
            s = NM_ERR_CUDA;
        if (cur >= 0)
            cudaSetDevice(cur);
    }
    if (plan->dmem) {
        int cur = -1;
        cudaGetDevice(&cur);
        cudaSetDevice(plan->dev);
        if (cudaDeviceSynchronize() != cudaSuccess || cudaFree(plan->dmem) != cudaSuccess)
            s = NM_ERR_CUDA;
        if (cur >= 0)
            cudaSetDevice(cur);
    }
    delete plan;
    return s;
}

// Read and clear a scratch's status word on `st`; after a timeout also clear
// its stream-K counters (a kernel that gave up may have left them mid-count).
static nm_status read_clear_status(const Scratch &sc, size_t counter_bytes, cudaStream_t st)
{
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, sc.status, sizeof word, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemsetAsync(sc.status, 0, sizeof word, st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
        return NM_ERR_CUDA;
    if (!(word & (1u << NM_ERR_TIMEOUT)))
        return (word & (1u << NM_ERR_BOUNDS)) ? NM_ERR_BOUNDS : NM_OK;
    if (cudaMemsetAsync(sc.counters, 0, counter_bytes, st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
        return NM_ERR_CUDA;
    return NM_ERR_TIMEOUT;
}

nm_status nm_device_status(void *stream)
{
    NvtxRange nvtx_("nm_device_status");
    cudaStream_t st = (cudaStream_t)stream;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return NM_ERR_CUDA;
    // nm_spmv_noalloc's static scratch, if a call has set it up on this device
    Scratch na;
    nm_status s_na = NM_OK;
    const bool have_na = noalloc_scratch(dev, &na);
    if (have_na && (s_na = read_clear_status(na, kScratchCounterBytes, st)) == NM_ERR_CUDA)
        return s_na;
    bool have_lib;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        have_lib = g_scratch[dev] != nullptr;
    }
    if (have_na && !have_lib)
        return s_na; // allocate nothing for a caller that only uses nm_spmv_noalloc
    LaunchCtx ctx;
    nm_status s = device_ctx(st, false, &ctx);
    if (s != NM_OK)
        return s;
    s = read_clear_status(ctx.scratch, kScratchCounterBytes, st);
    if (s == NM_OK)
        s = s_na;
    return s;
}

} // extern "C"
