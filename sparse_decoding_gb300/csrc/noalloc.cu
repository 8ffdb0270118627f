// noalloc.cu -- nm_spmv_noalloc: the decode SpMV for callers that cannot
// allocate device memory.
//
// nm_spmv keeps its stream-K scratch (partial sums of row blocks split between
// CTAs, their counters, a status word) in a buffer the library obtains with
// cudaMalloc on first use. Some callers cannot allow that: code that runs
// inside another framework's memory pool, or under a policy that forbids any
// allocation outside its own. This entry point gives them the same kernel with
// the scratch in a statically sized device array instead. The array belongs
// to the loaded library image: every GPU that loads the library holds it until
// the process exits, and no call allocates or frees anything.
#include <mutex>

#include "kernels.h"

namespace nm {

// Room for the stream-K scratch of up to kNoAllocMaxCtas CTAs.
constexpr int kNoAllocMaxCtas = 512;

// The Scratch layout below indexes counters and partials by CTA with the
// stride of the library's own scratch (kMaxCtas counters), so the array keeps
// that layout: status, kMaxCtas counters, then partials. Only the first
// kNoAllocMaxCtas counters and partial slots are ever used.
constexpr size_t kNoAllocArrayBytes =
    kScratchStatusBytes + kScratchCounterBytes + sizeof(float) * (size_t)kNoAllocMaxCtas * kPartialFloats;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocArrayBytes];

constexpr int kNoAllocMaxDevices = 64;
static std::mutex g_noalloc_mu;
static void *g_noalloc_ptr[kNoAllocMaxDevices];
static int g_noalloc_sms[kNoAllocMaxDevices];

// Device address of the array and the SM count, looked up once per device
// (with that device current). In host code the array's name only stands in
// for the symbol; the kernel must be given the address returned here.
static nm_status noalloc_setup(int dev, void **ptr, int *sms)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return NM_ERR_CUDA;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return NM_ERR_CUDA;
        g_noalloc_sms[dev] = n;
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    *sms = g_noalloc_sms[dev];
    return NM_OK;
}

// For nm_device_status: the array's status word and counters on this device
// if a call has set it up there (no lookup otherwise: nothing to report).
bool noalloc_scratch(int dev, Scratch *out)
{
    if (dev < 0 || dev >= kNoAllocMaxDevices)
        return false;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev])
        return false;
    *out = scratch_from_base(g_noalloc_ptr[dev]);
    return true;
}

} // namespace nm

extern "C" nm_status nm_spmv_noalloc(const uint32_t *masks, const void *values_bf16, const void *x_bf16,
                                     void *y_bf16, int64_t rows, int64_t K, int batch, void *stream)
{
    using namespace nm;
    if (rows < 0 || K < 0 || (K % 32) != 0)
        return NM_ERR_SHAPE;
    if (batch < 1 || batch > 8)
        return NM_ERR_UNSUPPORTED;
    if (rows == 0)
        return NM_OK;
    if (!y_bf16 || (K > 0 && (!masks || !values_bf16 || !x_bf16)))
        return NM_ERR_INVALID_ARG;
    const auto a16 = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
    if (!a16(y_bf16) || (K > 0 && (!a16(masks) || !a16(values_bf16) || !a16(x_bf16))))
        return NM_ERR_ALIGN;
    cudaStream_t st = (cudaStream_t)stream;
    if (K == 0)
        return cudaMemsetAsync(y_bf16, 0, (size_t)rows * batch * 2, st) == cudaSuccess ? NM_OK : NM_ERR_CUDA;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
        return NM_ERR_CUDA;
    void *base = nullptr;
    int sms = 0;
    nm_status s = noalloc_setup(dev, &base, &sms);
    if (s != NM_OK)
        return s;
    // The array has room for kNoAllocMaxCtas stream-K CTAs.
    if (spmv_max_ctas(sms) > kNoAllocMaxCtas)
        return NM_ERR_UNSUPPORTED;

    LaunchCtx ctx;
    ctx.stream = st;
    ctx.pdl = false;
    ctx.scratch = scratch_from_base(base);
    ctx.num_sms = sms;
    // The array keeps whatever the previous call left; the counters must start at zero.
    if (cudaMemsetAsync(ctx.scratch.counters, 0, sizeof(uint32_t) * kNoAllocMaxCtas, st) != cudaSuccess)
        return NM_ERR_CUDA;
    s = launch_spmv(masks, values_bf16, x_bf16, y_bf16, kOutBf16, rows, K, batch, ctx);
    if (s == NM_OK && cudaGetLastError() != cudaSuccess)
        s = NM_ERR_CUDA;
    return s;
}
