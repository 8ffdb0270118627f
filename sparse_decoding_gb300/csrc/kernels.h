// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "nm_common.cuh"
#include "nmspmv.h"

namespace nm {

struct LaunchCtx {
    cudaStream_t stream;
    bool pdl;        // launch with programmatic stream serialization
    Scratch scratch; // per-device scratch
    int num_sms;
};

// Which kernel nm_spmv uses for a shape (exposed for tests and tooling).
enum SpmvPath { kSpmvTma = 0, kSpmvSimple = 1 };
SpmvPath spmv_path(int64_t rows, int64_t K);

// Largest grid (CTAs) the SpMV launches on a device with `num_sms` SMs.
int spmv_max_ctas(int num_sms);

nm_status launch_spmv(const uint32_t *masks, const void *values, const void *x, void *y, bool f32out,
                      int64_t rows, int64_t K, int batch, const LaunchCtx &ctx);
nm_status launch_gemv(const void *W, const void *x, void *y, bool f32out, int64_t rows, int64_t K,
                      int batch, const LaunchCtx &ctx);
nm_status launch_select(const void *W, const float *a, int64_t rows, int64_t K, int N, int M,
                        void *out, const LaunchCtx &ctx);
nm_status launch_pack(const void *W, int64_t rows, int64_t K, int N, int M, uint32_t *masks,
                      void *values, const LaunchCtx &ctx);

// Returns the driver's cuTensorMapEncodeTiled, or nullptr if unavailable.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

} // namespace nm
