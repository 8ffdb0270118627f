// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "nm_common.cuh"
#include "nmspmv.h"

namespace nm {

struct LaunchCtx {
    cudaStream_t stream;
    bool pdl;        // launch with programmatic stream serialization
    Scratch scratch; // per-device scratch
    int num_sms;
    // Split K over every CTA slot and add the parts of a shared row block with
    // fp32 atomicAdd into y (fp32 output only; the launcher zeroes y first).
    bool splitk_atomic = false;
    // kOutQkv: rows [0, rows_q) go to y, [rows_q, rows_q + rows_k) to y_k, the rest to y_v.
    void *y_k = nullptr;
    void *y_v = nullptr;
    int64_t rows_q = 0;
    int64_t rows_k = 0;
};

// Which kernel nm_spmv uses for a shape (exposed for tests and tooling).
enum SpmvPath { kSpmvTma = 0, kSpmvSimple = 1 };
SpmvPath spmv_path(int64_t rows, int64_t K);

// Largest grid (CTAs) the SpMV launches on a device with `num_sms` SMs.
int spmv_max_ctas(int num_sms);

// What the SpMV stores: y in bf16, y in fp32, or (gate/up row pairs, see
// nm_spmv_swiglu) h = silu(gate) * up in bf16.
// kOutQkv: bf16 y split by rows into three buffers (see nm_spmv_qkv).
enum OutMode { kOutBf16 = 0, kOutF32 = 1, kOutSwiglu = 2, kOutQkv = 3 };

nm_status launch_spmv(const uint32_t *masks, const void *values, const void *x, void *y, int out, int64_t rows,
                      int64_t K, int batch, const LaunchCtx &ctx);
nm_status launch_gemv(const void *W, const void *x, void *y, bool f32out, int64_t rows, int64_t K,
                      int batch, const LaunchCtx &ctx);
nm_status launch_select(const void *W, const float *a, int64_t rows, int64_t K, int N, int M,
                        void *out, const LaunchCtx &ctx);
nm_status launch_select_pack(const void *W, const float *a, int64_t rows, int64_t K, int N, int M, uint32_t *masks,
                             void *values, const LaunchCtx &ctx);
// pair_off < 0: row r of W is row r of the output; 0 / 16: row r goes to
// (r / 16) * 32 + r % 16 + pair_off (the gate / up half of the pair layout).
nm_status launch_pack(const void *W, int64_t rows, int64_t K, int N, int M, uint32_t *masks,
                      void *values, const LaunchCtx &ctx, int pair_off = -1);

// The persistent stack kernel: a whole decode-token stack in one launch
// (spmv.cu for sparse linears, gemv.cu for dense ones). Only shapes on the
// TMA path qualify (spmv_path == kSpmvTma, gemv_tma_ok).
struct StackOp; // one op's descriptor in device memory (streamk.cuh)
bool gemv_tma_ok(int64_t rows, int64_t K);
// CTAs of the (cooperative) launch for this batch on a device of num_sms SMs.
nm_status stack_grid_sparse(int batch, int num_sms, int *ctas);
nm_status stack_grid_dense(int batch, int num_sms, int *ctas);
// Descriptor of one op for a launch of `ctas` CTAs, written to host memory.
nm_status stack_encode_sparse(const nm_linear &op, int batch, int ctas, StackOp *out);
nm_status stack_encode_dense(const nm_linear &op, int batch, int ctas, StackOp *out);
// One launch over ops[0..n_ops) (device memory); gbar: the grid-barrier counter.
nm_status stack_launch_sparse(const StackOp *ops, int n_ops, int batch, uint32_t *gbar, int ctas,
                              const LaunchCtx &ctx);
nm_status stack_launch_dense(const StackOp *ops, int n_ops, int batch, uint32_t *gbar, int ctas,
                             const LaunchCtx &ctx);

// Launches `kern` on `st` with programmatic dependent launch: it may be
// scheduled while the previous kernel on the stream finishes, so it must run
// pdl_wait_upstream() (griddepcontrol.wait) before it reads or writes anything
// earlier work on the stream touches. The chains of short dependent kernels of
// the OBS pruning hide their launch latency this way.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---- tensor-core GEMM of the OBS pruning (tc_gemm.cu) ----
// Structure flags (coordinates of the GEMM itself: C row i, column j, k
// index kk): kTcALower: A[i][kk] = 0 for kk > i; kTcBLower: B[j][kk] = 0 for
// kk > j; kTcBUpper: B[j][kk] = 0 for kk < j (B as the N x k operand);
// kTcCLower: only the 128 x 128 tiles on and below the diagonal are written
// (nothing reads the others); kTcCSym: C is symmetric, the tiles on and below
// the diagonal are computed and the others written as their transposes.
constexpr unsigned kTcALower = 1u, kTcBLower = 2u, kTcBUpper = 4u, kTcCLower = 8u, kTcCSym = 16u;
// C = alpha A B^T + beta C: A bf16 [M][kt][nparts][64], B bf16 [N][kt][nparts][64]
// (nparts 1, or 3 for fp32 emulated: the bf16 parts of each 64-column k-tile
// side by side), C fp32 with row stride ldc (16-byte aligned, N and ldc
// multiples of 4). k_base: the global k index of this call's first column,
// against which the flags' triangles are placed. A bounded wait that runs
// out sets NM_ERR_TIMEOUT in *status.
nm_status tc_gemm_bf16(const uint16_t *A, const uint16_t *B, int64_t kt, int nparts, float *C, int64_t ldc, int64_t M,
                       int64_t N, float alpha, float beta, uint32_t *status, cudaStream_t st, unsigned flags = 0,
                       int64_t k_base = 0);
// fp32 C = alpha A op(B) + beta C with fp32 emulated by bf16 parts (six
// products): A (M x k) row-major with stride lda (a_trans: stored k x M);
// op(B) = B^T for B (N x k) row-major, or B for B (k x N) row-major when
// b_trans. work_a / work_b: tc_operand_bytes(M or N, k, true) bytes each
// (the k range is done in chunks of 1024, whose results add up in C).
// flags: as for tc_gemm_bf16, for A and op(B)^T.
nm_status tc_gemm_f32(const float *A, int64_t lda, bool a_trans, const float *B, int64_t ldb, bool b_trans, int64_t M,
                      int64_t N, int64_t k, float *C, int64_t ldc, float alpha, float beta, uint16_t *work_a,
                      uint16_t *work_b, uint32_t *status, cudaStream_t st, unsigned flags = 0);
size_t tc_operand_bytes(int64_t rows, int64_t k, bool emulated);
// Xt [K][Tp] = X^T (bf16 X [T][K]), zero in columns T .. Tp.
nm_status tc_transpose_bf16(const uint16_t *X, int64_t T, int64_t K, uint16_t *Xt, int64_t Tp, cudaStream_t st);
// The same product for small shapes (32 x 32 tiles, double-buffered k steps).
nm_status simt_small_f32(const float *A, int64_t lda, const float *B, int64_t ldb, bool b_kn, int64_t M, int64_t N,
                         int64_t k, float *C, int64_t ldc, float alpha, float beta, cudaStream_t st);
// The same product in plain fp32 on the CUDA cores (b_kn: B stored k x N).
nm_status simt_gemm_f32(const float *A, int64_t lda, const float *B, int64_t ldb, bool b_kn, int64_t M, int64_t N,
                        int64_t k, float *C, int64_t ldc, float alpha, float beta, cudaStream_t st);
// The library scratch's status word on the current device (allocated if need be).
nm_status library_status_word(uint32_t **status);

// The static scratch of nm_spmv_noalloc on device `dev`, if a call has set it
// up there (noalloc.cu).
bool noalloc_scratch(int dev, Scratch *out);

// Returns the driver's cuTensorMapEncodeTiled, or nullptr if unavailable.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

} // namespace nm
