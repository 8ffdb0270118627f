/*
 * nmspmv.h -- C ABI of the GB300 (sm_103a) bitmask N:M decode SpMV library.
 *
 * The operation is the decode-time sparse matrix-vector product of
 * SparseDecoding ("Decoding-Aware Pruning for Accurate and Efficient LLM
 * Inference"): weights pruned to a 50% N:M pattern are stored row by row as
 * 32-bit bitmasks plus the kept values, and each decode step multiplies them
 * with the current token's activations (paper.rainbus.top summary, section
 * "方法步骤详情", steps 3-4; ai.info summary, "Methodology in Plain English",
 * steps 2-3).
 *
 * Storage format (the ABI format):
 *   masks  : uint32 [rows][K/32], row-major. Bit j (LSB = 0) of word g of row r
 *            is set when column 32g+j is kept.
 *   values : bf16   [rows][K/2],  row-major. values[r][16g+k] is the k-th kept
 *            weight of word g, counting set bits from the LSB (ascending
 *            column order). Every word has exactly 16 set bits.
 *   x      : bf16   [batch][K],   one contiguous row per token.
 *   y      : bf16 (or fp32) [batch][rows].
 *
 * Conventions for every call below:
 *   - bf16 data is passed as raw 16-bit patterns (uint16_t / void *).
 *   - Device pointers are caller-owned device memory; the library never frees
 *     them. Host pointers are caller-owned host memory.
 *   - Every pointer that the call reads or writes must be 16-byte aligned
 *     (NM_ERR_ALIGN otherwise). Pointers may be NULL only when the call has
 *     nothing to read or write through them (rows == 0).
 *   - K must be a multiple of 32 (NM_ERR_SHAPE). rows, K >= 0.
 *   - (N, M) must be one of (2,4), (4,8), (8,16), (16,32) (NM_ERR_UNSUPPORTED):
 *     the 50% patterns with M <= 32 dividing the word.
 *   - batch must be 1..8 (NM_ERR_UNSUPPORTED).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Device calls
 *     are asynchronous on it unless stated otherwise.
 *   - A failed CUDA call or launch returns NM_ERR_CUDA. No kernel spin-waits
 *     without a bound: a bounded wait that runs out records NM_ERR_TIMEOUT in
 *     a per-device status word that nm_device_status() reports.
 *   - The library keeps one small scratch buffer per device (the stream-K
 *     partial sums and their counters, and the pack error flag). It is
 *     allocated by the first call on that device that needs it and kept until
 *     the process exits; make that first call outside CUDA graph capture.
 *     Calls that use it must not run concurrently on different streams of the
 *     same device.
 */
#ifndef NMSPMV_H
#define NMSPMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nm_status {
    NM_OK = 0,
    NM_ERR_INVALID_ARG = 1, /* NULL where data is needed, bad count */
    NM_ERR_SHAPE = 2,       /* K % 32 != 0, negative size */
    NM_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
    NM_ERR_UNSUPPORTED = 4, /* (N, M) not a 50% pattern, batch outside 1..8 */
    NM_ERR_NOT_NM = 5,      /* an M-subgroup holds more than N nonzeros */
    NM_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed */
    NM_ERR_TIMEOUT = 7,     /* a kernel's bounded wait ran out */
    NM_ERR_NOT_PD = 8,      /* nm_obs_prune: the damped Hessian is not positive definite */
    NM_ERR_BOUNDS = 9       /* reported only by the bounds-checking build (NM_BOUNDS_CHECK): a
                               kernel found an index outside its buffer and skipped the access */
} nm_status;

/* Version of this ABI (bumped on any incompatible change). */
int nm_abi_version(void);

/* Human-readable name of a status code; never NULL. */
const char *nm_status_str(int status);

/*
 * nm_pack_host -- bitmask conversion on the host (paper.rainbus.top summary,
 * "方法步骤详情" step 3: each pruned row becomes a compact value array plus
 * 32-bit bitmasks whose set bits mark the kept weights).
 *   W_bf16 : host, bf16 [rows][K], the pruned dense matrix (read).
 *   masks  : host, uint32 [rows][K/32] (written).
 *   values : host, bf16 [rows][K/2] (written).
 * A weight is kept when it is nonzero (+0 and -0 count as zero; NaN and Inf
 * as nonzero). An M-subgroup with fewer than N nonzeros is filled up to N with
 * its lowest-index zero positions; kept values are copied bit for bit.
 * Returns NM_ERR_NOT_NM when an aligned M-subgroup holds more than N
 * nonzeros (outputs then unspecified). Synchronous, no CUDA.
 */
nm_status nm_pack_host(const uint16_t *W_bf16, int64_t rows, int64_t K, int N, int M,
                       uint32_t *masks, uint16_t *values);

/*
 * nm_select -- Wanda N:M selection on the GPU (daiwk.github.io notes,
 * section "核心公式": score s_ij = |W_ij| * sqrt(sum_t X_jt^2), keep N per
 * M-column group, no weight update).
 *   W_bf16   : device, bf16 [rows][K] (read).
 *   a        : device, fp32 [K], the per-column activation norm (read).
 *   W_pruned : device, bf16 [rows][K] (written); may equal W_bf16 (in place).
 * In every aligned M-column subgroup of every row the N entries with the
 * largest fp32 score |W| * a_j are kept (bit for bit) and the others become
 * +0. Larger score wins; a NaN score counts as larger than any number; equal
 * scores go to the lower column index. Asynchronous.
 */
nm_status nm_select(const void *W_bf16, const float *a, int64_t rows, int64_t K, int N, int M,
                    void *W_pruned, void *stream);

/*
 * nm_select_pack -- nm_select and nm_pack in one pass over W (the selection
 * rule of the daiwk.github.io notes, section "核心公式", then the bitmask
 * conversion of the paper.rainbus.top summary, "方法步骤详情" step 3).
 *   W_bf16 : device, bf16 [rows][K], the dense weights (read).
 *   a      : device, fp32 [K], the per-column activation norm (read).
 *   masks, values_bf16 : device (written), as nm_pack writes them for the
 *            matrix nm_select would return.
 * (N, M) must be a 50% pattern (NM_ERR_UNSUPPORTED otherwise). The result is
 * bit-identical with nm_select followed by nm_pack, without the pruned matrix
 * being written and read back. The mask word is the selection's keep mask,
 * except where a kept weight is zero and outranks a lower-index zero (possible
 * only with a NaN or infinite column norm), where the pack's fill rule
 * decides. It cannot be NM_ERR_NOT_NM: the rule keeps N per subgroup.
 * Asynchronous.
 */
nm_status nm_select_pack(const void *W_bf16, const float *a, int64_t rows, int64_t K, int N, int M, uint32_t *masks,
                         void *values_bf16, void *stream);

/*
 * nm_pack -- bitmask conversion on the GPU, bit-exact with nm_pack_host.
 *   W_bf16 : device, bf16 [rows][K] (read). masks, values_bf16: device (written).
 * Synchronous with respect to `stream`: it waits for the stream so that it can
 * report NM_ERR_NOT_NM. Uses the per-device scratch (error flag).
 */
nm_status nm_pack(const void *W_bf16, int64_t rows, int64_t K, int N, int M, uint32_t *masks,
                  void *values_bf16, void *stream);

/*
 * nm_spmv -- decode SpMV over the bitmask format (paper.rainbus.top summary,
 * "核心方法" and "方法步骤详情" step 4; ai.info summary, "Methodology in Plain
 * English" step 3): for each mask word, 16 fixed steps each take the next set
 * bit as the column of the next kept value and multiply-accumulate.
 *   y[b][r] = sum_j W[r][j] * x[b][j] for b < batch, accumulated in fp32 and
 *   rounded to bf16 (nearest even).
 *   masks, values_bf16, x_bf16: device (read). y_bf16: device (written).
 * Masks are not validated: on words that do not hold exactly 16 set bits, y is
 * unspecified but no access leaves the caller's buffers. The summation order
 * is fixed for a given device and shape (the result is repeatable).
 * Asynchronous. Uses the per-device scratch (stream-K partial sums).
 */
nm_status nm_spmv(const uint32_t *masks, const void *values_bf16, const void *x_bf16,
                  void *y_bf16, int64_t rows, int64_t K, int batch, void *stream);

/* As nm_spmv, but y is the fp32 accumulator before rounding: float [batch][rows]. */
nm_status nm_spmv_f32out(const uint32_t *masks, const void *values_bf16, const void *x_bf16,
                         float *y_f32, int64_t rows, int64_t K, int batch, void *stream);

/*
 * nm_spmv_f32out_atomic -- nm_spmv_f32out computed as a split reduction with
 * atomicAdd (paper.rainbus.top summary, "方法步骤详情" step 4, where the
 * decode kernel splits a reduction and combines it with atomicAdd when
 * needed). The K range of every row block is split over all CTA slots of the
 * device (at least 8 units of 32 rows x 256 columns each); the CTAs that
 * share a row block add their partial sums into y with fp32 atomicAdd after
 * the call has zeroed y on `stream`. Arguments, layouts and errors are those
 * of nm_spmv_f32out; the result obeys the same error bound, but the order of
 * the additions (and so the last bits) may change from call to call.
 * nm_spmv_f32out's default combine is the deterministic one: the last CTA to
 * finish a shared row block adds all parts in CTA order.
 */
nm_status nm_spmv_f32out_atomic(const uint32_t *masks, const void *values_bf16, const void *x_bf16, float *y_f32,
                                int64_t rows, int64_t K, int batch, void *stream);

/*
 * dense_gemv -- the dense bf16 reference on the same GPU (the pages' 1.00x
 * baseline: aitest123.com article, Table 3; ai.info summary, Main Findings).
 *   W_bf16: device bf16 [rows][K]; x_bf16: device bf16 [batch][K];
 *   y: device bf16 [batch][rows] (fp32 accumulation, rounded to nearest even).
 * Asynchronous.
 */
nm_status dense_gemv(const void *W_bf16, const void *x_bf16, void *y_bf16, int64_t rows,
                     int64_t K, int batch, void *stream);

/* As dense_gemv with the fp32 accumulator as output: float [batch][rows]. */
nm_status dense_gemv_f32out(const void *W_bf16, const void *x_bf16, float *y_f32, int64_t rows,
                            int64_t K, int batch, void *stream);

/*
 * One linear of a decode-token stack. `W` is the dense bf16 matrix for the
 * dense stack and unused (may be NULL) for the sparse one; `masks`/`values`
 * are the packed form for the sparse stack and unused for the dense one.
 */
typedef struct nm_linear {
    const uint32_t *masks;
    const void *values; /* bf16 [rows][K/2] */
    const void *W;      /* bf16 [rows][K] */
    const void *x;      /* bf16 [batch][K] */
    void *y;            /* bf16 [batch][rows] ([batch][rows/2] with NM_LINEAR_SWIGLU;
                           the q part [batch][rows_q] with NM_LINEAR_QKV) */
    int64_t rows;
    int64_t K;
    uint32_t flags;     /* 0, NM_LINEAR_SWIGLU or NM_LINEAR_QKV (sparse ops only) */
    void *y_k;          /* NM_LINEAR_QKV: bf16 [batch][rows_k]; unused otherwise */
    void *y_v;          /* NM_LINEAR_QKV: bf16 [batch][rows - rows_q - rows_k]; unused otherwise */
    int64_t rows_q;     /* NM_LINEAR_QKV: rows of the q and k parts; unused otherwise */
    int64_t rows_k;
} nm_linear;

/* The op is a gate/up pair matrix in the pair layout of nm_pack_swiglu
 * (rows = 2 * rows_h, a multiple of 32) and stores h as nm_spmv_swiglu does. */
#define NM_LINEAR_SWIGLU 1u
/* The op stores its rows in three buffers (y, y_k, y_v) as nm_spmv_qkv does. */
#define NM_LINEAR_QKV 2u

/*
 * nm_spmv_stack / dense_gemv_stack -- the linear stack of one decode token
 * (every pruned linear of every layer; only linear layers are sparse, per the
 * ai.info summary, "Methodology" step 4 and paper.rainbus.top "局限与改进").
 * Runs ops[0..n_ops) in order on `stream`, each as nm_spmv / dense_gemv (an op
 * with NM_LINEAR_SWIGLU as nm_spmv_swiglu, one with NM_LINEAR_QKV as
 * nm_spmv_qkv; dense ops take flags 0).
 * Consecutive launches are chained with programmatic dependent launch: a
 * kernel may start streaming its own weights before the previous one ends,
 * but reads its x only after the previous kernel has completed, exactly as if
 * x were that kernel's output. `ops` is host memory, read during the call.
 * The sequence may be captured into a CUDA graph by the caller.
 */
nm_status nm_spmv_stack(const nm_linear *ops, int n_ops, int batch, void *stream);
nm_status dense_gemv_stack(const nm_linear *ops, int n_ops, int batch, void *stream);

/*
 * nm_pack_swiglu / nm_spmv_swiglu -- an MLP's gate and up projections as one
 * SpMV whose epilogue applies the SwiGLU activation, so that its output h is
 * directly the x of the down projection. Not described on the pages, whose
 * kernel is the plain SpMV; this is the step after it in a decode layer (only
 * the linear layers are pruned: ai.info summary, "Methodology in Plain
 * English" step 4).
 *
 * Pair layout: the packed matrix has 2 * rows_h rows; row block t (rows 32t ..
 * 32t+31) holds gate rows 16t .. 16t+15 followed by up rows 16t .. 16t+15, so
 * that each gate row and its up row meet in one row block.
 *   nm_pack_swiglu: W_gate, W_up: device bf16 [rows_h][K], pruned (read);
 *     masks: uint32 [2*rows_h][K/32], values: bf16 [2*rows_h][K/2] (written)
 *     in the pair layout. rows_h % 16 == 0 (NM_ERR_SHAPE). Otherwise as
 *     nm_pack (synchronous; NM_ERR_NOT_NM as there).
 *   nm_spmv_swiglu: masks, values in the pair layout; x: bf16 [batch][K];
 *     h: bf16 [batch][rows_h] (written) with
 *       g = sum_j W_gate[r][j] x[b][j],  u = sum_j W_up[r][j] x[b][j]  (fp32),
 *       h[b][r] = bf16_rn(g / (1 + exp(-g)) * u)                       (fp32).
 *     rows_h % 16 == 0 (NM_ERR_SHAPE). Otherwise as nm_spmv (asynchronous).
 */
nm_status nm_pack_swiglu(const void *W_gate_bf16, const void *W_up_bf16, int64_t rows_h, int64_t K, int N, int M,
                         uint32_t *masks, void *values_bf16, void *stream);
nm_status nm_spmv_swiglu(const uint32_t *masks, const void *values_bf16, const void *x_bf16, void *h_bf16,
                         int64_t rows_h, int64_t K, int batch, void *stream);

/*
 * nm_spmv_qkv -- nm_spmv of a fused q/k/v projection whose output goes to
 * three buffers, one per projection, so that each is contiguous per token at
 * any batch size (the step after the SpMV in a decode layer's attention
 * block; the pages prune only the linear layers: ai.info summary,
 * "Methodology in Plain English" step 4).
 *   masks, values_bf16: the packed matrix of rows_q + rows_k + rows_v rows
 *     (the q rows, then the k rows, then the v rows); x_bf16: [batch][K].
 *   q_bf16 [batch][rows_q], k_bf16 [batch][rows_k], v_bf16 [batch][rows_v]:
 *     device bf16 (written); row r of the product goes to q when r < rows_q,
 *     to k row r - rows_q when r < rows_q + rows_k, else to v row
 *     r - rows_q - rows_k. Values and summation order are nm_spmv's.
 * A part with no rows may be NULL. Errors and the rest as for nm_spmv
 * (NM_ERR_SHAPE for a negative row count). Asynchronous.
 */
nm_status nm_spmv_qkv(const uint32_t *masks, const void *values_bf16, const void *x_bf16, void *q_bf16, void *k_bf16,
                      void *v_bf16, int64_t rows_q, int64_t rows_k, int64_t rows_v, int64_t K, int batch, void *stream);

/*
 * nm_stack_plan -- a decode-token stack prepared once, run many times.
 * The linears, their order and the dependency rule are those of
 * nm_spmv_stack / dense_gemv_stack: op i+1 reads its x only after every part
 * of op i's y has been stored. Two ways to run it:
 *   default: one kernel per op, chained with programmatic dependent launch
 *     (as nm_spmv_stack; the fastest on GB300 for decode-sized ops). The
 *     chain is captured once into a CUDA graph when the plan is created, and
 *     each run launches that graph (one host call instead of one per op);
 *     a run on a stream that is itself being captured launches the kernels
 *     one by one instead, so the caller's graph records them;
 *   NM_STACK_PERSISTENT: one persistent cooperative kernel walks all ops; a
 *     grid-wide barrier stands in for each kernel boundary, and each warp
 *     starts streaming the next op's weights before it arrives there. Used
 *     only when every op is on the TMA path (sparse: K % 128 == 0; dense:
 *     K % 64 == 0; rows, K > 0); otherwise the plan runs the default way.
 *
 * nm_stack_plan_create -- validates ops[0..n_ops) (host memory, read during
 *   the call; each op as for nm_spmv, or dense_gemv with NM_STACK_DENSE, with
 *   `batch` rows of x) and prepares the plan; with NM_STACK_PERSISTENT it
 *   encodes every op's descriptors into device memory that the plan owns
 *   (cudaMalloc; synchronous); by default it captures the chained launches
 *   on a private stream (nothing runs). The plan holds the ops' device pointers: the
 *   buffers must stay allocated, and each run reads and writes whatever they
 *   hold then. Make this call outside CUDA graph capture, on the device the
 *   plan will run on. *plan is set on NM_OK only. Errors: those of the per-op
 *   checks, NM_ERR_INVALID_ARG (NULL plan, n_ops < 0, unknown flag),
 *   NM_ERR_CUDA.
 * nm_stack_plan_run -- runs the plan on `stream` (asynchronous). The current
 *   device must be the plan's (NM_ERR_INVALID_ARG otherwise). Runs of one
 *   plan, and runs of different plans or other calls of this library on the
 *   same device, must not overlap on the GPU (they share the per-device
 *   scratch, and a persistent plan its barrier word). May be captured in a
 *   CUDA graph. A bounded wait that runs out is reported by nm_device_status.
 * nm_stack_plan_destroy -- frees the plan (waits for the device first);
 *   NULL is accepted.
 */
typedef struct nm_stack_plan nm_stack_plan;

#define NM_STACK_DENSE 1u      /* ops are dense GEMVs (W), not sparse SpMVs */
#define NM_STACK_PERSISTENT 2u /* one persistent launch per run */

nm_status nm_stack_plan_create(const nm_linear *ops, int n_ops, int batch, unsigned flags, nm_stack_plan **plan);
nm_status nm_stack_plan_run(const nm_stack_plan *plan, void *stream);
nm_status nm_stack_plan_destroy(nm_stack_plan *plan);

/*
 * nm_spmv_noalloc -- nm_spmv for callers that cannot allocate device memory.
 * The pages describe no such entry point; it exists for integration only.
 * nm_spmv obtains its per-device scratch with cudaMalloc on first use. Code
 * that runs inside another framework's memory pool, or under a rule that no
 * allocation may happen outside it, cannot allow that. This call computes the
 * same y (same kernel, same summation order) with its scratch in a fixed
 * device array that is part of the loaded library: about 1 MB on every GPU
 * that loads the library, held until the process exits. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   Arguments, layouts and errors are those of nm_spmv. Asynchronous.
 *   Limit: the array holds the scratch of 512 CTAs; on a device whose grid
 *   would need more (over 256 SMs) the call returns NM_ERR_UNSUPPORTED.
 *   The first call on a device looks up the array's device address (with that
 *   device current); make that first call outside CUDA graph capture.
 *   Every call on a device shares the one array and finds it as the previous
 *   call left it; each call clears the counters it needs at its start (one
 *   2 KB cudaMemsetAsync on `stream` before the kernel). Calls whose
 *   executions overlap on the GPU (other streams, or other host threads) race
 *   on the array: serialize them. A bounded wait that runs out is reported by
 *   nm_device_status (below), which reads and clears the array's status word
 *   as well as the library scratch's.
 */
nm_status nm_spmv_noalloc(const uint32_t *masks, const void *values_bf16, const void *x_bf16,
                          void *y_bf16, int64_t rows, int64_t K, int batch, void *stream);

/*
 * nm_device_status -- waits for `stream`, then returns and clears the status
 * words of the current device: NM_ERR_TIMEOUT if any kernel's bounded wait ran
 * out since the last call, NM_ERR_BOUNDS if (in the bounds-checking build) a
 * kernel skipped an access outside its buffer, NM_OK otherwise (NM_ERR_CUDA if
 * CUDA failed). It
 * covers the library scratch and, once nm_spmv_noalloc has run on the device,
 * that call's static array. After a timeout it also clears the stream-K
 * counters (outputs of the calls that ran meanwhile are unspecified); call it
 * before reusing the device. It allocates the library scratch if that does not
 * exist yet -- except on a device where only nm_spmv_noalloc has run, where it
 * reads that call's array alone and allocates nothing.
 */
nm_status nm_device_status(void *stream);

/*
 * ---- N:M pruning by the OBS rule: the step that produces the weights ----
 *
 * A layer is pruned against the Hessian of its calibration inputs, H = 2 X X^T
 * (paper.rainbus.top summary, "前置知识" on the OBS framework and "方法步骤详情"
 * step 2; ai.info summary, "Methodology in Plain English" step 1). Removing
 * weight q costs w_q^2 / (2 [H^-1]_qq) and the remaining weights move by
 * -(w_q / [H^-1]_qq) H^-1_{:,q}; SparseGPT applies the rule column by column.
 * Readings where the pages stop (SparseGPT's published procedure):
 *   - columns are fixed left to right; at column j the inverse is that of the
 *     still-free columns, inv(H[j:, j:]);
 *   - at the first column of every aligned M-column group, each row keeps the
 *     N weights with the largest w_c^2 / [inv(H[c:, c:])]_00, using the values
 *     as compensated so far; equal saliencies keep the lower column;
 *   - damping: a zero diagonal entry (an input that is always zero) becomes 1
 *     and its weights 0, then percdamp * mean(diag H) is added to the diagonal.
 */

/* Flag of nm_obs_prune: the GEMM-shaped steps (the factorisation's off-diagonal
 * blocks and the lazy trailing updates) run in plain fp32 on the CUDA cores
 * instead of fp32 emulated on the bf16 tensor cores (the default: each fp32
 * operand split into three bf16 parts, the six products of order up to 2
 * accumulated in fp32 in tensor memory, k in chunks of 1024 added in fp32). */
#define NM_OBS_SGEMM 1u

/*
 * nm_obs_hessian -- H = 2 X^T X for calibration inputs X, or H += 2 X^T X.
 *   X_bf16 : device, bf16 [T][K], one row per calibration token (read).
 *   H      : device, fp32 [K][K], symmetric (written; accumulated into when
 *            `accumulate` is nonzero, so long calibration sets go in chunks).
 * Products are exact; sums are fp32 (one bf16 pass on the tensor cores; the
 * tiles on and below the diagonal are computed and mirrored). T == 0 writes
 * zeros (or leaves H as it is when accumulating). K must be a multiple of 32;
 * T and K at most 2^31 - 1. Workspace: X transposed, 2 K ceil(T/64)*64 bytes
 * from the library's workspace pool. Asynchronous on `stream`. Calls on one
 * device are serialized by a lock.
 */
nm_status nm_obs_hessian(const void *X_bf16, int64_t T, int64_t K, float *H, int accumulate, void *stream);

/*
 * nm_obs_prune -- N:M pruning of one linear layer by the OBS rule above.
 *   W_bf16      : device, bf16 [rows][K], the dense weights (read).
 *   H           : device, fp32 [K][K], the symmetric calibration Hessian (read).
 *                 W and H must be finite (outputs are unspecified otherwise).
 *   N, M        : keep N of every aligned M columns; M in {2, 4, 8, 16, 32},
 *                 1 <= N <= M (NM_ERR_UNSUPPORTED otherwise). The decode
 *                 format wants the 50% patterns 2:4, 4:8, 8:16, 16:32.
 *   percdamp    : damping fraction, >= 0 and finite (0.01 is SparseGPT's).
 *   flags       : 0 or NM_OBS_SGEMM.
 *   W_out_bf16  : device, bf16 [rows][K] (written): the pruned weights, removed
 *                 entries +0. This is what nm_pack / nm_pack_host take.
 *   keep_masks  : device, uint32 [rows][K/32] or NULL (written): bit j of word g
 *                 is set when column 32g + j is kept (the decode mask format).
 *   W_out_f32   : device, fp32 [rows][K] or NULL (written): the pruned weights
 *                 in fp32, before the rounding to bf16.
 * Arithmetic is fp32: the Cholesky factorisation of the reversed Hessian, the
 * inverses it needs, the column sweep and the GEMM-shaped steps all run in
 * this library's kernels (the GEMMs on the tensor cores with fp32 emulated,
 * see NM_OBS_SGEMM). Workspace: 12 K^2 + 4 rows K + 4096 rows bytes, plus
 * 6144 (max(rows, K/2) + K) bytes for the GEMMs' split operands (none with
 * NM_OBS_SGEMM), taken from the library's workspace pool and returned to it
 * before the call ends (the pool keeps the memory for the next call; see
 * nm_obs_release_workspace). SYNCHRONOUS: returns after the result is written (NM_ERR_NOT_PD when
 * the damped Hessian cannot be factorised; outputs are then unspecified).
 * Calls on one device are serialized by a lock. Pointers 16-byte aligned
 * (NM_ERR_ALIGN).
 */
nm_status nm_obs_prune(const void *W_bf16, const float *H, int64_t rows, int64_t K, int N, int M, float percdamp,
                       unsigned flags, void *W_out_bf16, uint32_t *keep_masks, float *W_out_f32, void *stream);

/*
 * nm_obs_release_workspace -- returns to the device the memory that
 * nm_obs_prune and nm_obs_hessian keep for their workspaces. Those calls take
 * their workspaces from a library-owned stream-ordered pool on the current
 * device that keeps what it has mapped between calls (mapping several GB
 * afresh cost every call time); this trims the pool to the memory still in use
 * by work in flight. Calls on one device are serialized by a lock.
 */
nm_status nm_obs_release_workspace(void);

#ifdef __cplusplus
}
#endif

#endif /* NMSPMV_H */
