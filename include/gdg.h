/*
 * gdg.h -- C ABI of the deterministic ragged BF16 grouped GEMM for B300 (sm_103a).
 *
 * The three operations are the rows of the computation table on the "Cake
 * ragged BF16 grouped GEMM (experimental)" docs page; group e of the packed
 * activations covers rows [s_e, t_e) as stated in that page's intro
 * paragraph:
 *
 *   offs_kind == GDG_OFFS_ENDS   : offs[E] cumulative ends,  s_e = offs[e-1] (0 for e = 0), t_e = offs[e]
 *   offs_kind == GDG_OFFS_INDPTR : m_indptr[E+1],            s_e = m_indptr[e], t_e = m_indptr[e+1]
 *
 *   fwd    Y[s_e:t_e]  = X[s_e:t_e] @ W[e]^T     X [rows,K], W [E,N,K] -> Y  [rows,N] bf16
 *   dgrad  dX[s_e:t_e] = G[s_e:t_e] @ W[e]      G [rows,N], W [E,N,K] -> dX [rows,K] bf16
 *   wgrad  dW[e]       = G[s_e:t_e]^T @ X[s_e:t_e]  G, X             -> dW [E,N,K] bf16 or fp32
 *
 * All inputs are bf16, row-major and dense; outputs are row-major with unit
 * stride along the last dimension and may be strided views (out_ld, out_es
 * below).  N and K are multiples of 8 (16-byte rows for the TMA copies);
 * neither needs to be a multiple of a tile.  Products accumulate in fp32 on the tensor cores
 * and every reduction runs in a fixed order with no atomics, so results are
 * bitwise identical from run to run and independent of the GPU's SM count.
 * An empty group gives a weight gradient of exactly +0.0.
 *
 * accumulate (wgrad only) follows the deterministic weight-gradient
 * accumulation section of the MoE grouped GEMM pull request: out[e] +=
 * G[e]^T X[e].  For an fp32 out the stored value is RN32(out + dW) with dW
 * the fp32 weight gradient of the same call with accumulate = 0; for a bf16
 * out it is bf16(float(out) + float(bf16(dW))).  Both are exactly the bits
 * of out.add_(dW) in out's dtype.  The add is fused into the kernel's
 * epilogue: no scratch copy of dW is made.
 *
 * Offsets live in DEVICE memory and are read only by the kernels: the host
 * never synchronises on them.  Groups may be empty, a single row, or any
 * size.  Offsets that are decreasing, negative or beyond rows are not
 * detected (that would need a host sync); the kernels clamp every group to
 * [0, rows] and treat a reversed range as empty, so such input gives
 * unspecified values but never touches memory outside the given buffers.
 * Rows outside every group are never written by fwd / dgrad and never read
 * by wgrad ("row padding").
 *
 * Ownership: the caller owns every buffer (operands, out, offsets,
 * workspace).  The library allocates no device memory, never synchronises
 * the host, and launches only on the given stream.  Every buffer and the
 * stream belong to the calling thread's current device (cudaSetDevice); the
 * tensor maps, the device error word and the launch all use that device.  Calls are stateless and
 * may be captured in a CUDA graph; every launch or replay with accumulate
 * adds again.  New offsets or values written into the same buffers are
 * honoured by the next launch.
 *
 * Errors: every argument check runs on the host before anything is
 * launched; on failure the call returns the status and launches nothing.
 * Asynchronous kernel faults surface through the stream as usual.  Each
 * in-kernel wait is bounded; a wait that runs out records GDG_ETIMEOUT in a
 * device error word that gdg_device_error() returns.
 */
#ifndef GDG_H
#define GDG_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDG_API __attribute__((visibility("default")))
#else
#define GDG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdg_status {
    GDG_OK = 0,
    GDG_EINVAL = 1,     /* null pointer, E outside [1, GDG_MAX_EXPERTS], N/K <= 0, rows outside
                           [0, GDG_MAX_ROWS],
                           bad dtype or offs_kind, fwd/dgrad with fp32 out or accumulate,
                           bad split_rows */
    GDG_EALIGN = 2,     /* N % 8 or K % 8 != 0 (every operand row must start on a 16-byte
                           boundary for the TMA copies), or a pointer not 16-byte aligned.
                           N and K need not be multiples of the 256-wide tiles: the docs
                           page's stable-API rule (N % 256, K % 64) is relaxed, with rows and
                           columns past N or K read as zeros and never written */
    GDG_EOVERLAP = 3,   /* out shares a byte with an input, the offsets or the workspace (the
                           accumulate checks of the MoE grouped GEMM pull request), or two
                           elements of a strided out share memory */
    GDG_EWORKSPACE = 4, /* workspace missing or smaller than grouped_det_gemm_workspace_bytes */
    GDG_ECUDA = 5,      /* a CUDA runtime or driver call failed (launch, tensor map encode) */
    GDG_ETIMEOUT = 6    /* reported by gdg_device_error(): an in-kernel wait ran out */
} gdg_status;

typedef enum gdg_dtype { GDG_BF16 = 0, GDG_FP32 = 1 } gdg_dtype;

typedef enum gdg_offs_kind { GDG_OFFS_ENDS = 0, GDG_OFFS_INDPTR = 1 } gdg_offs_kind;

typedef enum gdg_op { GDG_OP_FWD = 0, GDG_OP_DGRAD = 1, GDG_OP_WGRAD = 2 } gdg_op;

#define GDG_MAX_EXPERTS 1024

/* Largest rows a call takes (2^31 - 1024): every row coordinate a kernel forms, up to a tile
 * past the last row, stays inside the int32 range of the TMA copies. */
#define GDG_MAX_ROWS 2147482624LL

/*
 * Per-call buffers (all device pointers, 16-byte aligned):
 *   fwd:   a = X [rows,K]   b = W [E,N,K]   out = Y  [rows,N] bf16
 *   dgrad: a = G [rows,N]   b = W [E,N,K]   out = dX [rows,K] bf16
 *   wgrad: a = G [rows,N]   b = X [rows,K]  out = dW [E,N,K] bf16 or fp32
 * rows is the host-known number of packed rows (the operands' first
 * dimension); the offsets must not point past it.
 *
 * split_rows (wgrad only; 0 for fwd/dgrad):
 *    0  the library picks the form from the shapes alone (never from the SM count)
 *   -1  one CTA reduces each output tile over all rows of its group
 *   >0  (multiple of 64) every group's rows are cut into consecutive chunks of
 *       split_rows rows; each chunk writes an fp32 partial tile into the
 *       workspace and a second kernel adds the partials in chunk order
 *       p0 + p1 + ... before rounding or accumulating.
 * workspace / workspace_bytes: device scratch for the split form, at least
 * grouped_det_gemm_workspace_bytes(...) bytes; ignored when that is 0.
 *
 * Output strides (the accumulate contract of the MoE grouped GEMM pull request allows a
 * main_grad that is a strided view with unit stride along K): out element (row, col) of
 * fwd / dgrad is at out[row * out_ld + col], element (e, n, k) of wgrad at
 * out[e * out_es + n * out_ld + k]; 0 means the dense value (N or K for out_ld,
 * N * out_ld for out_es).  Each stride times the element size must be a multiple of 16
 * bytes (GDG_EALIGN), and no two output elements may share memory (GDG_EOVERLAP), checked
 * as: taking the row and expert dimensions in increasing order of stride, each stride is at
 * least the span of everything below it (so a permuted [N, E, K] buffer is accepted, rows
 * shorter than a row's columns are not).  Inputs (a, b) are always dense.
 */
typedef struct gdg_args {
    const void* a;
    const void* b;
    void* out;
    void* workspace;
    size_t workspace_bytes;
    int64_t rows;
    int32_t offs_kind;
    int32_t split_rows;
    int64_t out_ld;     /* row stride of out, in elements (0: dense) */
    int64_t out_es;     /* wgrad: expert stride of out, in elements (0: dense); 0 for fwd/dgrad */
} gdg_args;

/* Forward projection (docs page table, row "fwd"). out_dtype must be GDG_BF16 and
 * accumulate 0.  rows == 0 launches nothing.  stream is a cudaStream_t (NULL = legacy
 * default stream). */
GDG_API gdg_status grouped_det_gemm_fwd(const gdg_args* args, const int32_t* offs, int E, int N, int K,
                                gdg_dtype out_dtype, int accumulate, void* stream);

/* Data gradient (docs page table, row "dgrad"; W used as stored, [N,K]).  Same rules
 * as grouped_det_gemm_fwd. */
GDG_API gdg_status grouped_det_gemm_dgrad(const gdg_args* args, const int32_t* offs, int E, int N,
                                  int K, gdg_dtype out_dtype, int accumulate, void* stream);

/* Weight gradient (docs page table, row "wgrad"; accumulate per the MoE grouped GEMM
 * pull request).  Overwrite with rows == 0 writes +0.0 everywhere; accumulate with
 * rows == 0 launches nothing and leaves out unchanged. */
GDG_API gdg_status grouped_det_gemm_wgrad(const gdg_args* args, const int32_t* offs, int E, int N,
                                  int K, gdg_dtype out_dtype, int accumulate, void* stream);

/* Workspace bytes that grouped_det_gemm_<op> needs for these shapes and split_rows
 * (0 unless op is GDG_OP_WGRAD and the split form is chosen).  (size_t)-1 for
 * invalid arguments. */
GDG_API size_t grouped_det_gemm_workspace_bytes(int op, int64_t rows, int E, int N, int K,
                                        gdg_dtype out_dtype, int accumulate, int32_t split_rows);

/* The split_rows value that split_rows == 0 resolves to for these shapes (-1 = unsplit).
 * A split is chosen only when the output has fewer than 64 tiles of 256 x 256
 * (E * ceil(N/256) * ceil(K/256) < 64) and rows >= 6144 * E; it depends on the shapes
 * alone, never on the device.  -1 also for invalid arguments. */
GDG_API int32_t grouped_det_gemm_auto_split_rows(int64_t rows, int E, int N, int K);

/* Static text for a status code. */
GDG_API const char* gdg_status_string(gdg_status status);

/* Synchronises the current device, returns the device error word (GDG_OK or
 * GDG_ETIMEOUT) and clears it. */
GDG_API gdg_status gdg_device_error(void);

/* The device error word without a host synchronisation: enqueues on `stream` (a
 * cudaStream_t of the current device) a 4-byte copy of the word into *dst, then a reset of
 * the word to 0.  dst is device memory or pinned (page-locked) host memory of 4 bytes; once
 * the stream has reached the copy, *dst holds GDG_OK (0) or GDG_ETIMEOUT (6), covering every
 * launch of this device that completed before it.  Nothing is allocated and the call may be
 * captured in a CUDA graph.  Returns GDG_EINVAL for a NULL dst, GDG_ECUDA if enqueueing fails.
 *
 * A pair of CTAs whose wait ran out (GDG_ETIMEOUT) stopped early: the outputs of that launch
 * are unspecified and must not be used. */
GDG_API gdg_status gdg_device_error_async(unsigned int* dst, void* stream);

/*
 * Prepared launches (docs page, "Prepared launches": validate and bind once, then launch any
 * number of times).  gdg_plan_create runs every check of the matching entry point
 * (op = GDG_OP_FWD, GDG_OP_DGRAD or GDG_OP_WGRAD, the same arguments) and binds the result:
 * the kernel form, the encoded tensor maps of the given buffers and the grid.  On failure it
 * returns the entry point's status and sets *plan to NULL.  The plan lives in host memory
 * (the library allocates no device memory) until gdg_plan_destroy.
 *
 * gdg_plan_launch enqueues exactly what the entry point would, on the given stream, with no
 * other host work: it allocates nothing, never synchronises and may be captured in a CUDA
 * graph.  The buffers bound at creation must stay allocated while the plan is used; new
 * offsets or operand values written into them are honoured by every later launch or graph
 * replay, and with accumulate every launch or replay adds again.  The offsets must still
 * describe groups inside the bound rows.  A plan is read-only during launches, so one plan
 * may be launched from several threads; launches that overlap on the GPU and write the same
 * output race like any two kernels writing one buffer.  The first create or call on a device
 * does that device's set-up (kernel attributes, occupancy query): make it before a capture.
 */
typedef struct gdg_plan gdg_plan;

GDG_API gdg_status gdg_plan_create(int op, const gdg_args* args, const int32_t* offs, int E, int N,
                                   int K, gdg_dtype out_dtype, int accumulate, gdg_plan** plan);

/* TEST ONLY (the pages have no counterpart; it exists to test failure detection without a GPU
 * fault): launches the call like grouped_det_gemm_<op> (op = GDG_OP_*), except that the first
 * pipeline stage of CTA pair 0 is armed but never filled.  That pair's bounded waits run out
 * after about 2 s, it aborts cleanly (in-flight copies and MMAs drain, TMEM is freed) and
 * gdg_device_error() then reports GDG_ETIMEOUT; the other pairs finish normally, the context
 * stays usable, and out holds unspecified values.  Never use it for results. */
GDG_API gdg_status gdg_test_withhold_first_stage(int op, const gdg_args* args, const int32_t* offs,
                                                 int E, int N, int K, gdg_dtype out_dtype,
                                                 int accumulate, void* stream);

/* TEST ONLY (no counterpart on the pages): calls and plans made after it use at most `pairs`
 * CTA pairs per launch (0 or less: the device's full persistent grid again).  Process-wide and
 * not synchronised with launches in flight on other threads.  It exists to test that results
 * do not depend on the grid size; it changes only speed. */
GDG_API void gdg_test_set_max_pairs(int pairs);

/* NULL plan: GDG_EINVAL.  A launch failure: GDG_ECUDA. */
GDG_API gdg_status gdg_plan_launch(const gdg_plan* plan, void* stream);

/* Frees a plan (NULL is ignored).  Must not race with a launch of the same plan. */
GDG_API void gdg_plan_destroy(gdg_plan* plan);

/*
 * Non-deterministic weight gradient (the MoE grouped GEMM pull request's non-deterministic
 * package, "Mode rules": its weight gradient may add the row chunks of its split form in an
 * unordered way, every other path runs in a fixed order).  deterministic must be 0 (the
 * caller states that it accepts results that vary from run to run); any other value returns
 * GDG_EINVAL with nothing launched, and the deterministic entry is grouped_det_gemm_wgrad.
 *
 * Arguments, layouts, refusals and split_rows are those of grouped_det_gemm_wgrad.  When the
 * split form is chosen (split_rows > 0, or 0 and the shapes pick it), every row chunk adds
 * its fp32 tile into the result with unordered atomic fp32 adds instead of writing a partial
 * for an ordered reduce: the summation order of the chunks, and so the low bits of dW, vary
 * from run to run, and the adds flush subnormal values to zero.  An fp32 out receives the
 * adds directly (zeroed first unless accumulate); a bf16 out needs an fp32 workspace of
 * grouped_gemm_wgrad_workspace_bytes bytes that receives them, after which dW is rounded to
 * bf16 (and added to out in bf16 with accumulate).  An empty group leaves out as it was
 * (accumulate) or at +0.0.  The unsplit form (split_rows == -1, or 0 and the shapes pick it)
 * is the deterministic kernel, bitwise equal to grouped_det_gemm_wgrad.
 */
GDG_API gdg_status grouped_gemm_wgrad(const gdg_args* args, const int32_t* offs, int E, int N,
                                      int K, gdg_dtype out_dtype, int accumulate,
                                      int deterministic, void* stream);

/* Workspace bytes grouped_gemm_wgrad needs: E * N * K * 4 for a bf16 out in the split form,
 * else 0.  (size_t)-1 for invalid arguments. */
GDG_API size_t grouped_gemm_wgrad_workspace_bytes(int64_t rows, int E, int N, int K,
                                                  gdg_dtype out_dtype, int accumulate,
                                                  int32_t split_rows);

/* Bytes of the library's own fixed scratch used by grouped_det_gemm_wgrad_noalloc. */
#define GDG_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * Weight gradient for callers that cannot allocate device memory.  The pages have no
 * counterpart of this entry point; it exists for this library's users.
 *
 * Some callers cannot call cudaMalloc at the point where they need a weight gradient:
 * code running inside a memory pool or allocator that must not recurse into the driver,
 * runtimes that own all device memory and hand out only the tensors of the step, or
 * hosts where an allocation could block or fail at a bad moment.  The split form of
 * grouped_det_gemm_wgrad needs fp32 scratch for its partial tiles, normally passed as
 * args->workspace.  This variant uses instead one file-scope device array of
 * GDG_NOALLOC_SCRATCH_BYTES bytes inside the library (every GPU that loads the library
 * holds it until the process exits) and allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.  The caller still passes G, X, the offsets and out exactly as
 * for grouped_det_gemm_wgrad; args->workspace and args->workspace_bytes are ignored.
 *
 * It always runs the split form: args->split_rows > 0 (a multiple of 64) is used as given;
 * 0 takes the automatic value (grouped_det_gemm_auto_split_rows) when its partials fit in
 * the scratch, and otherwise the smallest multiple of 64 whose partials fit (partial tiles:
 * ceil(N/256) * ceil(K/256) * (ceil(rows / split_rows) + E), 256 KiB each, at most 64); a
 * negative value is refused with GDG_EINVAL.  A problem whose partials cannot fit
 * (grouped_det_gemm_workspace_bytes for the given or resolved split_rows above
 * GDG_NOALLOC_SCRATCH_BYTES, or ceil(N/256) * ceil(K/256) * (E + 1) > 64) is refused with
 * GDG_EWORKSPACE and nothing is launched.  Results are bitwise equal to
 * grouped_det_gemm_wgrad with the same (resolved) split_rows.
 *
 * The first call on a device looks up the array's device address (once per device, with
 * that device current); make that first call before any stream capture.  Every call shares
 * the one array and it keeps the last call's partials; each call writes every partial tile
 * it later reads, so nothing needs clearing between calls.  Calls whose kernels overlap on
 * the GPU (other streams, other host threads) race on the array and give wrong results:
 * serialise them.
 */
GDG_API gdg_status grouped_det_gemm_wgrad_noalloc(const gdg_args* args, const int32_t* offs,
                                                  int E, int N, int K, gdg_dtype out_dtype,
                                                  int accumulate, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDG_H */
