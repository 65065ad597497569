/*
 * tg_gemm.h -- C ABI of libtg_gemm.so, a tiled matrix multiply for GB300
 * (sm_103a).
 *
 * The operation is the tiled GEMM that the TileLang pages use as their
 * running example: C[M,N] = A[M,K] x B[K,N], row-major, fp16 (or fp32)
 * inputs, fp32 accumulation, fp16 or fp32 output.  Sources:
 *   - "企业官网建设流程全解析" (cf-1.com, a TileLang article), §3.3: the
 *     matmul kernel clears an fp32 fragment, pipelines the K loop over
 *     copy-A / copy-B / gemm, and copies the fragment out to an fp16 C.
 *   - "TileLang实战：用Python DSL自动生成高性能GPU计算内核" (gsyq.cn), §3.1:
 *     the fp32 128x128x128 triple loop C[i,j] += A[i,k] * B[k,j]; §3.3: the
 *     tensor-core variant with fp16 inputs and an fp32 result.
 *   - gsyq.cn/news/429607 (DeepSeek / Ascend TileLang toolchain article),
 *     §3.3: unaligned sizes such as M=127, N=255 must work.
 *
 * No symbol here takes or returns a framework type: plain pointers, sizes
 * and a CUDA stream handle.
 */
#ifndef TG_GEMM_H
#define TG_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (cudaStream_t / CUstream).  0 is the legacy default
 * stream. */
typedef void* tg_stream_t;

typedef enum {
    TG_F16 = 1, /* IEEE-754 binary16 */
    TG_F32 = 2, /* IEEE-754 binary32 */
    TG_E4M3 = 3 /* 8-bit float E4M3 (OCP FP8: bias 7, max 448, no infinities);
                   an input type only */
} tg_dtype;

typedef enum {
    TG_OK = 0,
    TG_ERR_INVALID_ARG = 1, /* bad size, pointer, leading dimension or aliasing */
    TG_ERR_UNSUPPORTED = 2, /* dtype pair or size the library does not handle */
    TG_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
    TG_ERR_TIMEOUT = 4      /* a kernel gave up on a bounded wait (device flag) */
} tg_status;

/*
 * tg_gemm -- C = A x B.
 *
 * Arguments
 *   M, N, K   problem sizes, each in [0, 2^31 - 1024].
 *   A         device pointer, M rows of K elements, row i at A + i*lda.
 *   lda       row stride of A in elements, lda >= K.
 *   B         device pointer, K rows of N elements, row k at B + k*ldb.
 *   ldb       row stride of B in elements, ldb >= N.
 *   C         device pointer, M rows of N elements, row i at C + i*ldc.
 *   ldc       row stride of C in elements, ldc >= N.
 *   in_dtype  element type of A and B.
 *   out_dtype element type of C.
 *   stream    CUDA stream the work is enqueued on.
 *
 * Semantics: C is overwritten with the product (no alpha/beta, no
 * accumulation into C), as in the pages' kernel, which clears its
 * accumulator and copies it out.  Accumulation is in fp32 in every path; the
 * fp32 -> fp16 output conversion rounds to nearest even.  Elements of C
 * between column N and the row stride ldc are never written.
 *
 * Supported dtype pairs: (F16 -> F16) and (F16 -> F32) run on the tensor
 * cores; (F32 -> F32) runs on the SIMT fp32 path; (E4M3 -> F16) and
 * (E4M3 -> F32) run on the tensor cores (tcgen05 kind::f8f6f4, fp32
 * accumulation).  Any other pair returns TG_ERR_UNSUPPORTED.  For fp16 and
 * fp32 inputs, pointer alignment and leading dimensions never cause an
 * error: operands that the TMA engine cannot address (base not 16-byte
 * aligned, or a row stride that is not a multiple of 16 bytes) go to a
 * predicated-load boundary kernel instead.  E4M3 inputs run on the TMA
 * kernels only: their bases must be 16-byte aligned and lda, ldb multiples
 * of 16, else TG_ERR_UNSUPPORTED.  The 8-bit path stands in for the INT8
 * GEMM that "TileLang：GPU异构计算的声明式分块编程范式" (kwkr.cn), §5.5,
 * discusses: GB300's tcgen05 has no integer MMA.
 *
 * Degenerate sizes: M == 0 or N == 0 is a no-op returning TG_OK (pointers
 * may then be NULL).  K == 0 writes zeros to C (the empty sum); A and B may
 * then be NULL.
 *
 * Errors (checked on the host before anything is enqueued; nothing is
 * written when an error is returned):
 *   TG_ERR_INVALID_ARG  a negative size; a NULL pointer that would be read
 *                       or written; a pointer that is not a multiple of its
 *                       element size; lda < K, ldb < N or ldc < N; or the
 *                       byte span of C overlapping the span of A or of B.
 *   TG_ERR_UNSUPPORTED  an unsupported dtype pair, a size above 2^31 - 1024,
 *                       or E4M3 operands the TMA engine cannot address.
 *   TG_ERR_CUDA         a CUDA call made while launching failed.
 *
 * Ownership and memory: the caller owns A, B and C.  The library allocates
 * no device memory per call; it keeps only per-device launch attributes, a
 * 4-byte device error word for bounded-wait failures (its address looked up
 * on the first call on each device), and a host-side cache of encoded TMA
 * descriptors keyed by pointer, sizes and strides (a repeated call with the
 * same operands skips the encoding).  This per-device state belongs to the
 * device's primary context: after cudaDeviceReset on a device, do not call
 * the library on that device again in the same process.
 *
 * Asynchrony: the call only enqueues work on `stream` and returns; it never
 * synchronizes.  A kernel that times out on a bounded wait records that in
 * the device error word; tg_gemm_check reports it.
 *
 * Thread safety: calls from several host threads are safe.
 */
tg_status tg_gemm(int64_t M, int64_t N, int64_t K,
                  const void* A, int64_t lda,
                  const void* B, int64_t ldb,
                  void* C, int64_t ldc,
                  tg_dtype in_dtype, tg_dtype out_dtype,
                  tg_stream_t stream);

/*
 * tg_gemm_batched -- C_b = A_b x B_b for b = 0 .. batch-1, a strided batch of
 * independent products in one launch.
 *
 * Source: the pages' GEMM (as for tg_gemm) has no batch; a batch is the
 * independent-problem form of the same operation, each product exactly the
 * one tg_gemm computes.  The matrices of one call share M, N, K, the row
 * strides and the dtypes.
 *
 * Arguments are those of tg_gemm plus
 *   batch    number of products, 0 .. 65535 (0 is a no-op).
 *   strideA  elements from A_b to A_(b+1): A_b = A + b*strideA.  0 uses one
 *            A for every b (broadcast).  Likewise strideB.
 *   strideC  elements from C_b to C_(b+1); with batch > 1 the C matrices
 *            must not overlap: strideC >= (M-1)*ldc + N.
 *
 * Semantics per product: those of tg_gemm (overwrite, fp32 accumulation,
 * RNE output rounding; K == 0 writes zeros).  Strides are in elements and
 * must be >= 0.  Operand strides that are multiples of 16 bytes and at least
 * one whole matrix (or 0) run on the TMA kernels, which walk every tile of
 * every product in one persistent launch; other strides (overlapping
 * operand matrices, odd strides) run on the predicated-load kernel.  The
 * path is chosen as for tg_gemm, counting the tiles of all products.
 *
 * Errors: those of tg_gemm, with the byte spans taken over the whole batch
 * (C's span, from C_0 to the end of C_(batch-1), may overlap neither A's nor
 * B's), plus TG_ERR_INVALID_ARG for a negative batch or stride or for
 * overlapping C matrices, and TG_ERR_UNSUPPORTED for batch > 65535 or more
 * than 2^31 tiles of 128 x 64 in the whole batch.  Ownership, asynchrony
 * and thread safety are as for tg_gemm.
 */
tg_status tg_gemm_batched(int64_t batch, int64_t M, int64_t N, int64_t K,
                          const void* A, int64_t lda, int64_t strideA,
                          const void* B, int64_t ldb, int64_t strideB,
                          void* C, int64_t ldc, int64_t strideC,
                          tg_dtype in_dtype, tg_dtype out_dtype,
                          tg_stream_t stream);

/* Activation of the fused epilogue (tg_gemm_ex). */
typedef enum {
    TG_ACT_NONE = 0, /* identity */
    TG_ACT_RELU = 1, /* max(x, 0) */
    TG_ACT_GELU = 2  /* x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)), Phi the
                        standard normal distribution function (exact form,
                        not the tanh approximation) */
} tg_activation;

/*
 * tg_gemm_ex -- C = act(alpha * (A x B) + beta * D + bias), a GEMM with a
 * fused epilogue.
 *
 * Source: "企业官网建设流程全解析" (cf-1.com, a TileLang article), §6.2, names
 * multi-operator fusion -- merging several operators into one kernel to save
 * launches and memory round trips -- as the next direction after the GEMM
 * kernel of its §3.3.  The pages give no formula, so the terms are the usual
 * GEMM epilogue ones with their textbook definitions.
 *
 * Arguments M..out_dtype and stream are those of tg_gemm; in addition
 *   alpha  scale of the product (fp32).
 *   beta   scale of D (fp32).  D is read only when beta != 0.
 *   D      device pointer, M rows of N elements of out_dtype, row i at
 *          D + i*ldd.  May be C itself (D == C and ldd == ldc: an in-place
 *          C = alpha*AB + beta*C); may be NULL when beta == 0.
 *   ldd    row stride of D in elements, ldd >= N when beta != 0.
 *   bias   device pointer to N fp32 values added to every row (bias[j] to
 *          column j), or NULL for none.
 *   act    TG_ACT_NONE, TG_ACT_RELU or TG_ACT_GELU, applied last.
 *
 * Semantics: for every output element, y = alpha * acc + bias[j] + beta *
 * D[i,j] in fp32, with acc the fp32-accumulated product; then act(y) is
 * rounded to out_dtype (to nearest even for fp16).  A and B are read even
 * when alpha == 0.  With alpha == 1, beta == 0, bias NULL and TG_ACT_NONE
 * the call is tg_gemm, bit for bit.  K == 0 gives C = act(beta*D + bias).
 * The epilogue runs in the same kernel as the product, on the accumulator
 * before the output conversion, in every path (see tg_gemm_path: the path
 * does not depend on the epilogue).
 *
 * Errors: those of tg_gemm, plus TG_ERR_INVALID_ARG for an act outside the
 * enum; beta != 0 with D NULL, ldd < N, or D not a multiple of its element
 * size; D overlapping C other than exactly in place; bias not 4-byte
 * aligned or overlapping C.  Ownership, asynchrony and thread safety are as
 * for tg_gemm; the library keeps no pointer after the call returns.
 */
tg_status tg_gemm_ex(int64_t M, int64_t N, int64_t K,
                     const void* A, int64_t lda,
                     const void* B, int64_t ldb,
                     void* C, int64_t ldc,
                     tg_dtype in_dtype, tg_dtype out_dtype,
                     float alpha, float beta,
                     const void* D, int64_t ldd,
                     const float* bias, tg_activation act,
                     tg_stream_t stream);

/*
 * tg_attention -- attention forward, O_b = softmax(scale * Q_b K_b^T) V_b for
 * b = 0 .. batch-1 (heads or sequences of a strided batch), row by row.
 *
 * Source: "TileLang实战：用Python DSL自动生成高性能GPU计算内核" (gsyq.cn), §4
 * (FlashAttention): the product softmax(Q K^T) V of §4.1, computed by §4.2
 * blockwise over the keys with a running maximum M and normaliser L per query
 * row, so the Nq x Nk score matrix never exists in memory.  The page applies
 * no 1/sqrt(d) factor: pass scale = 1 for its kernel (the usual 1/sqrt(d) for
 * transformer attention); any finite scale is accepted.  Full (non-causal)
 * attention, as on the page.
 *
 * Arguments (sizes >= 0; row strides and matrix strides in elements):
 *   Q  batch x Nq x d,  row i of matrix b at Q + b*strideQ + i*ldq.
 *   K  batch x Nk x d,  likewise with ldk, strideK.
 *   V  batch x Nk x dv, likewise with ldv, strideV.
 *   O  batch x Nq x dv, written; row i of matrix b at O + b*strideO + i*ldo.
 *   A stride of 0 uses one matrix for every b (e.g. keys shared by all
 *   heads); with batch > 1 the O matrices must not overlap.
 *   in_dtype  TG_F16 (Q, K and V); out_dtype TG_F16 or TG_F32.
 *
 * Semantics: s_ij = scale * sum_d Q_id K_jd with fp16 products accumulated in
 * fp32 on the tensor cores; probabilities 2^(s_ij log2(e) - m_i) rounded to
 * fp16 for the P V product, accumulated in fp32; O = (P V) / L rounded to
 * out_dtype.  Elements of O between column dv and ldo are never written.
 *
 * Errors (checked on the host before anything is enqueued):
 *   TG_ERR_INVALID_ARG  a negative size or stride; Nk == 0 or d == 0 (no
 *                       softmax to take) with work to do; a NULL pointer;
 *                       ld < row length; O not aligned to its element size;
 *                       overlapping O matrices; O overlapping Q, K or V.
 *   TG_ERR_UNSUPPORTED  other dtypes; Q, K or V not 16-byte aligned, a row
 *                       stride not a multiple of 8, or a nonzero matrix
 *                       stride that is not a multiple of 8 or smaller than a
 *                       whole matrix (the TMA engine reads them); batch >
 *                       65535, dv > 65535 * 128, or a size above 2^31 - 1024.
 * batch, Nq or dv == 0 is a no-op.  Ownership, asynchrony, the device error
 * word and the test hook are as for tg_gemm.
 */
tg_status tg_attention(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                       const void* Q, int64_t ldq, int64_t strideQ,
                       const void* K, int64_t ldk, int64_t strideK,
                       const void* V, int64_t ldv, int64_t strideV,
                       void* O, int64_t ldo, int64_t strideO,
                       float scale, tg_dtype in_dtype, tg_dtype out_dtype,
                       tg_stream_t stream);

/*
 * tg_attention_ws -- tg_attention with a caller-provided workspace.
 *
 * When the work of a call covers fewer CTAs than the GPU has SMs (few heads,
 * short sequences, or the page's single 1024 x 768 head), the keys are split
 * into ranges handled by separate CTAs, each writing an unnormalised partial
 * output with its running maximum and normaliser to `workspace`; a second
 * kernel merges them (the same merge of maxima and normalisers the blockwise
 * pass applies between key blocks).  For heads with d <= 128 and dv <= 128
 * the workspace serves a second purpose: when the query tiles fill the SMs
 * more than once and leave the last wave at most 45 % full, each tile of
 * that wave is cut into 2 or 4 ranges of at least four key blocks, run by
 * separate CTAs, and the range that finishes last merges all partial
 * results (the same merge, in the order of the ranges, so that the result
 * does not depend on which one merges) in the kernel; the workspace holds
 * the partials and one counter per tile, zeroed by a small kernel the call
 * launches first.  tg_attention_workspace_size reports the bytes either use
 * on the current device (0 when neither applies).  A NULL or smaller
 * workspace runs the single pass: the result is the same up to rounding
 * order.
 *
 * Arguments: those of tg_attention, plus
 *   workspace        device memory, 256-byte aligned, owned by the caller,
 *                    not overlapping Q, K, V or O; its contents on entry do
 *                    not matter and are undefined afterwards.
 *   workspace_bytes  its size.
 * Calls that share a workspace must not overlap in time (use one stream, or
 * one workspace per stream).  Errors: those of tg_attention, plus
 * TG_ERR_INVALID_ARG for a misaligned or overlapping workspace.
 */
tg_status tg_attention_ws(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                          const void* Q, int64_t ldq, int64_t strideQ,
                          const void* K, int64_t ldk, int64_t strideK,
                          const void* V, int64_t ldv, int64_t strideV,
                          void* O, int64_t ldo, int64_t strideO,
                          float scale, tg_dtype in_dtype, tg_dtype out_dtype,
                          void* workspace, size_t workspace_bytes,
                          tg_stream_t stream);

/* Workspace bytes tg_attention_ws uses for these sizes on the current device
 * (0: no key split and no split of the last wave, or invalid sizes, or no
 * device). */
size_t tg_attention_workspace_size(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv);

/*
 * tg_attention_noalloc -- tg_attention_ws with the partial results of its
 * splits (the key split, and the split of a short last wave) in the
 * library's own file-scope device scratch instead of a caller workspace.
 * The pages have no counterpart of this entry point: it exists for callers
 * that cannot allocate device memory at call time (code running under a
 * memory pool or allocator they do not own, or inside a region where an
 * allocation would synchronise the device).
 *
 * Arguments, semantics and errors are those of tg_attention, plus:
 *   - the scratch is a fixed 16 MB static device array, held by every GPU
 *     that loads the library until the process exits; a call whose key
 *     split needs more returns TG_ERR_UNSUPPORTED
 *     (tg_attention_workspace_size tells the need), a call whose split of
 *     the last wave would need more runs without it, and a call that needs
 *     no split runs the single pass;
 *   - the first call on a device looks up the scratch's device address
 *     (cudaGetSymbolAddress, with that device current); make that first
 *     call before any stream capture on the device;
 *   - the key split writes every partial before the combine kernel reads
 *     it, and the last-wave split's per-tile counters are zeroed by a small
 *     kernel in every call, so nothing left in the scratch by an earlier
 *     call is read;
 *   - no device memory is allocated or freed, ever;
 *   - all calls on a device share the scratch, so calls that overlap in time
 *     (on different streams, or from different host threads without
 *     ordering) race on it and give undefined results.  Serialise them, or
 *     use tg_attention_ws with one workspace per stream.
 *   - tg_attention_force_kernel is read once per call.
 */
tg_status tg_attention_noalloc(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                               const void* Q, int64_t ldq, int64_t strideQ,
                               const void* K, int64_t ldk, int64_t strideK,
                               const void* V, int64_t ldv, int64_t strideV,
                               void* O, int64_t ldo, int64_t strideO,
                               float scale, tg_dtype in_dtype, tg_dtype out_dtype,
                               tg_stream_t stream);

/*
 * tg_gemm_check -- synchronize `stream`, then read and clear the current
 * device's error word.  Returns TG_OK, TG_ERR_CUDA if the stream reported a
 * CUDA error, or TG_ERR_TIMEOUT if a kernel abandoned a bounded wait (its
 * output is then undefined).
 */
tg_status tg_gemm_check(tg_stream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* tg_status_string(tg_status status);

/*
 * Path selection, for tests and benchmarks.  tg_gemm_path reports, without
 * launching anything, which kernel tg_gemm would run for these arguments on
 * the current device:
 *   0 none (no-op or error), 1 zero-fill (K == 0), 2 SIMT fp32,
 *   3 TMA + tcgen05 main kernel (one CTA per 128-row tile),
 *   4 boundary kernel (predicated loads, any alignment),
 *   5 skinny kernel (small M, split-K across a thread-block cluster),
 *   6 TMA + tcgen05 main kernel on CTA pairs (256 x 256 tiles).
 * tg_gemm_force_path forces one of 2..6 for subsequent calls in this process
 * (0 restores automatic selection); a forced path that cannot serve a call
 * (e.g. the main kernel for misaligned operands, SIMT for fp16) makes that
 * call return TG_ERR_UNSUPPORTED.
 */
int tg_gemm_path(int64_t M, int64_t N, int64_t K,
                 const void* A, int64_t lda,
                 const void* B, int64_t ldb,
                 void* C, int64_t ldc,
                 tg_dtype in_dtype, tg_dtype out_dtype);
/* The path tg_gemm_batched would take for these arguments (same codes). */
int tg_gemm_batched_path(int64_t batch, int64_t M, int64_t N, int64_t K,
                         const void* A, int64_t lda, int64_t strideA,
                         const void* B, int64_t ldb, int64_t strideB,
                         void* C, int64_t ldc, int64_t strideC,
                         tg_dtype in_dtype, tg_dtype out_dtype);
void tg_gemm_force_path(int path);

/*
 * Test hook for failure detection, off (0) by default.  With hook 1, every
 * subsequent tensor-core launch leaves one pipeline stage unfilled (or, in
 * the boundary kernel, one MMA group uncommitted): nothing ever signals the
 * barrier that the kernel then waits on, so its bounded wait runs out after
 * about a second, the kernel records the expiry in the device error word,
 * releases what it holds and returns, and tg_gemm_check reports
 * TG_ERR_TIMEOUT.  C is undefined for those calls.  Nothing faults, traps
 * or hangs.  Any other value turns the hook off.  Process-wide, not
 * thread-specific; the SIMT fp32 path has no waits and ignores it.
 */
void tg_gemm_test_hook(int hook);

/*
 * Tiling override, for configuration sweeps, tests and benchmarks (the
 * pages' tuning harness: block sizes and rasterisation, screened per shape).
 *   bn       tile width of the one-CTA kernel (path 3): 64, 128 or 256
 *            (with 4, 3 or 4 pipeline stages of k-blocks of 128, 128 or 64
 *            fp16 elements); 0 = chosen per problem.
 *   group_m  height, in tile rows, of the grouped tile order of the one-CTA
 *            and pair kernels (1..64); 0 = each kernel's default (16 for
 *            128-row tiles, 8 for 256-row pair tiles).
 * Process-wide; stays in force until changed.  Returns TG_ERR_INVALID_ARG
 * (and changes nothing) for any other value.
 */
tg_status tg_gemm_force_tiling(int bn, int group_m);

/*
 * Pipeline-depth override, for configuration sweeps (the pages' num_stages,
 * tuned separately from the tile size): the number of shared-memory stages
 * in the TMA load ring of the one-CTA kernel (path 3; at most 4, 3 or 4 for
 * tiles 256, 128 or 64 wide, the default: stages of 48, 64 or 48 KB) and of
 * the CTA-pair kernel (path 6; at most 3, the default).
 *   stages  0: each kernel's default; 2..8: that many stages.
 * Process-wide; stays in force until changed.  Returns TG_ERR_INVALID_ARG
 * (and changes nothing) for other values.  A later call whose kernel holds
 * fewer stages returns TG_ERR_UNSUPPORTED; other paths ignore it.
 */
tg_status tg_gemm_force_stages(int stages);

/*
 * Split over K of the one-CTA kernel (path 3), for tests and benchmarks.  A
 * call whose 128 x BN output tiles (all products of a call together) leave
 * at least half of the SMs idle can share each tile over K among a cluster
 * of S CTAs: each CTA computes an fp32 partial over its range of k-blocks
 * (128 fp16 or 256 E4M3 elements each for tiles 64 or 128 wide, 64 or 128
 * for tiles 256 wide) and the cluster adds the S partials
 * in distributed shared memory, in rank order, before the epilogue.
 *   split  0: automatic (tg_gemm_main_plan's choice, with every cluster
 *          resident at once); 1: never; 2, 4 or 8: always that many CTAs
 *          per tile (halved while it exceeds the k-blocks), at the default
 *          or forced tile width.
 * Process-wide; stays in force until changed.  Returns TG_ERR_INVALID_ARG
 * (and changes nothing) for any other value.  Results can differ in the
 * last bits between splits (another order of fp32 additions) and are exact
 * for inputs whose partial sums are.
 */
tg_status tg_gemm_force_split_k(int split);

/*
 * The one-CTA kernel's automatic choice, computed on the host alone for an
 * M x N x K call (batch products) of in_dtype (TG_F16 or TG_E4M3) on
 * num_sms SMs: returns the split S (1: none) and writes the tile width
 * (64, 128 or 256) to *bn.  The default width (256 when 256-column tiles
 * fill the SMs, else 128 when 128-column tiles fill half of them, else 64;
 * never wider than N rounded up to 64 or 128), unsplit, competes with every
 * other width unsplit and with every width whose tiles fill at most half of
 * the SMs at its largest split (2, 4 or 8 with tiles * S <= num_sms and
 * S <= k-blocks), by a time estimate (waves of CTAs included; a challenger
 * must be 5 % faster) measured on GB300: a CTA's A and B bytes (its k-range
 * counted up to K) taken in at ~100 KB/us unsplit and ~110 KB/us split for
 * 64- and 128-column tiles (~86 and ~95 for 256 columns), plus 1.5, 2.5 or
 * 4.0 us for a split of 64-, 128- or 256-column tiles.  On a device the
 * library also requires every cluster to be resident at once (GB300 holds
 * 15 clusters of 8 of these CTAs), which can change the choice.
 * Returns 0 (and *bn = 0) for non-positive sizes or another dtype.
 */
int tg_gemm_main_plan(int64_t M, int64_t N, int64_t K, int64_t batch, tg_dtype in_dtype,
                      int num_sms, int* bn);

/*
 * Last-wave override of the CTA-pair kernel (path 6), for tests and
 * benchmarks.  The pair kernel hands its 256 x 256 tiles to the CTA pairs
 * in waves; when the last wave is at most half full, it cuts each of that
 * wave's tiles into two 256 x 128 halves so that twice as many pairs share
 * it (fp16 inputs; E4M3 calls never cut).
 *   tiles  -1: automatic (the rule above); 0: never cut; k > 0: cut the
 *          last k tiles of every call (capped at the call's tile count),
 *          whatever the wave shape.
 * Process-wide; stays in force until changed.  Returns TG_ERR_INVALID_ARG
 * (and changes nothing) for tiles < -1.  Results are the same either way.
 */
tg_status tg_gemm_force_split_tail(int tiles);

/*
 * The automatic rule above, computed on the host alone (no device needed):
 * how many of `tiles` 256 x 256 tiles (all products of a call together) the
 * pair kernel cuts in two on a GPU that holds `max_pairs` CTA pairs at once
 * (half the SM count when the kernel fills every SM).  The last wave holds
 * last = tiles - max_pairs * floor((tiles - 1) / max_pairs) tiles; they are
 * all cut when 2 * last <= max_pairs, else none.  0 for non-positive
 * arguments.
 */
int tg_gemm_pair_split_tail(int64_t tiles, int max_pairs);

/*
 * The boundary kernel's split over K (the kernel that serves operands the TMA
 * engine cannot address), computed on the host alone: a problem with `tiles`
 * 128 x 128 output tiles (all products of a call together) and `kblocks`
 * k-blocks of 64 is shared by clusters of S CTAs, S the largest of 2, 4 and 8
 * with tiles * S <= num_sms and S <= kblocks, else 1.  On a device the
 * library also requires that `tiles` clusters of S fit at once.  1 for
 * non-positive arguments.
 */
int tg_gemm_boundary_split(int64_t tiles, int kblocks, int num_sms);

/*
 * Attention kernel selection, for tests and benchmarks.  tg_attention_kernel
 * reports, without launching anything, which forward kernel a call with these
 * sizes would run on the current device: tg_attention (split_allowed = 0),
 * or tg_attention_ws / tg_attention_noalloc given the workspace that
 * tg_attention_workspace_size asks for (split_allowed = 1):
 *   0 none (sizes out of range or empty; tg_attention reports the error),
 *   1 the general kernel (any d and dv; P staged in shared memory),
 *   2 the same with the keys split over several CTAs and a combine kernel
 *     (calls with few query tiles, given the workspace),
 *   3 the kernel that keeps P in tensor memory, with two score buffers
 *     (heads with d <= 128 and dv <= 128).
 * tg_attention_force_kernel(1) keeps later calls off kernel 3;
 * tg_attention_force_kernel(3) runs kernel 3, with no key split, for every
 * later call whose head sizes it serves (others choose automatically); 0
 * restores automatic selection.  Process-wide.  Returns TG_ERR_INVALID_ARG
 * (and changes nothing) for any other value.
 */
int tg_attention_kernel(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                        int split_allowed);
tg_status tg_attention_force_kernel(int kernel);

/*
 * tg_attention_tail_plan -- the split of a short last wave (tg_attention_ws)
 * that kernel 3 would make for these sizes on a GPU with `num_sms` SMs,
 * computed on the host alone (no device needed).  The kernel gives each CTA
 * 128 query rows of one head; tiles = ceil(Nq / 128) * batch go to the SMs in
 * waves of num_sms.  When there are more tiles than SMs and the last wave
 * holds at most 45 % of num_sms tiles, each of its tiles is cut into 2 ranges
 * of key blocks (4 when it holds at most 20 %), fewer if that would leave a
 * range under four blocks of 128 keys, and none below two ranges.
 * Returns the number of tiles cut (0: no split; also for sizes kernel 3 does
 * not serve, d or dv above 128, or out of range) and stores the ranges per
 * tile in *pieces (0 with no split); `pieces` may be NULL.
 */
int tg_attention_tail_plan(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                           int num_sms, int* pieces);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int tg_gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TG_GEMM_H */
