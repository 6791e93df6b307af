/*
 * bqgemv.h -- block-quantized weight dequant + batch-1 GEMV for GB300 (sm_103a).
 *
 * The C ABI of libbqgemv.so.  Plain C: pointers, sizes and an opaque stream
 * handle; no CUDA or PyTorch types.
 *
 * What is computed (sources are the four pages this library restates):
 *  - The batch-1 decode step of a quantized LLM is a bandwidth-bound
 *    matrix-vector product over quantized weights, dequantized on the fly
 *    inside the dot product with no fp32 weight buffer ("We Wrote Our Own
 *    Inference Engine", "What actually moved it" #2; EdgeRunner blog post,
 *    "What worked" #2; RunIT README, optimisation table "Fused Q8_0 GEMV" /
 *    "Fused Q4_0 GEMV").
 *  - Block formats (GGUF-style, 32 weights per block; the RunIT README's
 *    "Quantization" table gives 1.06 B/elem for Q8_0 and 0.56 B/elem for Q4_0):
 *      Q8_0, 34 bytes: fp16 scale d (little-endian) then 32 int8 codes q;
 *            w = d * q.
 *      Q4_0, 18 bytes: fp16 scale d then 16 bytes qs; element j < 16 is the
 *            low nibble of qs[j], element j + 16 the high nibble; w = d*(n-8).
 *      Q4_K, 144 bytes per 256 weights (a super-block; the RunIT README's
 *            kernel table names gemv_q4k_f16 and its "Quantization" table
 *            Q4_K_M; the layout is read from the public GGUF definition):
 *            fp16 d, fp16 dmin, 12 bytes of eight 6-bit sub-block scales
 *            sc[j] and mins m[j] (j < 4: sc = s[j] & 63, m = s[j+4] & 63;
 *            j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4,
 *            m = (s[j+4] >> 4) | (s[j] >> 6) << 4), then 128 bytes qs where
 *            element i of sub-block 2g is the low nibble of qs[32g+i] and
 *            element i of sub-block 2g+1 its high nibble;
 *            w = d*sc[j]*q - dmin*m[j] for sub-block j (32 weights).
 *  - A packed matrix with M rows and K columns is M rows of K/32 blocks (Q4_K:
 *    K/256 super-blocks), rows contiguous with no padding: row m starts at
 *    byte m * (K/32) * {34, 18, 18} (Q8_0, Q4_0, Q4_K).
 *
 * Conventions for every call below:
 *  - All data pointers are DEVICE pointers (cudaMalloc / PyTorch CUDA memory)
 *    owned by the caller; the library allocates nothing and keeps no state
 *    except a per-device record of kernel attributes it has set.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Every call only enqueues work and returns; results are ready
 *    when the stream reaches that point.
 *  - Back-to-back GEMV calls on one stream overlap: a call may start while
 *    the GEMV call before it (of this library) drains, and copy its packed
 *    weights into shared memory then; it reads its inputs and writes its
 *    outputs only after that call has completed.  So the packed weights of a
 *    call must not be written by an earlier GEMV call of this library on the
 *    stream (those calls write only their outputs: the one thing excluded is
 *    an output buffer reused as a later call's packed weights).  Any other
 *    work before a call, bq_quantize_pack and foreign kernels included,
 *    completes before the call starts.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns an error status and enqueues nothing.  Launch failures
 *    return BQ_ERR_CUDA.  Faults inside a kernel surface at the caller's next
 *    synchronisation, as with any CUDA library.  No call aborts or throws.
 *  - Outputs are overwritten, never accumulated into.  Inputs and outputs
 *    must not overlap.
 *  - Shapes: 0 <= M <= 2^31 - 1, K a multiple of 32 (of 256 for Q4_K),
 *    32 <= K <= 2^18.
 *    M == 0 is an empty product: after the qtype and shape checks the call
 *    returns BQ_OK without reading or writing anything, so its pointers may
 *    be NULL (an empty PyTorch tensor has a NULL data pointer).  The fast
 *    streaming kernels need K % 256 == 0 (whole 8-block units per row); other
 *    multiples of 32 take a slower kernel with the same results.
 *  - Alignment: packed weights and fp32 vectors/matrices 16-byte aligned;
 *    fp32 outputs 4-byte aligned.
 *  - Determinism: every output element is computed in a fixed order that
 *    depends only on (qtype, K).  The same call on the same inputs gives the
 *    same bits on every run, and bq_gemv_verify row r is bit-identical to the
 *    single-row GEMV on X[r].
 */
#ifndef BQGEMV_H
#define BQGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BQ_OK = 0,
    BQ_ERR_NULL = 1,   /* a required pointer is NULL */
    BQ_ERR_SHAPE = 2,  /* M, K or R outside the documented range */
    BQ_ERR_ALIGN = 3,  /* a pointer is not aligned as documented */
    BQ_ERR_QTYPE = 4,  /* unknown quantization type */
    BQ_ERR_CUDA = 5,   /* a CUDA runtime call or kernel launch failed */
    BQ_ERR_DEVICE = 6  /* a kernel recorded a device-side error (see bq_device_status) */
} bq_status;

typedef enum { BQ_Q4_0 = 2, BQ_Q8_0 = 8, BQ_Q4_K = 12 } bq_qtype;

/* Largest R accepted by bq_gemv_verify (the multi-row verify pass of
 * speculative decoding runs 3-6 rows; "We Wrote Our Own Inference Engine",
 * Update). */
#define BQ_VERIFY_MAX_ROWS 6

/* Library version, major*10000 + minor*100 + patch. */
int bq_version(void);

/* Human-readable text for a bq_status value (never NULL). */
const char *bq_status_str(int status);

/* Bytes of a packed M x K matrix: M * (K/32) * {34 for Q8_0, 18 for Q4_0 and
 * Q4_K}.  Returns -1 for an unknown qtype, a negative size or K not a multiple
 * of 32 (of 256 for Q4_K).  (RunIT README, "Quantization" table: 1.06 / 0.56
 * bytes per element.) */
int64_t bq_packed_bytes(int qtype, int64_t M, int64_t K);

/* Quantize fp32 weights W [M, K] (row-major) into packed blocks Wq
 * (bq_packed_bytes(qtype, M, K) bytes).  Per block of 32 weights:
 *   Q8_0: d = fp16_rne(max|w| / 127);  q = clamp(round(w / d), -127, 127)
 *   Q4_0: d = fp16_rne(max|w| / 8);    n = clamp(round(w / d) + 8, 0, 15)
 * with fp32 IEEE divisions by the stored scale, round = half away from zero,
 * and d == 0 giving q = 0 / n = 8.  Q4_K, per super-block of 256 weights and
 * per sub-block j of 32: lo = min(0, min w), scale_j = (max w - lo) / 15,
 * min_j = -lo; d = fp16_rne(max scale_j / 63), dmin = fp16_rne(max min_j / 63);
 * sc_j = clamp(round(scale_j / d), 0, 63), m_j = clamp(round(min_j / dmin),
 * 0, 63); q = clamp(round((w + dmin*m_j) / (d*sc_j)), 0, 15) (0 where a
 * divisor is 0) -- the plainest quantizer that fills the GGUF layout (the
 * pages give none).  The output bytes are a pure function of the input bits.  This is the load-time conversion the pages do in their
 * converters ("We Wrote Our Own Inference Engine", "The recipe rule"), not
 * part of the per-token path.
 * W: 4-byte aligned; Wq: 16-byte aligned.  NaN/Inf weights are outside the
 * contract. */
bq_status bq_quantize_pack(int qtype, const float *W, int64_t M, int64_t K, void *Wq,
                           void *stream);

/* y[m] = sum_k w[m,k] * x[k] for packed Q8_0 weights Wq (M x K), fp32 x[K],
 * fp32 y[M]; dequantized on the fly, fp32 accumulation in a fixed order.
 * (RunIT README kernel table, gemv_q8_0_f32in_f32out; EdgeRunner blog post,
 * "What worked" #2.) */
bq_status bq_gemv_q8_0(const void *Wq, const float *x, float *y, int64_t M, int64_t K,
                       void *stream);

/* The same for packed Q4_0 weights.  (RunIT README kernel table,
 * gemv_q4_0_f32in_f32out; "We Wrote Our Own Inference Engine", "What actually
 * moved it" #2, the dedicated 4-bit GEMV.) */
bq_status bq_gemv_q4_0(const void *Wq, const float *x, float *y, int64_t M, int64_t K,
                       void *stream);

/* The same for packed Q4_K super-blocks (K % 256 == 0).  Per super-block the
 * fixed tree is: sub-block sums s_j = sum q*x (q = 0..15) in the order of the
 * 32-weight blocks of Q8_0/Q4_0, cq = sum_j (d*sc_j)*s_j and cm = sum_j
 * (dmin*m_j)*X_j in sub-block order (X_j the sum of the sub-block's x in a
 * fixed order), unit = cq - cm.  |y - exact| <= 1e-5 * SK with SK = sum over
 * sub-blocks of d*sc_j*sum|q x| + dmin*m_j*sum|x| (>= sum |w x|).  (RunIT
 * README kernel table, gemv_q4k_f16 / "gemv_q4k.metal"; "Quantization"
 * table, Q4_K_M.)  bq_gemv_gate_up_silu, bq_gemv_qkv_bias, bq_gemv_verify,
 * the stream plans and bq_stream_run_noalloc take BQ_Q4_K as well. */
bq_status bq_gemv_q4_k(const void *Wq, const float *x, float *y, int64_t M, int64_t K,
                       void *stream);

/* Fused feed-forward input stage:
 *   xn = gamma == NULL ? x : x * gamma / sqrt(mean(x^2) + eps)
 *   y[m] = silu(g[m]) * u[m],  g = Wg xn,  u = Wu xn,  silu(z) = z / (1 + e^-z)
 * Wg and Wu are packed M x K matrices of the same qtype; x, gamma: fp32[K];
 * y: fp32[M].  eps must be finite and >= 0 (with gamma != NULL).
 * (RunIT README kernel table, fused_ffn_q4_0_f32 "gate+up+silu fused" and
 * rms_norm_f32_f32_f32g; EdgeRunner blog post, "The progression", the
 * RMSNorm+GEMV fusion stage.) */
bq_status bq_gemv_gate_up_silu(int qtype, const void *Wg, const void *Wu, const float *x,
                               const float *gamma, float eps, float *y, int64_t M, int64_t K,
                               void *stream);

/* Fused q|k|v projection with bias: y[m] = sum_k w[m,k] * x[k] + bias[m] for
 * packed weights Wqkv (M x K) whose rows are the q, k and v projections
 * concatenated at load time (packed rows concatenate as they are: a packed
 * matrix is its rows, back to back), fp32 x[K], bias fp32[M] (the q, k and v
 * biases concatenated the same way) or NULL, fp32 y[M].  The dot product is
 * the single-row GEMV's, bit for bit; the bias is one fp32 add after it.
 * (RunIT README kernel table, fused_qkv_bias_q8_0_f32 "Q+K+V+bias in ONE
 * dispatch", and optimisation table "Fused QKV+bias": 6 dispatches -> 1 per
 * layer on the Qwen path.)  bias: 4-byte aligned. */
bq_status bq_gemv_qkv_bias(int qtype, const void *Wqkv, const float *x, const float *bias, float *y,
                           int64_t M, int64_t K, void *stream);

/* The unquantized fp16-weight GEMV: y[m] = sum_k w[m,k] * x[k] for W fp16
 * [M, K] row-major (IEEE binary16, little-endian), fp32 x[K], fp32 y[M]; each
 * product and sum in fp32 on a fixed tree that depends on K alone (runs are
 * bit-reproducible), within 1e-5 * sum_k |w x| of the exact value.  ("We
 * Wrote Our Own Inference Engine", "What actually moved it" #4: the GEMV for
 * the unquantized fp16 matrices; RunIT README kernel table,
 * gemv_f16w_f32in_f32out.)  Preconditions: 8 <= K <= 2^18 and K % 8 == 0,
 * M >= 0 (M = 0 does nothing), W and x 16-byte aligned, y 4-byte aligned, y
 * not overlapping W or x. */
bq_status bq_gemv_f16(const void *W, const float *x, float *y, int64_t M, int64_t K, void *stream);

/* bq_gemv_f16 with an fp16 output: y[m] is bq_gemv_f16's fp32 y[m] rounded
 * to the nearest binary16 value, ties to even (beyond +-65504 it rounds to
 * +-inf).  ("We Wrote Our Own Inference Engine", "What actually moved it" #5:
 * fp16-output GEMVs.)  y: fp16 [M], 2-byte aligned; otherwise the arguments,
 * preconditions and errors of bq_gemv_f16.  Both calls split K across the
 * warps of a CTA when M is small; the summation tree, and so every bit of y,
 * does not depend on that choice. */
bq_status bq_gemv_f16_f16out(const void *W, const float *x, void *y, int64_t M, int64_t K,
                             void *stream);

/* Multi-row verify GEMV: Y[r, m] = sum_k w[m,k] * X[r, k] for r < R,
 * 1 <= R <= BQ_VERIFY_MAX_ROWS, with the weights streamed once for all R rows.
 * X: fp32 [R, K] row-major; Y: fp32 [R, M] row-major.  Row r of Y is
 * bit-identical (memcmp-equal) to bq_gemv_q8_0 / bq_gemv_q4_0 on X[r].
 * ("We Wrote Our Own Inference Engine": the one-stream 3-6-row verify kernel
 * of the Update, and "Correctness first", verify checked against decode with
 * memcmp.) */
bq_status bq_gemv_verify(int qtype, const void *Wq, const float *X, float *Y, int R,
                         int64_t M, int64_t K, void *stream);

/* Device-side error word of the current device.  The kernels bound every
 * wait on their shared-memory pipeline; a wait that runs out sets a bit here
 * and the kernel returns early.  *flags receives the word (0 = no error);
 * clear != 0 resets it.  Synchronises the device.  Returns BQ_ERR_DEVICE if
 * the word is non-zero, else BQ_OK (or BQ_ERR_CUDA). */
bq_status bq_device_status(unsigned int *flags, int clear);

/* The fixed summation tree of a row: each row of K/256 units (8 blocks) is
 * split over bq_tree_lanes(K) lanes, lane l summing units l, l+G, l+2G, ...
 * in order, and the lane sums are folded pairwise.  Exposed so callers and
 * tests can reason about determinism; -1 if K is not a positive multiple of 32. */
int bq_tree_lanes(int64_t K);

/* ------------------------------------------------------------------------
 * Per-token stream plans.
 *
 * A decode step is a chain of dependent GEMV stages (per layer q|k|v, o,
 * gate+up, down, then the LM head).  The pages run it as one command buffer
 * per token because dispatch cost dominates small GEMVs (EdgeRunner blog
 * post, "What worked" #1; "We Wrote Our Own Inference Engine", 770 dispatches
 * per token).  A plan is that token's launch schedule, made once:
 *  - a list of independent ops (no op reads another's output) runs as ONE
 *    launch of the streaming kernel;
 *  - a list of dependent stages runs as one launch of the streaming kernel
 *    per stage, each allowed to start while the stage before drains
 *    (programmatic dependent launch): it fills its shared-memory weight ring
 *    first (the plan's stages write no weights), then waits for the stage
 *    before and reads its input, so an op may read an output written by an
 *    earlier stage.  Captured in a CUDA graph, the whole token is one graph
 *    launch: the command buffer of the pages.
 *  - the cooperative executor (one launch, grid-wide barriers between
 *    stages) runs a dependent list whose stages the streaming kernel cannot
 *    hold, and backs bq_stream_run_noalloc.
 * Every output is bit-identical to the single-op call (bq_gemv_q8_0 /
 * _q4_0 / _q4_k / bq_gemv_qkv_bias / bq_gemv_gate_up_silu) on the same
 * inputs, whichever way the plan runs.
 * ------------------------------------------------------------------------ */
typedef enum { BQ_OP_GEMV = 0, BQ_OP_GATE_UP_SILU = 1 } bq_op_kind;

typedef struct {
    int32_t kind;        /* bq_op_kind */
    int32_t stage;       /* 0 for the first op; then equal to, or one more than,
                            the previous op's stage */
    int64_t M, K;        /* M >= 1; K % 256 == 0, 256 <= K <= 2^18 */
    const void *W;       /* packed weights (the gate matrix for GATE_UP_SILU) */
    const void *W_up;    /* packed up matrix (GATE_UP_SILU), else ignored */
    const float *x;      /* fp32[K]; may be the output of an earlier stage */
    const float *gamma;  /* GATE_UP_SILU: RMSNorm gain fp32[K] or NULL */
    float eps;           /* GATE_UP_SILU with gamma: finite, >= 0 */
    float *y;            /* fp32[M]; must not overlap any input of its own stage */
    const float *bias;   /* GEMV: fp32[M] added to the output (the fused q|k|v + bias
                            op), or NULL; GATE_UP_SILU: must be NULL */
} bq_op;

typedef struct bq_stream_plan bq_stream_plan;

/* Device workspace a plan of n_ops ops in n_stages stages needs (descriptor
 * tables, per-stage CTA splits, barrier counters); -1 for bad counts.  Besides the
 * shape rules of bq_op, the distinct inputs of one stage (ops sharing an x and
 * its norm count once) must fit the executor's shared-memory x area together
 * with two ring slots per warp: about 150 KB of fp32 x per stage;
 * bq_stream_plan_create returns BQ_ERR_SHAPE otherwise. */
int64_t bq_stream_workspace_bytes(int n_ops, int n_stages);

/* Validate the ops (all of one qtype), plan their launch geometry and upload
 * the descriptor table into `workspace` (caller-owned device memory of at
 * least bq_stream_workspace_bytes bytes, 256-byte aligned, kept alive and
 * untouched until the plan is destroyed).  Synchronous (it copies host to
 * device): create plans before capturing a CUDA graph.  *plan is a small
 * host object owned by the caller until bq_stream_plan_destroy.  The device
 * that is current at creation runs the plan. */
bq_status bq_stream_plan_create(int qtype, const bq_op *ops, int n_ops, void *workspace,
                                int64_t workspace_bytes, bq_stream_plan **plan);

/* Enqueue one run of the plan on `stream`: one kernel launch (independent
 * ops), one per stage (dependent stages), or, for the executor, a memset of
 * its stage counters and one cooperative launch (bq_stream_plan_launches
 * says how many kernels); no host synchronisation, capturable in a CUDA
 * graph.  Two runs of one plan must not overlap on the GPU (an executor run
 * shares the counters, a staged run its stages' outputs). */
bq_status bq_stream_plan_launch(const bq_stream_plan *plan, void *stream);

/* Re-split a plan of independent ops (one launch of the streaming kernel)
 * among the GPU's CTAs by measured time, a set-up step.  (The pages have no
 * counterpart: they dispatch one kernel per GEMV.)  The planner first splits
 * the ops' tiles into one contiguous range per CTA of equal BYTES, but op
 * shapes stream at different rates per byte (idle lanes when K/256 is not a
 * multiple of the tree's lane count, per-tile folds, and the x staging at
 * every op boundary inside a range), so on GB300 the slowest CTA of a
 * Qwen3-0.6B-shaped Q8_0 token finished 12% after the median.  This call
 * runs the plan `rounds` + 1 times 3 launches each, with every CTA recording
 * its duration into the plan's workspace; after each measurement it charges
 * every tile its CTA's measured time per byte and re-splits for equal
 * estimated time.  The split whose slowest CTA was fastest is kept.  Only
 * the assignment of tiles to CTAs changes: every output row is computed by
 * the same arithmetic, so outputs are bit-identical before and after.
 *  - 1 <= rounds <= 16, else BQ_ERR_SHAPE; a plan of dependent stages
 *    returns BQ_OK untouched.
 *  - The runs read the ops' inputs and overwrite their outputs, on `stream`.
 *  - Synchronous (it reads the timings back): call it after
 *    bq_stream_plan_create and before capturing the plan in a CUDA graph. */
bq_status bq_stream_plan_tune(bq_stream_plan *plan, int rounds, void *stream);

/* Kernel launches one bq_stream_plan_launch enqueues: 1 for a list of
 * independent ops or a list run by the cooperative executor, the number of
 * stages for a staged plan; -1 for NULL. */
int bq_stream_plan_launches(const bq_stream_plan *plan);

/* Free the host object (the workspace stays the caller's). */
bq_status bq_stream_plan_destroy(bq_stream_plan *plan);

/* Allocation-free run of the stream executor.  (The pages have no
 * counterpart: this entry point exists for callers of this library, not for
 * the method.)
 *
 * Some callers cannot allocate device memory for the workspace above: a
 * serving process that has already handed all free HBM to its weight and
 * KV-cache pools, where a new cudaMalloc fails or fragments them; a host
 * framework that owns device memory through its own caching allocator and
 * forbids raw cudaMalloc beside it; or a latency-critical path that cannot
 * afford cudaMalloc/cudaFree, which can synchronise the device.  For them
 * this call runs the same ops as bq_stream_plan_create + bq_stream_plan_launch
 * (same validation, bit-identical outputs; a list of dependent stages runs
 * on the cooperative executor in one launch) with the descriptor
 * tables and stage counters kept in one fixed device array inside the
 * library, which every GPU that loads the library holds until the process
 * exits (82 KiB).  The caller still passes the inputs and outputs (in
 * the ops).  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *  - At most BQ_NOALLOC_MAX_OPS ops (and as many stages); more returns
 *    BQ_ERR_SHAPE without touching the device.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress), creates one CUDA event for that device (an
 *    event holds no device memory) and sets the kernel's shared-memory
 *    limit; make that first call before any stream capture.
 *  - Each call copies the tables from static host memory into the array on
 *    `stream` and clears the counters there, then launches.  All calls share
 *    the one array, which keeps the last call's contents: calls that overlap
 *    on the GPU (on different streams, or from different host threads
 *    without ordering) race on it and must be serialised by the caller.
 *    Host-side staging is serialised internally: a call first waits on the
 *    host until the previous call's table copies have run (they read the
 *    static host tables asynchronously), so back-to-back calls on one stream
 *    are safe but a call may block until the GPU reaches the previous one. */
#define BQ_NOALLOC_MAX_OPS 512
bq_status bq_stream_run_noalloc(int qtype, const bq_op *ops, int n_ops, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* BQGEMV_H */
