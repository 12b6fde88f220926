/*
 * flce.h -- C ABI of the GB300 (sm_103a) fused linear cross-entropy library.
 *
 * What the library computes. hidden is h[N,H], weight is W[V,H], bias is b[V]
 * (optional) and targets is t[N]. With s = logit_scale, c = softcap and
 * zeta = z_loss_multiplier:
 *
 *   a_ij = sum_k h_ik W_jk
 *   u_ij = (a_ij + b_j) * s
 *   z_ij = c * tanh(u_ij / c)   if c > 0, else u_ij
 *   lse_i = log sum_j exp z_ij
 *   loss_i = lse_i - z_{i,t_i} + zeta * lse_i^2   (valid rows, t_i != ignore_index)
 *   loss_i = 0                                    (ignored rows)
 *
 * Sources, by passage:
 * - The linear + cross-entropy definition: quack-kernels diff,
 *   quack/linear_cross_entropy.py, linear_cross_entropy_func_ref.
 * - bias, logit_scale, softcap and the metrics: fused-linear-ce README,
 *   sections "Full signature" and "Metrics for free".
 * - z-loss: "Chunked Linear Cross-Entropy", section "Usage". The page gives
 *   the keyword but not the formula; zeta * lse^2 is this library's reading.
 * - The global-mean semantics: "Chunked Linear Loss", section "Reduction
 *   semantics".
 *
 * The N x V logits are never stored.
 * - The forward sweeps vocabulary tiles and keeps an online log-sum-exp
 *   (fused-linear-ce README, "Algorithm").
 * - The backward recomputes each logit tile and forms dlogits from it in
 *   registers (same section). dlogits goes to HBM in 16 bits for one chunk
 *   at a time: a range of vocabulary columns for all rows when N < V, else
 *   a range of rows. Two tensor-core contractions then accumulate
 *   grad_hidden = dlogits W and grad_weight = dlogits^T h, as the quack diff
 *   and "Chunked Linear Loss", section "Gradient handling", do per chunk.
 *   grad_weight is computed transposed, (h^T dlogits)^T, so one row-major
 *   dlogits copy serves both contractions: half of the columns for all rows,
 *   or half of the rows for all columns. Only row chunks that add into
 *   existing gradients through the fp32 grad_weight partial also store each
 *   chunk transposed (two copies of a quarter of the rows). The copies hold
 *   about half of the N x V logits, and at most 4 GiB.
 *
 * Conventions common to every entry point:
 * - Pointers named "device" must point to device memory of the current CUDA
 *   device. All tensors are dense and row-major (the last index moves
 *   fastest) and 16-byte aligned, unless an entry point below states a
 *   smaller alignment for one of its arguments.
 * - The caller owns every buffer. The library allocates no device memory. It
 *   keeps only small per-device host state: attributes, tensor-map encoder,
 *   profiling events.
 * - Every call is asynchronous on `stream` and never synchronises the host,
 *   except flce_check_status and flce_profiling_read.
 * - Return codes are the FLCE_* values below. An argument error is reported
 *   before any work is enqueued. Errors the device detects (a target out of
 *   range, an expired bounded wait) are written to a status word at the start
 *   of the workspace. flce_check_status reads it.
 * - A forward whose bounded wait expired leaves no output that looks like a
 *   result: its loss, lse and entropy_sum are NaN and num_correct is -1 (the
 *   shard states of flce_forward_partial are NaN). A backward whose wait
 *   expired leaves its gradients undefined; only the status word tells.
 * - Outputs are overwritten, unless flce_params.accumulate asks the backward
 *   to add its gradients into the buffers it is given.
 * - Results do not depend on launch timing. Every reduction runs in a fixed
 *   order, so repeated calls on the same inputs give bit-identical outputs.
 * - The debug build of this library (libflce_debug.so, compiled with
 *   FLCE_DEBUG) checks every kernel store against the buffer it belongs to.
 *   A store that would land outside is skipped and flagged; each entry point
 *   then synchronises its stream and returns FLCE_ERR_BOUNDS. It is meant for
 *   tests, in place of a memory checker; the release build does no checks
 *   and never synchronises.
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. NULL is the legacy default stream. */
typedef struct CUstream_st* flce_stream_t;

typedef enum {
  FLCE_F32 = 0,  /* fp32 hidden/weight/bias/grads; SIMT fp32 arithmetic         */
  FLCE_BF16 = 1, /* bf16 hidden/weight/bias/grads; tcgen05 bf16 MMA, fp32 acc.  */
  FLCE_F16 = 2   /* fp16 hidden/weight/bias/grads; tcgen05 fp16 MMA, fp32 acc.
                    dlogits are stored in fp16 times an exact power of two that
                    keeps them out of the fp16 subnormal range                  */
} flce_dtype;

typedef enum { FLCE_SUM = 0, FLCE_MEAN = 1, FLCE_NONE = 2 } flce_reduction;

typedef enum {
  FLCE_PASS_FORWARD = 0,      /* flce_forward, flce_forward_partial, flce_forward_combine */
  FLCE_PASS_BACKWARD = 1,     /* flce_backward                                           */
  FLCE_PASS_CHUNK_LOGITS = 2, /* flce_chunk_logits (the status word only)                */
  FLCE_PASS_CHUNK_GRADS = 3,  /* flce_chunk_grads; N is the largest chunk's row count;
                                 the same workspace must be passed to every chunk of
                                 one loss, because it carries the fp32 grad_weight
                                 partial from chunk to chunk                            */
  FLCE_PASS_CHUNK_MSE = 4     /* flce_chunk_weighted_mse; N is the largest chunk's rows */
} flce_pass;

/* Position of a row chunk in flce_chunk_grads' accumulation of grad_weight. */
typedef enum {
  FLCE_CHUNK_ONLY = 0,  /* the loss has one chunk                                  */
  FLCE_CHUNK_FIRST = 1, /* first of several chunks                                 */
  FLCE_CHUNK_NEXT = 2,  /* neither first nor last                                  */
  FLCE_CHUNK_LAST = 3   /* last of several chunks: grad_weight is written here     */
} flce_chunk_phase;

/* Accumulator of grad_weight across row chunks ("Chunked Linear Loss",
 * section "Weight-gradient accumulation dtype"). FP32 keeps an fp32 partial
 * and casts once (the default). WEIGHT accumulates in the weight dtype, which
 * rounds between chunks but needs no fp32 [V,H] partial. */
typedef enum { FLCE_ACCUM_FP32 = 0, FLCE_ACCUM_WEIGHT = 1 } flce_accum;

/* Axis along which flce_backward cuts its work into chunks (see
 * flce_workspace_bytes). AUTO takes vocabulary chunks when N < V and row
 * chunks otherwise. The results are the same either way; the workspace size
 * and the speed differ. */
typedef enum {
  FLCE_CHUNK_AXIS_AUTO = 0,
  FLCE_CHUNK_AXIS_ROWS = 1,
  FLCE_CHUNK_AXIS_VOCAB = 2
} flce_chunk_axis;

enum {
  FLCE_OK = 0,
  FLCE_ERR_INVALID_ARG = 1,  /* NULL pointer, bad size, dtype, reduction or scalar   */
  FLCE_ERR_UNSUPPORTED = 2,  /* the current device is not sm_103 (GB300), or the
                                entry point does not take this dtype                */
  FLCE_ERR_ALIGNMENT = 3,    /* a pointer is not 16-B aligned, or H % 8 != 0       */
  FLCE_ERR_WORKSPACE = 4,    /* NULL workspace or ws_bytes below the required size */
  FLCE_ERR_CUDA = 5,         /* a CUDA runtime call failed                          */
  FLCE_ERR_TARGET_RANGE = 6, /* device: a target outside [0,V) and != ignore_index  */
  FLCE_ERR_TIMEOUT = 7,      /* device: a bounded wait in a kernel expired          */
  FLCE_ERR_BOUNDS = 8        /* device, debug build only: a kernel store would have
                                fallen outside its buffer and was skipped           */
};

typedef struct {
  int64_t N;                 /* rows (tokens), >= 0                                   */
  int64_t H;                 /* hidden size, >= 1; bf16/fp16 need H % 8 == 0 (16-B rows) */
  int64_t V;                 /* vocabulary size, >= 1                                 */
  int32_t dtype;             /* flce_dtype of hidden, weight, bias and all gradients  */
  int32_t reduction;         /* flce_reduction                                        */
  int64_t ignore_index;      /* rows whose target equals it are ignored (usually -100)*/
  float logit_scale;         /* s: finite and nonzero (1.0 = off)                     */
  float softcap;             /* c: > 0 enables the tanh softcap; <= 0 disables it     */
  float z_loss_multiplier;   /* zeta: finite, >= 0 (0.0 = off)                        */
  int32_t has_bias;          /* 1 if a bias vector is given                           */
  int32_t deterministic;     /* accepted for API parity; every reduction here is
                                already in fixed order, so both values give the same
                                bits                                                  */
  int32_t accumulate;        /* 1: the backward adds into grad_hidden, grad_weight and
                                grad_bias (beta = 1) instead of overwriting them, as
                                quack's fused accumulation into weight.grad does       */
  int32_t grad_weight_accum; /* flce_accum; FLCE_ACCUM_FP32 by default               */
  int64_t vocab_start;       /* vocabulary shards: `weight` (and bias) hold global ids
                                vocab_start .. vocab_start+V-1 of vocab_total. targets
                                are global ids. 0 when not sharded                     */
  int64_t vocab_total;       /* global vocabulary size; 0 means V (not sharded)       */
  int32_t bwd_chunk_axis;    /* flce_chunk_axis of the backward; 0 = AUTO             */
  int32_t max_chunk;         /* >= 0. If > 0, an upper bound on the rows or vocabulary
                                columns of one backward chunk, rounded down to whole
                                tiles (256 rows or columns on the 16-bit path, 64 rows
                                on the fp32 path; at least one tile). It lowers the
                                workspace at the cost of more launches. 0 = only the
                                4 GiB bound on the dlogits copies                     */
} flce_params;

/*
 * Device bytes the caller must provide as `workspace` for one pass. The
 * forward and backward need different amounts, and one workspace may serve
 * both passes in turn. For the headline size (N=8192, H=4096, V=128256,
 * bf16, with bias) the forward needs 16.6 MB and the backward 1.29 GB:
 * - N < V, so the backward chunks the vocabulary: half of V (64256 columns)
 *   of dlogits for all rows, row-major (1.05 GB), and h transposed (67 MB);
 * - the fp32 grad_hidden partial carried across the chunks (134 MB);
 * - per-128-row bias partial sums (33 MB).
 * With N >= V it chunks rows instead (half of the rows of dlogits per chunk,
 * and h transposed) and holds the fp32 grad_weight partial (H x round_up(V, 8)
 * x 4 bytes) with FLCE_ACCUM_FP32. Adding into existing gradients with
 * FLCE_ACCUM_FP32 keeps two dlogits copies of a quarter of the rows (row-major
 * and transposed) and a V x H x 4-byte partial instead. No workspace of either
 * layout reaches the N x V x 2 bytes of the logits in 16 bits.
 * Returns FLCE_OK and sets *bytes, or an argument error.
 */
int flce_workspace_bytes(const flce_params* p, int pass, size_t* bytes);

/*
 * The regions of a pass's workspace that its kernels may write, in address
 * order: name, byte offset from the start of the workspace and byte count.
 * Two regions share their bytes only where the pass uses them one after the
 * other (flce_chunk_grads: grad_hidden's split partials, then h transposed).
 * Every byte of the workspace outside them is left as the caller gave it.
 * This is the layout flce_workspace_bytes sizes; the same p and pass give the
 * same regions. It is a diagnostic: tests fill the workspace with a pattern
 * and check, after a call, that no byte outside a region changed (a stand-in
 * for a memory checker). Writes up to `max` records to `out` and the number
 * of regions to *count. Returns FLCE_OK or an argument error.
 */
typedef struct {
  char name[24];
  uint64_t offset;
  uint64_t bytes;
} flce_region;

int flce_workspace_regions(const flce_params* p, int pass, flce_region* out, int max,
                           int* count);

/*
 * Forward: loss, per-row log-sum-exp and optional metrics.
 *   hidden    device [N,H] dtype
 *   weight    device [V,H] dtype
 *   bias      device [V] dtype, or NULL when has_bias == 0
 *   targets   device [N] int64
 *   loss      device float: [1] for SUM and MEAN, [N] for NONE (ignored rows 0).
 *             MEAN divides by the number of valid rows in this call. With no
 *             valid row it is NaN (0/0, as F.cross_entropy gives).
 *   lse       device float [N]: lse_i of every row, ignored rows included.
 *             flce_backward needs it.
 *   num_correct  device int64 [1] or NULL: #{valid i : argmax_j z_ij == t_i}.
 *             Ties go to the lowest j.
 *   entropy_sum  device float [1] or NULL: sum over valid rows of the softmax
 *             entropy of z_i in nats.
 *   Whether or not the metric pointers are given, loss and lse are
 *   bit-identical (fused-linear-ce README, "Metrics for free").
 *   workspace device, >= flce_workspace_bytes(p, FLCE_PASS_FORWARD) bytes.
 *   With N == 0, hidden, targets and lse may be NULL (and loss too for NONE).
 *   SUM then gives 0 and MEAN gives NaN.
 *   The loss needs the whole vocabulary, so vocab_total must be 0 or V (see
 *   flce_forward_partial for shards).
 */
int flce_forward(const flce_params* p, const void* hidden, const void* weight,
                 const void* bias, const int64_t* targets, float* loss, float* lse,
                 int64_t* num_correct, float* entropy_sum, void* workspace,
                 size_t ws_bytes, flce_stream_t stream);

/*
 * Backward: gradients of the reduced loss, recomputing every logit tile.
 *   lse         device float [N], as written by flce_forward on the same inputs
 *   grad_loss   device float: [1] for SUM and MEAN, [N] for NONE. This is the
 *               upstream gradient of the loss output.
 *   grad_hidden device [N,H] dtype, or NULL to skip it
 *   grad_weight device [V,H] dtype, or NULL to skip it
 *   grad_bias   device [V] dtype, or NULL to skip it (requires has_bias == 1
 *               when given)
 * dlogits is rounded to the input dtype (fp16: times an exact power of two)
 * before the two contractions.
 * - N < V (vocabulary chunks): grad_hidden is accumulated in fp32 across the
 *   chunks, in chunk order, and cast once. Each grad_weight row is complete
 *   after one contraction over all N rows.
 * - N >= V (row chunks): grad_weight is accumulated across the chunks, in
 *   chunk order, in fp32 and cast once ("Chunked Linear Loss", section
 *   "Weight-gradient accumulation dtype", the "fp32" default), or in the
 *   weight dtype with FLCE_ACCUM_WEIGHT.
 *   workspace   device, >= flce_workspace_bytes(p, FLCE_PASS_BACKWARD) bytes
 * With N == 0, the row-indexed pointers may be NULL. grad_weight and grad_bias
 * are then zero-filled.
 */
int flce_backward(const flce_params* p, const void* hidden, const void* weight,
                  const void* bias, const int64_t* targets, const float* lse,
                  const float* grad_loss, void* grad_hidden, void* grad_weight,
                  void* grad_bias, void* workspace, size_t ws_bytes,
                  flce_stream_t stream);

/*
 * Vocabulary-parallel use (a W split by rows across ranks, or across calls).
 *
 * The per-row online state of one shard (20 bytes). Gathered from every shard,
 * these states give the exact loss, lse and metrics. The fused-linear-ce
 * README ("Metrics for free") asks for results that recombine across ranks;
 * the vocabulary-tiled forward merges exactly these states across vocabulary
 * tiles ("Algorithm").
 *   max_logit    largest z_ij of the row within the shard
 *   sum_exp      sum_j exp(z_ij - max_logit) over the shard
 *   sum_z_exp    sum_j z_ij exp(z_ij - max_logit) over the shard
 *   argmax       global vocabulary id of the first maximum within the shard
 *   target_logit z_{i,t_i} if t_i lies in the shard, else 0
 */
typedef struct {
  float max_logit;
  float sum_exp;
  float sum_z_exp;
  int32_t argmax;
  float target_logit;
} flce_row_state;

/*
 * The vocabulary sweep of one shard. p->V is the shard size. p->vocab_start
 * and p->vocab_total place the shard in the global vocabulary. targets hold
 * global ids. Writes states[N] (device, 4-byte aligned).
 * workspace: flce_workspace_bytes(p, FLCE_PASS_FORWARD) bytes.
 */
int flce_forward_partial(const flce_params* p, const void* hidden, const void* weight,
                         const void* bias, const int64_t* targets, flce_row_state* states,
                         void* workspace, size_t ws_bytes, flce_stream_t stream);

/*
 * Merges the states of num_shards shards into flce_forward's outputs. states is
 * [num_shards][N] (device), with the shards in increasing vocabulary order, so
 * that argmax ties go to the lowest global id. p->vocab_total (or p->V when 0)
 * is the global vocabulary size used to validate targets. The backward of a
 * shard is flce_backward with the same p and the merged lse. Its grad_hidden
 * is that shard's share, to be summed over shards (for example with
 * accumulate = 1 into one buffer). Its grad_weight and grad_bias are the
 * shard's rows.
 */
int flce_forward_combine(const flce_params* p, const flce_row_state* states, int32_t num_shards,
                         const int64_t* targets, float* loss, float* lse, int64_t* num_correct,
                         float* entropy_sum, void* workspace, size_t ws_bytes,
                         flce_stream_t stream);

/*
 * flce_forward without a workspace argument, for callers that cannot
 * allocate device memory. The pages have no counterpart; this entry point is
 * this library's own.
 *
 * Who needs it. Some callers cannot call cudaMalloc or any allocator:
 * - frameworks that forbid allocation on the hot path once their memory
 *   plan is fixed;
 * - runtimes that own every byte of device memory through a fixed arena;
 * - plain C hosts that only hold pointers to tensors they already have.
 *
 * Behaviour.
 * - Same arguments and results as flce_forward, minus the workspace. The
 *   kernels are identical, so the outputs are bit-identical too.
 * - The scratch (partial states, target logits, block sums) lives in one
 *   fixed 48 MiB device array inside this library. Every GPU that loads the
 *   library holds it until the process exits.
 * - Sizes whose forward scratch (flce_workspace_bytes with
 *   FLCE_PASS_FORWARD) exceeds 48 MiB are rejected with FLCE_ERR_WORKSPACE
 *   and a message on stderr, before any work is enqueued. The headline size
 *   N=8192, V=128256 needs about 17 MB.
 * - The first call on each device looks up the array's device address, with
 *   that device current. Make that first call before any stream capture.
 * - Every call on a device shares the one array, which keeps the last call's
 *   contents. The call zeroes the status word itself, and every other
 *   scratch byte is written before it is read. Calls that overlap on the GPU
 *   (different streams, or several host threads) race on the array, so
 *   serialise them.
 * - flce_check_status cannot reach the array, so the outputs carry the
 *   device-detected errors: a target out of range makes that row's loss NaN
 *   (and so a SUM or MEAN loss), and an expired bounded wait makes the loss,
 *   every lse and entropy_sum NaN and num_correct -1, whatever the array held
 *   from an earlier call.
 */
int flce_forward_noalloc(const flce_params* p, const void* hidden, const void* weight,
                         const void* bias, const int64_t* targets, float* loss, float* lse,
                         int64_t* num_correct, float* entropy_sum, flce_stream_t stream);

/*
 * Generic chunked linear loss ("Chunked Linear Loss": sections "Why chunk the
 * projection?", "What is fused?", "Loss function contract"). For a loss that
 * the caller evaluates one row chunk at a time, the library runs the parts
 * the strategy owns there: the projection of the chunk, and the folding of
 * the chunk's logits gradient into grad_input and grad_weight. Between the two
 * calls the caller's own code turns the logits chunk into the chunk's loss and
 * dlogits. Only one chunk of logits exists at a time.
 *
 * For one row chunk hidden[N,H] (N = p->N rows), with W[V,H]:
 *
 * flce_chunk_logits:  logits[r][v] = sum_k hidden[r][k] W[v][k]
 *   - Written in the input dtype, from fp32 accumulation. bf16 and fp16 use
 *     the tcgen05 GEMM; fp32 uses the SIMT path.
 *   - `logits` is device memory of N rows of ld_logits elements.
 *     ld_logits >= V and ld_logits % 8 == 0. The tensor path may write up to
 *     round_up(V, 8) elements of a row.
 *   - The workspace holds the status word: FLCE_PASS_CHUNK_LOGITS bytes.
 *   - Alignment: 16 bytes for bf16 / fp16. For fp32 inputs hidden, weight,
 *     logits, dlogits and the gradients need only 4-byte alignment, so a
 *     chunk may start at any row. Workspaces are always 16-byte aligned.
 *   - Of p, only N, H, V and dtype matter here; the other fields must still
 *     pass the usual checks.
 *
 * flce_chunk_grads:
 *   grad_hidden[r][k]  = sum_v dlogits[r][v] W[v][k]        (the chunk's rows)
 *   grad_weight[v][k] += sum_r dlogits[r][v] hidden[r][k]   (over all chunks)
 *   - dlogits is device memory of N rows of ld_dlogits elements in the input
 *     dtype (ld_dlogits >= V, ld_dlogits % 8 == 0), as the caller's loss
 *     returned it.
 *   - On the 16-bit path grad_weight is computed transposed, as
 *     (hidden^T dlogits)^T: the chunk's hidden rows are transposed into the
 *     workspace and dlogits is read along its rows, so no transposed copy is
 *     needed.
 *   - dlogits_t (optional, bf16 / fp16): the same values transposed, V rows of
 *     ld_dlogits_t >= N elements (ld_dlogits_t % 8 == 0), as
 *     flce_chunk_weighted_mse writes them. Read only when an fp32-accumulated
 *     grad_weight is added into an existing one (FLCE_ACCUM_FP32 with
 *     p->accumulate = 1), where grad_weight then reads it K-major, about 20 %
 *     faster than reading dlogits across its rows. NULL if absent.
 *   - grad_hidden points to the chunk's rows. It is overwritten, or added to
 *     when p->accumulate is 1. NULL skips it.
 *   - grad_weight (V x H) is summed over the chunks of one loss, which the
 *     caller numbers with `phase`:
 *     - with p->grad_weight_accum = FLCE_ACCUM_FP32 (the default, "Chunked
 *       Linear Loss", "Weight-gradient accumulation dtype") the sum runs in
 *       an fp32 partial in the workspace. FIRST starts it (from grad_weight
 *       when p->accumulate is 1), NEXT adds, and LAST adds and writes
 *       grad_weight. With ONLY, grad_weight is written (or added to) directly;
 *     - with FLCE_ACCUM_WEIGHT every chunk after the first adds into
 *       grad_weight in the weight dtype.
 *     NULL skips it.
 *   - N must be at least 1.
 *   - The workspace holds FLCE_PASS_CHUNK_GRADS bytes, queried with the
 *     largest chunk's N. The same workspace must go to every chunk of one
 *     loss, in order, on one stream.
 *   - Errors: as for flce_backward.
 */
int flce_chunk_logits(const flce_params* p, const void* hidden, const void* weight, void* logits,
                      int64_t ld_logits, void* workspace, size_t ws_bytes, flce_stream_t stream);

int flce_chunk_grads(const flce_params* p, const void* hidden, const void* weight,
                     const void* dlogits, int64_t ld_dlogits, const void* dlogits_t,
                     int64_t ld_dlogits_t, int32_t phase, void* grad_hidden, void* grad_weight,
                     void* workspace, size_t ws_bytes, flce_stream_t stream);

/*
 * A loss computed on the device for the chunked linear loss: the row- and
 * feature-weighted squared error that "Chunked Linear Loss" ("Direct logits
 * gradients") writes as a caller's callback,
 *
 *   L       = sum_rv r_r f_v (z_rv - y_rv)^2,   z = hidden W^T (this chunk)
 *   dlogits = 2 r_r f_v (z_rv - y_rv)
 *
 * It replaces flce_chunk_logits plus the callback for one chunk. The logits
 * stay in the GEMM's fp32 accumulator: the epilogue reads the target and the
 * weights, writes dlogits (input dtype) and per-tile row sums of the loss.
 * A fixed-order reduction then sets *loss (fp64, device) to the chunk's loss,
 * or adds it when accumulate_loss is 1. Pass dlogits to flce_chunk_grads.
 *
 * - bf16 / fp16 only (FLCE_ERR_UNSUPPORTED for fp32 inputs).
 * - target: fp32 [N][ld_target], ld_target >= V and a multiple of 4.
 * - row_weight: fp32 [N], 4-byte aligned; feature_weight: fp32 [V], 16-byte
 *   aligned; target 16-byte aligned.
 * - dlogits: [N][ld_dlogits] in the input dtype, ld_dlogits >= V and a
 *   multiple of 8; up to round_up(V, 8) elements of a row may be written.
 * - dlogits_t (optional): the same values transposed, [V][ld_dlogits_t] with
 *   ld_dlogits_t >= N and a multiple of 8, for flce_chunk_grads' grad_weight.
 *   NULL skips it.
 * - loss: one device double, 8-byte aligned.
 * - workspace: FLCE_PASS_CHUNK_MSE bytes (the status word and the partials).
 */
int flce_chunk_weighted_mse(const flce_params* p, const void* hidden, const void* weight,
                            const float* target, int64_t ld_target, const float* row_weight,
                            const float* feature_weight, void* dlogits, int64_t ld_dlogits,
                            void* dlogits_t, int64_t ld_dlogits_t, double* loss,
                            int32_t accumulate_loss, void* workspace, size_t ws_bytes,
                            flce_stream_t stream);

/*
 * dst[i] = src[i] * (*scale) for i < count, in dtype (flce_dtype): the
 * chunked linear loss's backward, which returns the gradients computed in
 * the forward scaled by the upstream scalar gradient ("Chunked Linear Loss",
 * "Gradient handling"). scale is one device float, read by the kernel, so the
 * call never synchronises. src == dst scales in place; then a scale of 1
 * costs one launch and no memory traffic. src and dst must not overlap
 * otherwise, and must be aligned to their element size.
 */
int flce_scale(const void* src, void* dst, int64_t count, int32_t dtype, const float* scale,
               flce_stream_t stream);

/*
 * Synchronises `stream`, then returns the device-detected status of the last
 * pass that used `workspace`. The status is FLCE_OK, FLCE_ERR_TARGET_RANGE,
 * FLCE_ERR_TIMEOUT or (debug build) FLCE_ERR_BOUNDS, or FLCE_ERR_CUDA if the
 * synchronisation itself failed.
 */
int flce_check_status(const void* workspace, flce_stream_t stream);

/* Static English description of a return code. Never NULL. */
const char* flce_error_string(int code);

/* Static text naming the last CUDA or tensor-map failure on this host
 * thread (empty if none). It is meant for diagnostics after FLCE_ERR_CUDA or
 * FLCE_ERR_UNSUPPORTED. Never NULL. */
const char* flce_last_error_detail(void);

/*
 * Test hook for the bounded waits; not for production use. From this call on,
 * every forward pass launched from the calling host thread starves one TMA
 * pipeline stage: the even CTA of the CTA pair that takes the first unit (row
 * block 0, vocabulary tile 0) arms the stage of K slice `drop_kblock` of that
 * tile but never issues its loads, so the MMA's
 * wait on it must expire. wait_ms > 0 shortens every wait of those launches
 * to that many milliseconds (0 keeps the default of 4 s). The kernel then
 * records FLCE_ERR_TIMEOUT in the status word, stops its other roles, drains
 * its copies in flight, frees its tensor memory and returns; the forward's
 * outputs are NaN as described above. drop_kblock = -1 (with wait_ms = 0)
 * turns the hook off again. Other host threads are not affected. Returns
 * FLCE_ERR_INVALID_ARG for drop_kblock < -1 or wait_ms < 0.
 */
int flce_test_fault(int32_t drop_kblock, int32_t wait_ms);

/* Number of kernels this library has launched in this process. */
uint64_t flce_launch_count(void);

/*
 * Per-kernel timing on the launching stream. While enabled, each launch is
 * bracketed by two CUDA events, and each tensor-core launch also sums its
 * CTAs' SM clock cycles and elapsed nanoseconds into a record of a fixed
 * 4096-entry array in the library's static device memory (no allocation;
 * launches past the 4096th before a read get no record; the first profiled
 * launch after a read zeroes the whole array on its stream, and a launch on
 * another stream zeroes its own record).
 * flce_profiling_read synchronises those events. It fills up to `max`
 * records, in first-launch order, with the kernel name, the number of
 * launches, their total duration in milliseconds and their mean SM clock in
 * MHz (cycles over nanoseconds; 0 for kernels without a record). For the
 * tensor-core kernels it adds the share of the MMA-issuing thread's cycles
 * spent waiting for operands to land in shared memory, and waiting for the
 * epilogue to free an accumulator; the rest is issuing MMAs and waiting for
 * the tensor cores to take them. It then clears the counts. *count is set to
 * the number of distinct kernels.
 */
typedef struct {
  char name[48];
  uint64_t launches;
  double total_ms;
  double sm_mhz;
  double mma_wait_operands;     /* fraction of the MMA thread's cycles, 0..1 */
  double mma_wait_accumulator;  /* fraction of the MMA thread's cycles, 0..1 */
} flce_kernel_time;

int flce_profiling_enable(int on);
int flce_profiling_read(flce_kernel_time* out, int max, int* count);

#ifdef __cplusplus
}
#endif
#endif /* FLCE_H_ */
