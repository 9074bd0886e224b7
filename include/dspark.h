/*
 * dspark.h -- C ABI of the DSpark decode-cycle hot path on one GB300 GPU.
 *
 * One DSpark decode cycle, as the pages describe it:
 *   1. draft   -- the Markov-head block draft: per position k the drafter's
 *                 logits are the backbone's base logits U_k plus a low-rank
 *                 bias of the previous sampled token, sampled left to right
 *                 ("DSpark explainer", papers.franksyz.com topic 31, sections
 *                 6-7; llama.cpp PR 25173 "spec: add DSpark speculative
 *                 decoding", description: anchor-first block,
 *                 bias(prev) = markov_w2 . markov_w1[prev]);
 *   2. select  -- survival a = cumulative product of the confidences and a
 *                 prefix-closed choice of verify lengths within a physical
 *                 capacity (explainer sections 5, 8, 9, 10);
 *   3. verify  -- left-to-right acceptance min(1, p/q), residual
 *                 max(0, p - q) on the first rejection, a bonus token when
 *                 every draft is accepted (explainer sections 2-3), over
 *                 target rows packed back to back (section 13);
 *   4. commit  -- lengths of what each request commits and rolls back
 *                 (sections 2 and 11).
 *
 * Conventions shared by every call:
 *   - Every array argument is a DEVICE pointer owned by the caller; the
 *     library allocates no memory and keeps no state between calls (apart
 *     from the two process-wide wait settings of dspark_set_wait_limit_ns and
 *     dspark_set_fault_injection, which default to "off").  Scratch
 *     lives in a caller-provided workspace of dspark_workspace_size() bytes
 *     (any 256-byte aligned device buffer; its contents need no
 *     initialisation and are clobbered).
 *   - Arrays are row-major and densely packed; the shapes are given beside
 *     each argument.  Token ids and lengths are int32.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream), never synchronises and never throws.  It
 *     returns DSPARK_OK once its kernels are enqueued, or a negative status
 *     after a host-side check failed, in which case nothing was enqueued.
 *   - Errors found by the kernels (a token id outside [0, V), a verify
 *     length outside [0, gamma], a confidence outside [0, 1], a bounded
 *     device wait that expired) are written asynchronously to *dev_status
 *     (an int32 the caller zeroes; first error wins) when dev_status is not
 *     NULL, and the affected request's outputs are set to -1.
 *   - Random numbers: counter-based Philox4x32-10 keyed by the request's
 *     64-bit seed, counter (vocab index / 4, block position, request index,
 *     cycle << 4 | purpose), purposes 0 draft noise, 1 acceptance, 2
 *     residual noise, 3 bonus noise; the uniform from a 32-bit word x is
 *     ((x >> 9) + 0.5) * 2^-23.  cycle must be < 2^28.  Reusing (seed,
 *     cycle) reproduces a cycle exactly.
 *   - temperature == 0 means greedy decoding on both sides; otherwise the
 *     logits are multiplied by invT = 1.0f / temperature computed in fp32.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; declared opaquely so that this header needs no CUDA header. */
typedef struct CUstream_st* dspark_stream_t;

/* ---- status codes ---------------------------------------------------------- */
#define DSPARK_OK 0
#define DSPARK_ERR_INVALID_ARG (-1)  /* NULL pointer, bad size, gamma > 16, T < 0 ...  */
#define DSPARK_ERR_UNSUPPORTED (-2)  /* a shape or dtype no kernel here handles        */
#define DSPARK_ERR_CAPACITY (-3)     /* R > K_cap, or more rows than max_rows          */
#define DSPARK_ERR_CUDA (-4)         /* a CUDA launch or driver call failed            */
#define DSPARK_ERR_TIMEOUT (-5)      /* device side: a bounded wait gave up            */
#define DSPARK_ERR_DEVICE_INPUT (-6) /* device side: bad token id / length / confidence */
#define DSPARK_ERR_WORKSPACE (-7)    /* workspace NULL, misaligned or too small        */
#define DSPARK_ERR_BOUNDS (-8)       /* DSPARK_DEBUG builds only: a device-side index
                                        check failed; the access was skipped, so the
                                        outputs of that call are invalid            */

/* Largest R the verify calls accept (their per-round request list is kept in
 * shared memory). */
#define DSPARK_VERIFY_MAX_R 16384

/* ---- element types ------------------------------------------------------- */
#define DSPARK_F32 0
#define DSPARK_BF16 1

/* ---- workspace owners ------------------------------------------------------ */
#define DSPARK_OP_DRAFT 0
#define DSPARK_OP_VERIFY 1
#define DSPARK_OP_SELECT 2
#define DSPARK_OP_VERIFY_MARKOV 3
#define DSPARK_OP_CALIBRATE 4
#define DSPARK_OP_DRAFT_FUSED 5

/* Largest hidden size dspark_markov_draft_fused takes. */
#define DSPARK_FUSED_MAX_D 16384

/* ---- dspark_workspace_size flags for DSPARK_OP_VERIFY_MARKOV --------------------- */
#define DSPARK_VERIFY_HOST_TARGET 1u /* target_logits will be pinned host memory */

/* ---- dspark_markov_draft flags ---------------------------------------------- */
#define DSPARK_DRAFT_FORCE_SIMT 1u   /* use the CUDA-core kernels even where the
                                        tensor-core kernel applies (testing) */

/* ---- selection modes --------------------------------------------------------- */
#define DSPARK_SELECT_FIXED 0      /* capacity K = K_cap                              */
#define DSPARK_SELECT_HISTORY 1    /* capacity from c_hist (the confidences of an
                                      earlier cycle), explainer section 10            */
#define DSPARK_SELECT_CURRENT 2    /* capacity from the current c; it looks at values
                                      that admission must not see (section 4), kept
                                      only to study the planner                       */
#define DSPARK_SELECT_FIRST_STOP 3 /* the theoretical greedy of section 9: add the best
                                      remaining candidate while Theta strictly grows  */
#define DSPARK_SELECT_CONF_CUTOFF 4     /* static per-request cutoff on the per-position
                                           confidence: positions before the request's first
                                           c[r][k] < conf_min (llama.cpp PR 25173's conf_min
                                           pruning; the Strata plan's first milestone)     */
#define DSPARK_SELECT_SURVIVAL_CUTOFF 5 /* static per-request cutoff on the survival:
                                           positions with a[r][k] >= conf_min (the fixed
                                           per-request threshold section 9 compares with)   */

/* Static text for a status code. */
const char* dspark_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch (1.1.0: cutoff modes,
 * conf_min in dspark_select_prefix, dspark_plan_cycles, the wait settings,
 * dspark_fit_temperatures, dspark_kv_reserve and dspark_kv_commit; 1.2.0:
 * dspark_markov_draft_fused). */
int dspark_version(void);

/* Bytes of workspace one call of `op` needs for these sizes (0 on bad
 * arguments).  For DSPARK_OP_DRAFT pass the weights' element type and the
 * draft flags; for DSPARK_OP_VERIFY, max_rows bounds cu_seqlens[R]; other
 * arguments may be 0 where unused. */
size_t dspark_workspace_size(int op, int R, int gamma, int V, int rank, int max_rows,
                             int w_dtype, unsigned flags);

/* 1 if dspark_markov_draft would use the tcgen05 tensor-core kernel for these
 * arguments, 0 for the CUDA-core kernels.  The tensor-core kernel takes bf16 U
 * and factors, rank a multiple of 64 up to 512, V a multiple of 8, and at most
 * 128 requests per SM of the current device (all positions run in one launch
 * whose CTAs are resident together).  Everything else -- fp32 operands, rank
 * 576 .. 1024, rank not a multiple of 64, V % 8 != 0, more requests -- runs on
 * the CUDA-core kernels, about 40x slower at the R = 128, V = 151936, rank 512
 * shape. */
int dspark_markov_draft_uses_tensor_cores(int u_dtype, int w_dtype, int R, int V, int rank,
                                          unsigned flags);

/*
 * dspark_philox4x32_10 -- the generator every random draw of the cycle comes
 * from (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 * 1, 2, 3", SC'11), exposed so that callers and tests can reproduce draws.
 *   ctr [n, 4] uint32 counters, keys [n] uint64, out [n, 4] uint32 (device).
 */
int dspark_philox4x32_10(const uint32_t* ctr, const uint64_t* keys, int n, uint32_t* out,
                         dspark_stream_t stream);

/*
 * dspark_markov_draft -- semi-autoregressive Markov-head block draft
 * (explainer sections 6-7; PR 25173 description, draft-dspark bullet).
 *
 * For k = 0 .. gamma-1, for every request r:
 *   prev = anchor[r] at k = 0 (anchor < 0: no bias at k = 0), else y[r][k-1]
 *   s_v  = (U[r][k][v] + sum_j W2[v][j] * W1[prev][j]) * invT   (T > 0)
 *   s_v  =  U[r][k][v] + sum_j W2[v][j] * W1[prev][j]           (T = 0)
 *   y[r][k] = argmax_v (s_v + Gumbel(u_v)) with u from purpose 0 at position k
 *             (T = 0: argmax_v s_v); ties go to the lowest v
 *   q_lse[r][k] = log sum_v exp(s_v),  q_tok[r][k] = exp(s_y - q_lse)   (T > 0 only)
 *   q_logits[r][k][v] = s_v                                            (if not NULL)
 * The steps run in order on `stream`; step k reads the tokens of step k-1.
 *
 *   U          [R, gamma, V]  u_dtype (F32 or BF16)
 *   W1, W2     [V, rank]      w_dtype (F32 or BF16), the Markov factors
 *   anchor     [R] int32      last committed token of each request
 *   seeds      [R] uint64     per-request Philox keys (may be NULL iff T == 0)
 *   draft_tokens [R, gamma] int32 out
 *   q_lse, q_tok [R, gamma] fp32 out (may be NULL iff T == 0)
 *   q_logits   [R, gamma, V] fp32 out; NULL skips it (needed by dspark_verify at T > 0)
 *   ws, ws_bytes  workspace of dspark_workspace_size(DSPARK_OP_DRAFT, R, gamma, V,
 *                 rank, 0, w_dtype, flags) bytes
 * Limits: 1 <= gamma <= 16, R >= 1, V >= 1, rank >= 1.  The tensor-core kernel
 * applies to BF16 U and weights with rank % 64 == 0, rank <= 512, V % 8 == 0
 * and R <= 128 x the SM count (dspark_markov_draft_uses_tensor_cores says
 * which); everything else runs on the CUDA-core kernels (a per-position bias
 * GEMV and a sampling pass; correct, but far slower).
 */
int dspark_markov_draft(const void* U, int u_dtype, const void* W1, const void* W2,
                        int w_dtype, const int32_t* anchor, const uint64_t* seeds,
                        uint32_t cycle, float temperature, int R, int gamma, int V,
                        int rank, int32_t* draft_tokens, float* q_lse, float* q_tok,
                        float* q_logits, unsigned flags, void* ws, size_t ws_bytes,
                        int32_t* dev_status, dspark_stream_t stream);

/*
 * dspark_markov_draft_fused -- the block draft with the drafter's logits formed
 * in one contraction from its hidden states (explainer section 6: the parallel
 * backbone gives every block position's hidden state in one pass, the base
 * logits come from it; PR 25173 description: the drafter shares the target's
 * lm_head, bias(prev) = markov_w2 . markov_w1[prev]).
 *
 * Exactly dspark_markov_draft with
 *   U[r][k][v] = sum_i W_lm[v][i] * h[r][k][i]
 * except that U is never stored: per position the kernel contracts
 * [W_lm | W2] (V x (d + rank)) with [h[r][k] ; W1[prev]] in one fp32
 * accumulator, so U keeps fp32 precision instead of a bf16 rounding.  It reads
 * W_lm once per position (gamma * V * d * 2 bytes), so it pays off against
 * writing and reading U (R * gamma * V * 2 bytes twice, plus a separate lm_head
 * GEMM) where the contraction is tensor-bound, i.e. at large R.
 *
 *   h          [R, gamma, d]  bf16: hidden state of request r at block position k
 *   W_lm       [V, d]         bf16: the lm_head shared with the target
 *   d          hidden size, a multiple of 64, <= DSPARK_FUSED_MAX_D
 *   W1, W2     [V, rank]      bf16 Markov factors (rank % 64 == 0, rank <= 512)
 *   everything else as dspark_markov_draft (V % 8 == 0; at most 128 requests
 *   per SM of the current device; h, W_lm, W1, W2 16-byte aligned).
 *   ws, ws_bytes  workspace of dspark_workspace_size(DSPARK_OP_DRAFT_FUSED, R,
 *                 gamma, V, rank, 0, DSPARK_BF16, 0) bytes
 * Tensor cores only: shapes outside these limits return DSPARK_ERR_UNSUPPORTED
 * (there is no CUDA-core variant).
 */
int dspark_markov_draft_fused(const void* h, const void* W_lm, int d, const void* W1, const void* W2,
                              const int32_t* anchor, const uint64_t* seeds, uint32_t cycle,
                              float temperature, int R, int gamma, int V, int rank,
                              int32_t* draft_tokens, float* q_lse, float* q_tok, float* q_logits,
                              void* ws, size_t ws_bytes, int32_t* dev_status, dspark_stream_t stream);

/*
 * dspark_verify -- lossless left-to-right verification (explainer sections
 * 2, 3 and 13).
 *
 * Request r owns target rows cu_seqlens[r] .. cu_seqlens[r+1]-1, that is
 * l_r + 1 rows with 0 <= l_r <= gamma: rows for the l_r drafts to check and
 * the row after them.  With t = row * invT (T = 0: the row itself),
 * p = softmax(t) and the drafter's q = softmax(q_logits[r][j]):
 *   draft j is accepted iff u_j < p(y_j) / q_tok[r][j], u_j from purpose 1 at
 *   position j (T = 0: iff y_j == argmax of row j); checking stops at the first
 *   rejection.  n_accepted[r] = number accepted.
 *   After a rejection at j the extra token is drawn from max(0, p - q) of row j
 *   by Gumbel-max over log weights (purpose 2, position j); if that residual
 *   is empty in fp32 it is drawn from p with the same noise.  If every draft is
 *   accepted the extra token is drawn from p of row l_r (purpose 3, position
 *   l_r).  T = 0: the extra token is the argmax of row n_accepted.
 *   out_tokens[r] = y[r][0 .. n-1], extra token, then -1 up to gamma + 1 entries.
 *   p_tok[r][j] = p(y_j) for the drafts examined (T = 0: 1 if y_j is the row's
 *   argmax else 0); entries not examined are left untouched.
 *   Rows after a request's first rejection are not read.  R <= DSPARK_VERIFY_MAX_R
 *   (else DSPARK_ERR_UNSUPPORTED).
 *
 *   target_logits [cu_seqlens[R], V] fp32, packed rows without padding
 *   cu_seqlens   [R + 1] int32, cu_seqlens[0] = 0, non-decreasing
 *   draft_tokens [R, gamma] int32;  q_tok, q_lse [R, gamma] fp32 (T > 0)
 *   q_logits     [R, gamma, V] fp32 from dspark_markov_draft (T > 0)
 *   seeds        [R] uint64 (T > 0)
 *   n_accepted [R], out_tokens [R, gamma + 1] int32 out; p_tok [R, gamma] fp32 out or NULL
 *   ws, ws_bytes  dspark_workspace_size(DSPARK_OP_VERIFY, R, gamma, V, 0, max_rows, 0, 0)
 *                 with max_rows >= cu_seqlens[R]
 *   max_rows     the host's bound on cu_seqlens[R] (<= R * (gamma + 1))
 */
int dspark_verify(const float* target_logits, const int32_t* cu_seqlens,
                  const int32_t* draft_tokens, const float* q_logits, const float* q_lse,
                  const float* q_tok, const uint64_t* seeds, uint32_t cycle,
                  float temperature, int R, int gamma, int V, int max_rows,
                  int32_t* n_accepted, int32_t* out_tokens, float* p_tok, void* ws,
                  size_t ws_bytes, int32_t* dev_status, dspark_stream_t stream);

/*
 * dspark_verify_markov -- dspark_verify for a Markov-head drafter, without the
 * drafter's logits in memory (explainer sections 2-3 and 7).
 *
 * Same decisions and outputs as dspark_verify.  Instead of q_logits it takes
 * the drafter's own inputs -- U [R, gamma, V], W1 and W2 [V, rank] (bf16, the
 * shapes dspark_markov_draft_uses_tensor_cores accepts) and anchor [R] -- and
 * recomputes, on the tensor cores, the drafter's scaled logits
 * s_v = (U[r][j][v] + W2[v] . W1[prev_j]) * invT of the one row j each request
 * needs for its residual; q = exp(s - q_lse[r][j]).  One pass over W2 per
 * verify replaces writing and re-reading R * gamma * V fp32 logits.  The
 * draft call then passes q_logits = NULL.
 *   ws, ws_bytes  dspark_workspace_size(DSPARK_OP_VERIFY_MARKOV, R, gamma, V, rank,
 *                 max_rows, DSPARK_BF16, 0)
 * Returns DSPARK_ERR_UNSUPPORTED for factor types or shapes the tensor-core
 * kernel does not take (use dspark_verify with q_logits there), and at
 * temperature > 0 when target_logits, U, W1 or W2 is not 16-byte aligned (the
 * residual kernel reads the rows in 16-byte pieces).
 *
 * Target rows in host memory.  target_logits may also point to pinned
 * (page-locked) host memory that the device can read (cudaHostAlloc /
 * cudaHostRegister; on a Grace-Blackwell node the link is NVLink-C2C): the
 * kernels then read across the link only the rows they examine -- each
 * request's rows up to its first rejection -- instead of the caller copying
 * every presented row.  The decision pass keeps a device copy of each request's
 * latest row for the residual draw, so at temperature > 0 the workspace must be
 * dspark_workspace_size(DSPARK_OP_VERIFY_MARKOV, R, gamma, V, rank, max_rows,
 * DSPARK_BF16, DSPARK_VERIFY_HOST_TARGET) bytes (R * V * 4 more).  Pageable host
 * memory is refused (DSPARK_ERR_UNSUPPORTED), and so is any host memory in
 * dspark_verify.
 */
int dspark_verify_markov(const float* target_logits, const int32_t* cu_seqlens,
                         const int32_t* draft_tokens, const void* U, const void* W1,
                         const void* W2, const int32_t* anchor, int rank, const float* q_lse,
                         const float* q_tok, const uint64_t* seeds, uint32_t cycle,
                         float temperature, int R, int gamma, int V, int max_rows,
                         int32_t* n_accepted, int32_t* out_tokens, float* p_tok, void* ws,
                         size_t ws_bytes, int32_t* dev_status, dspark_stream_t stream);

/*
 * dspark_verify_static_scratch -- dspark_verify for callers that cannot
 * provide a workspace.  The pages have no counterpart of this call; it exists
 * for callers that are not allowed to allocate device memory, such as a plugin
 * inside a serving engine whose device memory is all owned and accounted by
 * the engine's own pool (an extra cudaMalloc can synchronise the device and
 * escapes that accounting), or code that has no spare buffer to pass down.
 *
 * Same arguments, results and status codes as dspark_verify, minus ws and
 * ws_bytes.  The scratch is a static device array of
 * DSPARK_VERIFY_STATIC_SCRATCH_BYTES (4 MiB) compiled into the library; every
 * GPU that loads the library holds it until the process exits.  The call
 * allocates nothing.  Sizes whose scratch need
 * (dspark_workspace_size(DSPARK_OP_VERIFY, R, gamma, V, 0, max_rows, 0, 0),
 * about R * (32 * ceil(V / 1024) + 32 * ceil(V / 8192) + 56) bytes) exceeds the
 * array return DSPARK_ERR_CAPACITY and enqueue nothing: R <= 772 at
 * V = 151936, R <= 905 at V = 129280, R <= 3482 at V = 32000.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it for the life
 * of the process; make that first call before any stream capture starts.  The
 * kept address belongs to the device's primary context: do not call this
 * function again after cudaDeviceReset() (the module is then loaded anew,
 * possibly at another address).  All calls on a device share the array and it
 * keeps the last call's contents; the kernels reset their own counters, flags
 * and per-request rows at the start of every call, so nothing has to be
 * cleared beforehand.  Calls whose kernels overlap on the GPU (for example on
 * two streams at once) race on the array: serialise them.
 */
#define DSPARK_VERIFY_STATIC_SCRATCH_BYTES (4u * 1024u * 1024u)

int dspark_verify_static_scratch(const float* target_logits, const int32_t* cu_seqlens,
                                 const int32_t* draft_tokens, const float* q_logits,
                                 const float* q_lse, const float* q_tok, const uint64_t* seeds,
                                 uint32_t cycle, float temperature, int R, int gamma, int V,
                                 int max_rows, int32_t* n_accepted, int32_t* out_tokens,
                                 float* p_tok, int32_t* dev_status, dspark_stream_t stream);

/*
 * ---- failure handling: the grid-wide waits --------------------------------
 * The verify rounds (every verify call) and the tensor-core draft (all block
 * positions in one launch) run as cooperative launches whose CTAs meet at
 * grid-wide barriers: between verify rounds, and between draft positions.
 * Every such wait is bounded (explainer section 16: a fault must fall back to
 * target-only decoding, not hang the engine): when it runs out the kernel
 * raises an abort word, every CTA drains the asynchronous copies and tensor-
 * core operations it has in flight and exits, DSPARK_ERR_TIMEOUT is written to
 * *dev_status, and the CUDA context stays usable.  Outputs of a call that
 * reported DSPARK_ERR_TIMEOUT are invalid (requests decided before the wait
 * ran out may have been written; the others are left untouched).  The waits
 * of a CTA on its own asynchronous copies (mbarriers) keep a fixed 2 s limit.
 *
 * dspark_set_wait_limit_ns sets the limit of the grid-wide waits for every
 * later call of this process (0 or anything above 2 s: the default, 2 s) and
 * returns the previous limit.
 *
 * dspark_set_fault_injection is for tests of this failure path: with
 * DSPARK_INJECT_VERIFY_BARRIER the verify rounds' barriers, with
 * DSPARK_INJECT_DRAFT_BARRIER the draft's position barriers, count one
 * arrival more than the grid has, so that no CTA is ever released and every
 * wait runs out after the limit above.  Returns the previous mask; 0 turns
 * injection off.  Both settings are read when a call is enqueued.
 */
#define DSPARK_INJECT_VERIFY_BARRIER 1u
#define DSPARK_INJECT_DRAFT_BARRIER 2u

uint64_t dspark_set_wait_limit_ns(uint64_t limit_ns);
unsigned dspark_set_fault_injection(unsigned mask);

/*
 * dspark_select_prefix -- survival, capacity and prefix-closed top-K
 * (explainer sections 5, 8, 9 and 10).
 *
 *   a[r][k] = a[r][k-1] * c[r][k] in fp32, a[r][0] = c[r][0]
 *   candidates (r, k) are ranked by a descending, then k ascending, then r
 *   ascending; a is non-increasing in k, so every top-n set is prefix-closed.
 *   Theta(n) = SPS(B) * (R + sum of the n best a), B = R + n physical rows; for
 *   a capture size S the step rate is sps[i] for the smallest S_i >= B.
 *   n = min(K_cap - R, R*gamma)                                      (FIXED)
 *   n = n_S of the capture size S >= R maximising
 *       sps_S * (R + sum of the n_S best a_plan), n_S = min(min(S, K_cap) - R, R*gamma),
 *       ties to the smaller S; a_plan from c_hist (HISTORY) or c (CURRENT)
 *   n = the first-stop greedy of section 9, at most K_cap - R         (FIRST_STOP)
 *   n = min(eligible, K_cap - R), the n best eligible candidates in the order above,
 *       where request r is eligible up to its first position k with
 *       c[r][k] < conf_min (CONF_CUTOFF) or a[r][k] < conf_min (SURVIVAL_CUTOFF)
 *   l[r] = selected positions of request r; cu_seqlens[r+1] = cu_seqlens[r] + l[r] + 1
 *   K_used[0] = R + n (the physical rows the verify step will see)
 *
 *   c, c_hist    [R, gamma] fp32 in [0, 1]; c_hist may be NULL except in HISTORY mode
 *   capture_sizes [n_steps] int32, sps [n_steps] fp32 (read by HISTORY, CURRENT and
 *                FIRST_STOP only)
 *   conf_min     the cutoff of the two cutoff modes (not NaN; ignored otherwise)
 *   a [R, gamma] fp32 out; l [R], cu_seqlens [R + 1], K_used [1] int32 out
 * Limits: R * gamma <= 8192, n_steps <= 64.
 */
int dspark_select_prefix(const float* c, const float* c_hist, const int32_t* capture_sizes,
                         const float* sps, int n_steps, int K_cap, int mode, float conf_min, int R,
                         int gamma, float* a, int32_t* l, int32_t* cu_seqlens, int32_t* K_used,
                         void* ws, size_t ws_bytes, int32_t* dev_status,
                         dspark_stream_t stream);

/*
 * dspark_plan_cycles -- the scheduler over a run of consecutive cycles
 * (explainer section 10: the physical capacity of cycle t is planned on the
 * confidences of cycle t - lag, two steps back in the paper's implementation,
 * while the top of cycle t's own survival fills it; section 15: watch the
 * verify work wasted after first rejections).  One launch, one CTA per cycle.
 *
 * Cycle t runs dspark_select_prefix's selection on c_seq[t] in `mode`; in
 * HISTORY mode its c_hist is c_seq[t - lag], and the first lag cycles (no
 * history yet) use the capacity K_cap.  n_full[t][r] is how many leading
 * drafts of request r the target would accept in cycle t (so the cycle accepts
 * n_acc[r] = min(n_full[t][r], l[r])).  With B = K_used[t] and SPS the step
 * rate of the smallest capture size >= B (0 if none):
 *   stats[t][0] = SPS * (R + sum of the selected a)      predicted Theta
 *   stats[t][1] = SPS * (R + sum_r n_acc[r])             achieved Theta (tokens/s)
 *   stats[t][2] = sum_r n_acc[r]                         accepted drafts
 *   stats[t][3] = sum_r (l[r] - n_acc[r])                wasted verify rows
 * (stats[t][1..3] are 0 when n_full is NULL).
 *
 *   c_seq [n_cycles, R, gamma] fp32; n_full [n_cycles, R] int32 or NULL
 *   capture_sizes [n_steps] int32, sps [n_steps] fp32 (always read)
 *   l_seq [n_cycles, R] int32 out, K_seq [n_cycles] int32 out, stats [n_cycles, 4] fp64 out
 * Limits as dspark_select_prefix; lag >= 1; n_cycles <= 2^20.
 */
int dspark_plan_cycles(const float* c_seq, const int32_t* n_full, const int32_t* capture_sizes,
                       const float* sps, int n_steps, int K_cap, int mode, float conf_min, int lag,
                       int n_cycles, int R, int gamma, int32_t* l_seq, int32_t* K_seq, double* stats,
                       int32_t* dev_status, dspark_stream_t stream);

/*
 * dspark_fit_temperatures -- sequential temperature scaling of the confidence
 * head (explainer section 8: the per-position confidences are calibrated left
 * to right by a post-hoc temperature so that their products are calibrated
 * survival probabilities; PR 25173 "Future work": the paper's Sequential
 * Temperature Scaling).
 *
 * Position k is fitted on the samples that reached it (accepted[i][j] != 0 for
 * every j < k), so that c_k = sigmoid(z_k / tau_k) estimates the conditional
 * acceptance rate.  tau_k minimises the labels' negative log-likelihood
 *   NLL(beta) = sum_i softplus(beta z_i[k]) - accepted_i[k] * beta z_i[k],
 * beta = 1 / tau_k (convex in beta), by Newton's method from beta = 1 (halving
 * beta when a step would leave (0, inf)) until the step is below 1e-12 of beta,
 * then beta is clamped to [1e-3, 1e3].  A position no sample reached gets
 * tau = 1 and count 0.
 *
 *   z        [N, gamma] fp32 raw confidence logits
 *   accepted [N, gamma] uint8 labels (0 rejected; entries after a sample's first
 *            rejection are ignored)
 *   tau [gamma] fp32 out; nll [gamma] fp64 out (mean NLL at tau) or NULL;
 *   count [gamma] int32 out (samples that reached the position) or NULL
 *   ws, ws_bytes  dspark_workspace_size(DSPARK_OP_CALIBRATE, 0, gamma, 0, 0, 0, 0, 0)
 * Limits: 1 <= gamma <= 16, N >= 1.  The CTAs of a position meet at bounded
 * barriers between Newton steps (DSPARK_ERR_TIMEOUT if one runs out).
 */
int dspark_fit_temperatures(const float* z, const uint8_t* accepted, int N, int gamma, float* tau,
                            double* nll, int32_t* count, void* ws, size_t ws_bytes, int32_t* dev_status,
                            dspark_stream_t stream);

/*
 * dspark_kv_reserve / dspark_kv_commit -- the paged KV cache's bookkeeping
 * around one verify (explainer section 11: verify writes its candidate rows
 * into temporary pages; after the first rejection only the accepted prefix is
 * promoted and every other candidate's state is released; section 15: leaked
 * or double-freed temporary state is a failure class).
 *
 * State (device memory, owned by the caller):
 *   kv_len      [R] int32    committed tokens of each request
 *   block_table [R, max_blocks] int32  page ids; page b holds positions
 *               [b * page_size, (b + 1) * page_size); a request's committed
 *               pages are its leading ceil(kv_len / page_size) entries, the
 *               rest are -1
 *   free_pages  [pool_pages] int32 stack of free page ids, free_pages[0 .. *free_top)
 *   free_top    [1] int32
 *   pool_pages  the stack's capacity (every page of the pool); no call writes
 *               past it (a state that would make it do so is rejected)
 *
 * dspark_kv_reserve: before the verify, request r needs
 *   need[r] = ceil((kv_len + l + 1) / page_size) - ceil(kv_len / page_size)
 * more pages for its l[r] + 1 verify rows (positions kv_len .. kv_len + l).
 * The top T = sum of needs pages of the stack are handed out in request order
 * (request r takes free_pages[*free_top - T + o_r + i], o_r = the needs of the
 * requests before it) into its next block-table entries; *free_top -= T;
 * reserved[r] = need[r] (reserved may be NULL).  All or nothing: when T >
 * *free_top or a request would pass max_blocks, nothing changes and
 * DSPARK_ERR_CAPACITY goes to *dev_status (DSPARK_ERR_DEVICE_INPUT for a
 * negative length, whichever request comes first).
 *
 * dspark_kv_commit: after the verify (with the l of the reserve), request r
 * keeps its committed prefix plus the rows of its accepted drafts:
 *   kv_len[r] += n_accepted[r] + 1
 * (the same count dspark_commit_lengths reports).  The pages past
 * ceil(kv_len / page_size) held only rejected rows: they go back on the stack
 * in request order (request r's at *free_top + o_r + i, o_r = the pages the
 * requests before it release), their entries become -1 (an entry holding no
 * page is skipped), and *free_top grows by the total.  A request with
 * n_accepted outside [0, l] commits nothing, releases all its reserved pages
 * and is reported (DSPARK_ERR_DEVICE_INPUT).  If the stack could not take the
 * released pages (a state the reserve did not produce), nothing changes and
 * DSPARK_ERR_DEVICE_INPUT is reported.
 * Both calls run in one CTA; R >= 1, page_size >= 1, max_blocks >= 1.
 */
int dspark_kv_reserve(const int32_t* kv_len, const int32_t* l, int R, int page_size, int32_t* block_table,
                      int max_blocks, int32_t* free_pages, int32_t* free_top, int pool_pages, int32_t* reserved,
                      int32_t* dev_status, dspark_stream_t stream);
int dspark_kv_commit(int32_t* kv_len, const int32_t* l, const int32_t* n_accepted, int R, int page_size,
                     int32_t* block_table, int max_blocks, int32_t* free_pages, int32_t* free_top, int pool_pages,
                     int32_t* dev_status, dspark_stream_t stream);

/*
 * dspark_commit_lengths -- per-request commit and rollback counts
 * (explainer sections 2 and 11: the accepted prefix plus one target-correct
 * token is committed, the rest of what was verified is rolled back).
 *
 *   commit_len[r] = n_accepted[r] + 1
 *   cu_commit[0] = 0, cu_commit[r+1] = cu_commit[r] + commit_len[r]
 *   discard[r] = l[r] - n_accepted[r]  (l == NULL: every request verified gamma)
 *   total[0] = cu_commit[R]
 * A request with n_accepted outside [0, l] commits 0 and is reported through
 * dev_status.
 */
int dspark_commit_lengths(const int32_t* n_accepted, const int32_t* l, int R, int gamma,
                          int32_t* commit_len, int32_t* cu_commit, int32_t* discard,
                          int32_t* total, int32_t* dev_status, dspark_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
