/*
 * fattn: exact softmax attention forward on GB300 (sm_103a), C ABI.
 *
 * The operation ("understand-flashattention", forward-pass formulas and the
 * logsumexp derivation; scale-then-mask order and the -inf mask of "PyTorch
 * profiling part 3: attention", section "Naive attention"):
 *
 *     S   = scale * Q K^T                 per (batch b, head h), N x N
 *     S'  = S with masked entries = -inf  (causal: key j visible to query i
 *                                          iff j <= i; key padding: key j
 *                                          visible iff j < key_len[b]; both
 *                                          masks combine with AND)
 *     O   = softmax(S') V                 row-wise softmax
 *     LSE = log(sum_j exp(S'_ij))         natural log, per query row
 *
 * computed tile by tile with the online-softmax recurrence (running max,
 * normaliser and rescaled partial output, normalised once at the end: the
 * two-block derivation of "understand-flashattention").  A row with no
 * visible key returns O = 0 and LSE = -inf (the safe-softmax convention of
 * the profiling page, section "The safe softmax").
 *
 * All entry points are plain C; tensors are raw pointers.  There is no CPU
 * fallback: every result comes from the CUDA kernel.
 */
#ifndef FATTN_H_
#define FATTN_H_

#include <stdint.h>

#if defined(__GNUC__)
#define FATTN_API __attribute__((visibility("default")))
#else
#define FATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Status codes returned by every entry point.  Zero is success and any
 * configuration the library does not run gets a non-zero code instead of a
 * launch: the convention of the host dispatch of the "Linear Attention CUDA
 * kernel" page (its `lmha` entry returns a non-zero value for a feature size
 * it has no kernel for), with the cause split into the codes below.
 */
typedef enum {
  FATTN_OK = 0,
  FATTN_ERR_INVALID_ARG = 1, /* a pointer, size, alignment or scale is invalid */
  FATTN_ERR_UNSUPPORTED = 2, /* valid, but not a configuration the library runs (head dim,
                                no-alloc size) */
  FATTN_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
  FATTN_ERR_TIMEOUT = 4      /* a bounded wait inside the kernel gave up (see fattn_last_error) */
} fattn_status;

/*
 * fattn_fwd: O = softmax(mask(scale * Q K^T)) V and the row log-sum-exp.
 *
 *   q, k, v  device pointers, bf16, [B, H, N, d] contiguous (head dim
 *            innermost, as "PyTorch profiling part 3: attention" lays out
 *            q, k, v: [batch, heads, seq, head_dim]); 16-byte aligned.
 *   o        device pointer, bf16, [B, H, N, d] contiguous, written; 16-byte aligned.
 *   lse      device pointer, fp32, [B, H, N] contiguous, written (natural log).
 *   B, H, N  batch, heads, sequence length (queries = keys = N); each >= 0.
 *            If B*H*N == 0 the call does nothing and returns FATTN_OK.
 *   d        head dim: a multiple of 8 from 8 to 256 (others return
 *            FATTN_ERR_UNSUPPORTED).  d <= 64 runs in the 64-column kernel,
 *            72..128 in the 128-column one, 136..256 in the 256-column
 *            kernel (one query tile per CTA, never split); the columns past d
 *            are read as zeros and never stored, so rows stay d elements long.
 *   scale    softmax scale applied to Q K^T before the mask; finite and >= 0
 *            (usually 1/sqrt(d)).
 *   causal   nonzero: key j is visible to query i only if j <= i.
 *   key_len  device pointer to int32[B] or NULL (all N keys).  Keys
 *            j >= key_len[b] are masked for batch entry b; values are
 *            clamped to [0, N].  Query rows are never masked.
 *   stream   a cudaStream_t (NULL = legacy default stream).
 *
 * Ownership: the caller allocates and owns every tensor; the library keeps
 * no reference after the call returns.  The library owns a 16-byte error
 * word per device and a private stream-ordered memory pool per device (both
 * created on first use, kept until process exit).  Each call takes
 * B*H*N*d*2 bytes (+ one byte per 128-row V tile) of scratch from that pool
 * on `stream` and returns it in stream order after its kernels: V stored in
 * the operand type of the P V product (fp16 per 128-row tile where V's
 * range allows, else bf16), so the probabilities P are rounded to fp16.
 *
 * Split-KV (head dims up to 128): when the problem has fewer blocks of 256
 * query rows than the GPU has SMs, the call may split each block's key range (the split count that
 * fattn_splitkv_plan(B, H, N, causal, SMs, 0) returns) and merge the
 * splits' partial results with the two-block rule ("understand-
 * flashattention", two-block online-softmax derivation); the scratch then
 * grows by n_splits*B*H*N*(d+1)*4 bytes (fp32 partial O and LSE).  The
 * result is the same function, rounded once to bf16 at the end.
 *
 * Asynchrony: the call validates its arguments synchronously, then enqueues
 * two kernels on `stream` (the V pre-pass and the attention kernel; a third,
 * the split-KV combine, when it splits) and returns without synchronising.
 * Time-outs of the kernel's bounded waits are reported later by
 * fattn_last_error().
 *
 * Returns FATTN_OK, FATTN_ERR_INVALID_ARG (null pointer with B*H*N > 0,
 * negative size, misaligned pointer, host pointer, non-finite or negative
 * scale, sizes beyond int32 index space), FATTN_ERR_UNSUPPORTED (d not a
 * multiple of 8 in [8, 256]) or FATTN_ERR_CUDA (launch failed; no kernel ran).  Argument errors
 * are detected before anything is enqueued.
 */
FATTN_API int fattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
              int d, float scale, int causal, const int32_t* key_len, void* stream);

/*
 * fattn_bwd: gradients of a scalar loss through the forward above.
 *
 * What it computes ("understand-flashattention", section "Attention forward
 * and backward formulas", backward pass steps 1-5; P recomputed from the
 * saved logsumexp as in "recomputing P needs logsumexp"), with
 * S = scale * Q K^T masked as in fattn_fwd and P = exp(S - LSE):
 *     dV = P^T dO,   dP = dO V^T,   dS = P * (dP - rowsum(dO * O)),
 *     dQ = scale * dS K,   dK = scale * dS^T Q.
 * (rowsum(dO * O)_i equals sum_k dP_ik P_ik, the row term of step 3.)
 *
 *   q, k, v  the forward's inputs, bf16 [B, H, N, d] (as for fattn_fwd).
 *   o, lse   the forward's outputs for the same q, k, v, scale, causal and
 *            key_len: bf16 O [B, H, N, d] and fp32 LSE [B, H, N].
 *   dout     dL/dO, bf16 [B, H, N, d].
 *   dq, dk, dv  written: bf16 [B, H, N, d]; each rounded once from fp32.
 *   B, H, N, scale, causal, key_len, stream: as for fattn_fwd.
 *   d        head dim: a multiple of 8 from 8 to 256.  Up to 128 one
 *            kernel forms dK and dV together and another dQ; from 136 the
 *            256-column accumulators leave room for one of them at a time in
 *            tensor memory, so dV, dK and dQ each take a pass of their own
 *            (S recomputed in each, dP in the last two).
 *
 * A query row with no visible key gets dQ = 0; a key visible to no query
 * (key_len) gets dK = dV = 0.  All device pointers 16-byte aligned (lse and
 * key_len 4-byte); dq, dk and dv overlap neither each other nor any input
 * (the kernels after the first start before it ends); the caller owns every
 * tensor.  Each call takes
 * 2 * B*H*ceil(N/128)*128 * 4 bytes of scratch from the library's pool on
 * `stream` (per-row D and LSE in base 2) and returns it in stream order;
 * it enqueues three kernels (four from head dim 136) on `stream` and returns
 * without synchronising.
 *
 * With FATTN_BWD_FUSED=1 in the environment (read once per process), head
 * dims 72..128 run instead a single kernel that also forms dQ, adding each
 * key tile's share into an fp32 buffer with atomic reductions (another
 * B*H*ceil(N/128)*128 * 128 * 4 bytes of scratch; two more kernels zero and
 * convert it).  Its dQ is not bit-reproducible from run to run (the order of
 * the fp32 additions varies); dK and dV are.
 *
 * Returns FATTN_OK, FATTN_ERR_INVALID_ARG, FATTN_ERR_UNSUPPORTED (d not a
 * multiple of 8 in [8, 256]) or FATTN_ERR_CUDA, with argument errors detected before anything
 * is enqueued; time-outs of the kernels' bounded waits are reported by
 * fattn_last_error().
 */
FATTN_API int fattn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                        int causal, const int32_t* key_len, void* stream);

/*
 * fattn_fwd_splitkv: fattn_fwd with the split-KV choice made by the caller.
 *
 *   n_splits  0: the library's choice (exactly fattn_fwd); 1: no split (the
 *             attention kernel writes O and LSE itself); k > 1: min(k,
 *             ceil(N/128)) splits.  The n key tiles of 128 that a block of
 *             256 query rows visits (after the causal and key_len masks) are
 *             cut into near-equal runs, split s taking tiles
 *             [s*n/k, (s+1)*n/k); each split's normalised output and
 *             log-sum-exp over its keys are kept in fp32 and merged by a
 *             combine kernel:
 *                 LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s
 *             over the splits that hold keys of the row.
 *             Above head dim 128 the 256-column kernel works on one 128-row
 *             query tile per CTA and on key tiles of 64: k > 1 gives
 *             min(k, ceil(N/64)) splits, cutting the n key tiles of 64 that
 *             the query tile visits in the same way, merged by the same rule
 *             (a split may hold no visible key for some rows of its tile:
 *             those carry O_s = 0 and LSE_s = -inf and weigh nothing).
 *             Negative: FATTN_ERR_INVALID_ARG.  Head dims as for fattn_fwd
 *             at every split count: multiples of 8 from 8 to 256.
 *
 * Every other argument, the layouts, ownership and errors are those of
 * fattn_fwd (head dims: multiples of 8 from 8 to 256); the scratch is as
 * described there for the split count used.
 */
FATTN_API int fattn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                int N, int d, float scale, int causal, const int32_t* key_len, int n_splits,
                                void* stream);

/*
 * fattn_fwd_host: fattn_fwd on HOST buffers, with the host <-> device copies
 * overlapped with the computation.
 *
 *   q, k, v  host pointers, bf16 [B, H, N, d] (pinned memory lets the copies
 *            run asynchronously; pageable memory works, with copies that
 *            block the calling thread).
 *   o, lse   host pointers, written: bf16 O [B, H, N, d] and fp32 LSE [B, H, N].
 *   key_len  host pointer to int32[B] or NULL.
 *   Other arguments as for fattn_fwd; head dims as for fattn_fwd
 *   (multiples of 8 from 8 to 256).
 *
 * The call takes device buffers for Q, K, V, O, LSE and key_len from the
 * library's pool, cuts the problem into up to eight chunks (ranges of whole
 * batch entries, or of heads within one entry), and enqueues per chunk: the
 * copies of its inputs on a library stream, fattn_fwd on `stream` once they
 * have landed, and the copies of its outputs on a second library stream, so
 * that copies in both directions overlap other chunks' kernels.  Both
 * library streams are joined back into `stream` and the buffers are
 * released there: o and lse hold the results once `stream` has reached this
 * point (synchronise it before reading them).  Results are those of
 * fattn_fwd on the same data (each chunk is a smaller fattn_fwd problem, so
 * the library's split-KV choice may differ per chunk).
 *
 * Returns the codes of fattn_fwd; FATTN_ERR_INVALID_ARG also for a device
 * pointer among the buffers.  Argument errors are detected before anything
 * is enqueued.
 */
FATTN_API int fattn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                             int d, float scale, int causal, const int32_t* key_len, void* stream);

/*
 * fattn_splitkv_plan: the split count the forward uses, computed on the host
 * alone (no GPU, no CUDA call).  n_splits as for fattn_fwd_splitkv: k > 0
 * returns min(k, ceil(N/128)); 0 returns the library's choice: 1 whenever
 * B*H*ceil(N/256) >= num_sms, else the count up to 16 with the least
 * estimated time of the kernel's static schedule over num_sms SMs (each work
 * unit's key tiles plus a fixed per-unit cost, plus the combine pass when
 * split; all N keys assumed visible apart from the causal mask).  Returns 0
 * for B, H, N or num_sms <= 0 or n_splits < 0.
 */
FATTN_API int fattn_splitkv_plan(int B, int H, int N, int causal, int num_sms, int n_splits);

/*
 * fattn_unit_schedule: the order in which the forward's persistent kernel
 * deals its work units to CTAs for a causal call with all keys visible
 * (key_len NULL), no split and head dim up to 128, computed on the host
 * alone (no GPU, no CUDA call).  A work unit is one batch*head and block of
 * 256 query rows; units are numbered heaviest first (unit u is block
 * ceil(N/256) - 1 - u / (B*H) of batch*head u % (B*H)) and taken in rounds of
 * num_ctas = min(units, SMs).  The kernel's default is the snake (CTA c takes
 * unit c of even rounds and num_ctas-1-c of odd ones); where some CTAs'
 * totals then run well above the mean (rounds that do not divide evenly),
 * the library deals each later round's units (the same set as the snake's)
 * so that the totals come out even, the first round as the snake.  Work of
 * a unit: the key tiles its two query tiles visit plus 2.
 *
 *   table     host int[capacity] or NULL: on return table[r*num_ctas + c] is
 *             the unit CTA c takes in round r (units >= B*H*ceil(N/256) are
 *             empty places of the last round).
 *   capacity  entries table can hold.
 *
 * Returns the number of entries (rounds * num_ctas) of the table when the
 * library uses one for this shape (written to table unless table is NULL),
 * 0 when it keeps the snake (or for B, H, N or num_ctas <= 0), -1 when table
 * is not NULL and capacity is below that number (nothing written).
 */
FATTN_API long long fattn_unit_schedule(int B, int H, int N, int num_ctas, int* table, long long capacity);

/*
 * fattn_linear_fwd: causal linear attention, the second workload ("Linear
 * Attention CUDA kernel" page: CausalLinearAttention.forward with its causal
 * dot product and normaliser):
 *     qt_i = phi(q_i), kt_j = phi(k_j) (zero for j >= key_len[b]),
 *     phi(x) = elu(x) + 1,
 *     out_i = (sum_{j <= i} (qt_i . kt_j) v_j) / (qt_i . sum_{j <= i} kt_j + eps).
 *
 *   q, k     device pointers, fp32 [B, H, N, E] contiguous (the page's
 *            kernels take float tensors); 16-byte aligned.
 *   v        device pointer, fp32 [B, H, N, M]; 16-byte aligned.
 *   out      device pointer, fp32 [B, H, N, M], written; 16-byte aligned.
 *   E, M     feature sizes: multiples of 4 from 4 to 128 (others return
 *            FATTN_ERR_UNSUPPORTED).
 *   key_len  device pointer to int32[B] or NULL (all N keys); clamped to
 *            [0, N].  Query rows are never masked.
 *   eps      the normaliser's epsilon (the page's default is 1e-6); finite, >= 0.
 *
 * The rows are cut into chunks of 64: each chunk's share of the running state
 * (sum of kt v^T and of kt) is formed, an exclusive prefix over the chunks
 * gives the state each chunk starts from, and each chunk's outputs combine
 * its own rows with that state -- the same sums as the page's row-by-row
 * recurrence, regrouped.  Takes 2*B*H*ceil(N/64)*(E*M + E)*4 bytes of scratch
 * from the library's pool on `stream`; enqueues three kernels and returns
 * without synchronising.  Returns FATTN_OK, FATTN_ERR_INVALID_ARG,
 * FATTN_ERR_UNSUPPORTED or FATTN_ERR_CUDA (argument errors before anything
 * is enqueued).
 */
FATTN_API int fattn_linear_fwd(const float* q, const float* k, const float* v, float* out, int B, int H, int N, int E,
                               int M, const int32_t* key_len, float eps, void* stream);

/*
 * fattn_set_kernel_events: measurement hook.  While set (non-NULL), every
 * forward or backward call made by the calling thread records `start`
 * (a cudaEvent_t) on its stream just before its dominant kernel and `stop`
 * just after it: the attention kernel of the forward (not the V pre-pass or
 * the split-KV combine; with fattn_fwd_host, around each chunk's, so the last
 * chunk's pair remains), the dK/dV kernel of the backward, and the output
 * kernel of fattn_linear_fwd.  The events
 * belong to the caller and must stay valid while set; cudaEventElapsedTime
 * on them then gives that kernel's device time.  NULL, NULL clears the hook.
 * Always returns FATTN_OK.
 */
FATTN_API int fattn_set_kernel_events(void* start, void* stop);

/*
 * A static, human-readable name for a status code (the non-zero codes of the
 * return-code convention described at fattn_status); never NULL: an unknown
 * code gives "unknown status".
 */
FATTN_API const char* fattn_status_string(int status);

/*
 * Synchronises `stream` and reports whether any fattn kernel on the current
 * device timed out in a bounded wait since the last call: FATTN_ERR_TIMEOUT
 * (and clears the flag), FATTN_ERR_CUDA if the synchronisation failed, else
 * FATTN_OK -- a device-side failure reported as a non-zero code, the same
 * convention as the entry points' own returns (see fattn_status).  It reads
 * the error word of the pool-backed entry points and the one inside the
 * no-alloc array (fattn_fwd_noalloc), each only once that kind of call has
 * set itself up on this device, so it allocates nothing itself.  If detail
 * is not NULL it receives 4 ints: status, role (1 softmax, 2 TMA producer,
 * 3 MMA issuer), barrier id and work unit of the first time-out (the
 * pool-backed word's when both hold one), or zeros.
 */
FATTN_API int fattn_last_error(void* stream, int* detail);

/*
 * Size of the static device scratch behind fattn_fwd_noalloc (64 MiB), plus
 * a 256-byte error word.  Every GPU that loads the library holds this array
 * until the process exits.
 */
#define FATTN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * fattn_fwd_noalloc: fattn_fwd for callers that must not allocate device
 * memory: code that runs where neither cudaMalloc nor a stream-ordered pool
 * may be used, for instance inside a host framework that owns all device
 * memory through its own arena, or a real-time path that must not take the
 * driver's allocation locks.  The pages have no counterpart; this is a
 * property of the library, not of the method.
 *
 * Arguments, layouts, semantics and results are exactly those of fattn_fwd,
 * except that it never splits the key range (split-KV; see fattn_fwd).
 * Instead of per-call scratch from a pool, the call uses one static device
 * array of FATTN_NOALLOC_SCRATCH_BYTES (+256) bytes compiled into the
 * library, and calls no cudaMalloc, cudaFree or allocating routine.
 *
 *   - Limit: the problem must fit the array:
 *       round_up(B*H*N*d*2, 256) + round_up(B*H*round_up(ceil(N/128), 8), 256)
 *         <= 64 MiB
 *     (for example B*H <= 63 at N = 4096, d = 128); larger problems return
 *     FATTN_ERR_UNSUPPORTED before anything is enqueued.  Head dims as for
 *     fattn_fwd: multiples of 8 from 8 to 256.
 *   - Set-up: the first call on a device (with that device current) looks up
 *     the array's device address and sets kernel attributes; make that first
 *     call before any stream capture.
 *   - Sharing: every call uses the same array and it keeps the last call's
 *     contents.  Each call rewrites the V copy and tile modes it reads, so no
 *     data carries over from one call to the next; but calls whose kernels
 *     overlap on the GPU (different streams with no ordering between them)
 *     race on the array and give wrong results.
 *   - Time-outs of the kernel's bounded waits land in an error word after
 *     the array (zero at load).  fattn_last_error() reads and clears it, so
 *     a time-out stays readable until then, even across later calls.
 */
FATTN_API int fattn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                int N, int d, float scale, int causal, const int32_t* key_len, void* stream);

/*
 * Tensor-map cache counters (a diagnostic).  Each call describes its Q, K and
 * V tiles to the GPU's tensor-memory-access (TMA) unit with tensor maps.  The
 * library keeps the last 64 maps it encoded, keyed by everything a map is
 * made from (address, shape, element type, box), and reuses one on an exact
 * key match, so a loop that passes the same buffers encodes nothing after its
 * first call.  Writes the number of reuses and of fresh encodings since the
 * library was loaded (either pointer may be NULL).  Always returns FATTN_OK.
 */
FATTN_API int fattn_tensor_map_stats(long long* hits, long long* misses);

/* Library version, major*10000 + minor*100 + patch. */
FATTN_API int fattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_H_ */
