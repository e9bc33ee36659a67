/*
 * streamkl.h -- C ABI of the GB300 (sm_103a) attention-KL primitive.
 *
 * The operation ("StreamKL: Fast and Memory-Efficient KL Divergence for
 * Boosting Attention Distillation", abstract and gist.science technical
 * summary): for every batch b, head h and query row i,
 *
 *     S_t = scale * Q_t K_t^T (+ causal mask),  P_t = softmax(S_t),  t = 1, 2
 *     KL[b,h,i] = sum_j P1[i,j] * log(P1[i,j] / P2[i,j])
 *
 * with P1 the teacher and P2 the student, computed without ever writing the
 * N_Q x N_K matrices S1, S2, P1, P2 to device memory.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Q1, Q2 are [B, H, N_Q, d] and K1, K2 are [B, H, N_K, d], bf16, dense,
 *   row-major (d contiguous), 16-byte aligned device pointers. d is 64 or 128.
 * - Per-row vectors (kl, lse1, lse2, dkl) are [B, H, N_Q] fp32, dense.
 * - Causal masking is bottom-right aligned: key j is visible to query i iff
 *   j <= i + (N_K - N_Q) (j <= i when N_Q == N_K); it needs N_Q <= N_K.
 * - All pointers are device pointers owned by the caller. The library
 *   allocates no memory, never synchronises, and enqueues all work on
 *   `stream` (a cudaStream_t; NULL means the legacy default stream), so the
 *   calls can be captured into a CUDA graph once their kernels have run
 *   eagerly (the first call sets their shared-memory attributes).
 * - Synchronous argument errors return STREAMKL_ERR_INVALID_ARG or
 *   STREAMKL_ERR_UNSUPPORTED before anything is enqueued; a failed launch
 *   returns STREAMKL_ERR_CUDA. streamkl_last_error() gives the detail.
 * - dev_status is a caller-owned device int the kernels write when a bounded
 *   wait inside them gives up (STREAMKL_ERR_TIMEOUT), when packed sequence
 *   offsets are malformed (STREAMKL_ERR_INVALID_ARG) or, in the debug build,
 *   when a range check fails (STREAMKL_ERR_DEVICE_CHECK); they never clear it.
 *   Clear it before use and read it after synchronising the stream. Results
 *   of a call that set it are undefined.
 */
#ifndef STREAMKL_H_
#define STREAMKL_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  STREAMKL_OK = 0,
  STREAMKL_ERR_INVALID_ARG = 1,
  STREAMKL_ERR_UNSUPPORTED = 2,
  STREAMKL_ERR_CUDA = 3,
  STREAMKL_ERR_TIMEOUT = 4,
  /* Written to dev_status only by the debug build (libstreamkl_debug.so,
   * compiled with STREAMKL_DEVICE_CHECKS): a kernel found an operand of a
   * TMA copy, TMEM access or mbarrier outside its layout, skipped that access
   * and stopped (the first failing source line is printed from the device).
   * The release build never writes it. */
  STREAMKL_ERR_DEVICE_CHECK = 5
} streamkl_status;

/* Human-readable name of a status code (static string). */
const char* streamkl_status_string(streamkl_status s);

/* Detail message of the last failing call on this host thread ("" if none). */
const char* streamkl_last_error(void);

/*
 * Split count the forward pass uses when num_splits == 0 (split-K over the
 * key dimension; gist.science technical summary, section 3 "Variante
 * Split-K": keys are partitioned across thread blocks so that few query rows
 * still fill the GPU). Returns >= 1; 0 on invalid sizes.
 */
int streamkl_choose_splits(int B, int H, int NQ, int NK, int d, int causal);

/*
 * Workspace bytes the forward pass needs with `num_splits` splits (0 = the
 * automatic choice). The split partial states are five fp32 per (split, b, h,
 * row): running maxima, exponential sums and the weighted-logit-difference
 * accumulator. 0 when no split is used.
 */
size_t streamkl_fwd_workspace_size(int B, int H, int NQ, int NK, int d, int causal,
                                   int num_splits);

/*
 * Whether the forward runs as CTA pairs for these sizes: 1 = two CTAs of a
 * thread-block cluster take two query blocks of one (batch, head) slice and
 * compute their score tiles as one tcgen05 MMA with M = 256 (cta_group::2),
 * each CTA loading its own query tile and half of every key tile; 0 = one
 * CTA per query block. Pairs need dense batches without a key split
 * (num_splits as for streamkl_fwd; 0 = automatic) and an even number of
 * 128-row query blocks, and are off unless streamkl_set_fwd_pairs(1) was
 * called (on GB300 they match the one-CTA forward at the 64K causal
 * workload and are slower on smaller ones). Same results either way up to
 * fp32 rounding. Returns -1 on invalid sizes. The paper has no counterpart
 * (it is a scheduling choice of this implementation).
 */
int streamkl_fwd_pairs(int B, int H, int NQ, int NK, int d, int causal, int num_splits);

/*
 * CTA pairs in the forward for the process: 0 = never (default), 1 = when
 * the sizes allow. Returns 0, or -1 for another value.
 */
int streamkl_set_fwd_pairs(int mode);

/*
 * Backward algorithm used for these sizes (gist.science technical summary,
 * section 2, kernel fusion paragraph: a fused kernel with atomic dQ updates,
 * or separate kernels when the atomics contend too much):
 *   0 = separate dK and dQ kernels: each keeps its accumulators on chip for
 *       its whole sweep; no atomics; a workspace only for the dQ kernel's
 *       key split (below);
 *   1 = fused: every (query, key) pair visited once, dK on chip, dQ summed
 *       into an fp32 workspace, then converted to bf16. At most 64 query
 *       rows at d = 128: a persistent kernel over (batch-head, key tile)
 *       items keeping dQ on chip per batch-head; otherwise one CTA per key
 *       tile adding each query block's dQ with TMA bulk reductions (128-row
 *       blocks at d = 64, 64-row steps at d = 128).
 * The automatic choice (from the fused-vs-separate sweep on GB300) is 1 for
 * at most 64 query rows at d = 128; with one gradient set (want_grad1 = 0)
 * for at least 512 query rows at d = 64, and at d = 128 for at least 512
 * query rows without the mask or 1,024 with causal = 1; 0 otherwise.
 * Configuration 2 alone runs 0 except at most 64 query rows at d = 128.
 * Returns -1 on invalid sizes.
 */
int streamkl_bwd_algorithm(int B, int H, int NQ, int NK, int d, int causal, int want_grad1);

/*
 * Process-wide override of that choice: -1 = automatic, 0 = separate,
 * 1 = fused. Its initial value comes from the environment variable
 * STREAMKL_BWD_ALGO=separate|fused (automatic when unset). The workspace
 * size queries follow it; change it only while no other host thread is
 * between a size query and the matching streamkl_bwd call. Returns 0, or -1
 * for an invalid value.
 */
int streamkl_set_bwd_algorithm(int algo);

/*
 * Key split of the separate algorithm's dQ kernel. With few query blocks
 * against many keys (B H ceil(N_Q/128) below 8 per SM) the dQ kernel's
 * key range is cut into splits of 64-key steps, like the forward's split-K
 * (gist.science technical summary, section 3 "Variante Split-K": keys
 * partitioned across thread blocks); each split writes an fp32 partial dQ
 * into the workspace and a
 * combine kernel sums them into the bf16 output. Dense batches only (varlen
 * batches never split).
 *   streamkl_bwd_dq_splits: the split count streamkl_bwd will use for these
 *        sizes (want_grad1 != 0: both gradient sets); -1 on invalid sizes.
 *   streamkl_set_bwd_dq_splits: process-wide override, 0 = automatic, n >= 1
 *        forces n splits (clamped to the number of 64-key steps); same
 *        threading caveat as streamkl_set_bwd_algorithm. Returns 0, or -1
 *        for a negative value.
 */
int streamkl_bwd_dq_splits(int B, int H, int NQ, int NK, int d, int causal, int want_grad1);
int streamkl_set_bwd_dq_splits(int splits);

/*
 * Persistent dK kernel of the separate algorithm for short query sweeps
 * (N_Q <= 384, dense batches, more (key block, batch-head) items than SMs):
 * one CTA per SM takes the items in turn, heavy key blocks first, and loads
 * the next item's key block while the current one finishes, instead of one
 * CTA per key block paying its start and end each time. No counterpart in
 * the paper; same results.
 *   streamkl_bwd_dk_persist: the number of persistent CTAs streamkl_bwd will
 *        launch for these sizes (0: one CTA per key block); -1 on invalid sizes.
 *   streamkl_set_bwd_dk_persist: process-wide override, 0 = automatic,
 *        -1 = never, n >= 1 = always, with n CTAs; same threading caveat as
 *        streamkl_set_bwd_algorithm. Returns 0, or -1 below -1.
 */
int streamkl_bwd_dk_persist(int B, int H, int NQ, int NK, int d, int causal);
int streamkl_set_bwd_dk_persist(int ctas);

/*
 * Workspace bytes the backward pass needs, for one gradient set or, with
 * want_grad1 != 0, both (an upper bound for configuration 2 alone): for the
 * separate-kernel algorithm the fp32 partials of the dQ kernel's key split
 * (0 without a split); for the fused one, one fp32 [B, H, N_Q, d] dQ
 * accumulator per requested gradient set (with want_grad1 = 0 also enough
 * for configuration 2 alone where that runs the separate kernels).
 */
size_t streamkl_bwd_workspace_size(int B, int H, int NQ, int NK, int d, int causal,
                                   int want_grad1);

/* max(forward with automatic splits, backward): one buffer serves both. */
size_t streamkl_workspace_size(int B, int H, int NQ, int NK, int d, int causal,
                               int want_grad1);

/*
 * Forward pass (gist.science technical summary, "Metodologia" section 1:
 * online formulation; section 2 "Estado Guardado": only KL and the two
 * log-sum-exps are saved).
 *   in : q1, k1, q2, k2 (bf16, layout above); scale > 0; causal 0/1;
 *        num_splits: 0 = automatic, >= 1 forces that many key splits
 *        (clamped to the number of key tiles).
 *   out: kl[b,h,i] = KL(P1 || P2) of row i (nats), lse1/lse2[b,h,i] =
 *        log sum_j exp(S_t[i,j]) over the visible keys (fp32).
 *   workspace: device buffer of ws_bytes >= streamkl_fwd_workspace_size(...)
 *        (may be NULL when that is 0); contents need no initialisation.
 */
streamkl_status streamkl_fwd(const void* q1, const void* k1, const void* q2, const void* k2,
                             int B, int H, int NQ, int NK, int d, float scale, int causal,
                             int num_splits, float* kl, float* lse1, float* lse2,
                             void* workspace, size_t ws_bytes, int* dev_status, void* stream);

/*
 * Forward pass that allocates nothing and takes no workspace. The paper has
 * no counterpart; this entry point exists for callers that only hold the
 * input and output buffers handed to them and cannot obtain device memory of
 * their own: a plug-in operator inside another runtime that offers no
 * workspace, or code whose device memory is owned by a host framework's pool,
 * where a cudaMalloc would fail, fragment that pool or stall the device.
 *
 * Same arguments, results and errors as streamkl_fwd, minus the workspace.
 * The split partial states go to a scratch array built into the library:
 * 16 MiB (16777216 bytes) of device memory that every GPU which loads the
 * library keeps until the process exits. A call whose split plan needs more
 * than that (5 floats per split, batch, head and query row, rounded up to 256
 * bytes; see streamkl_fwd_workspace_size) returns STREAMKL_ERR_INVALID_ARG
 * with the sizes in streamkl_last_error(); pass fewer splits or use
 * streamkl_fwd. Calls without splits do not touch the scratch.
 *
 * The first call that uses the scratch on a device looks up its device
 * address (with that device current) and caches it together with the current
 * driver context; make that first call before any stream capture. A call
 * made in another context than the cached one (after cudaDeviceReset, which
 * drops the library's module and the array with it, or with a non-primary
 * context current) looks the address up again, so the first such call should
 * also come before any capture. All calls on a device share the one array and
 * each leaves its partial states in it; nothing there needs clearing because
 * every call writes all the states it reads, but calls whose kernels may
 * overlap on the GPU (different streams, other host threads) race on it and
 * must be ordered by the caller.
 */
streamkl_status streamkl_fwd_noalloc(const void* q1, const void* k1, const void* q2,
                                     const void* k2, int B, int H, int NQ, int NK, int d,
                                     float scale, int causal, int num_splits, float* kl,
                                     float* lse1, float* lse2, int* dev_status, void* stream);

/*
 * Backward pass of L = sum_{b,h,i} dkl[b,h,i] * KL[b,h,i] (gist.science
 * technical summary, section 2: probabilities regenerated tile by tile as
 * P_t = exp(S_t - LSE_t); "Configuracion 1": P1 fixed, gradients to Q2, K2;
 * "Configuracion 2": P2 fixed, gradients to Q1, K1; section 3 "Estabilidad
 * Numerica": log(P1/P2) from logits and saved LSEs).
 *   in : q1, k1, q2, k2, sizes, scale, causal exactly as given to streamkl_fwd;
 *        kl, lse1, lse2 as produced by streamkl_fwd; dkl = upstream gradient
 *        per row (fp32 [B, H, N_Q]).
 *   out: dq2 [B,H,N_Q,d], dk2 [B,H,N_K,d] (bf16) for configuration 1;
 *        dq1, dk1 likewise for configuration 2. Either pair may be NULL to
 *        skip that configuration (both of a pair NULL or neither; at least one
 *        pair is required). Configuration 2 alone runs the separate dK/dQ
 *        kernels, or the fused algorithm's short-sweep kernel where that is
 *        the algorithm chosen (at most 64 query rows at d = 128).
 *   workspace: ws_bytes >= streamkl_bwd_workspace_size(..., want_grad1) (may be
 *        NULL when that is 0); the call clears the part it uses (stream-ordered).
 */
streamkl_status streamkl_bwd(const void* q1, const void* k1, const void* q2, const void* k2,
                             int B, int H, int NQ, int NK, int d, float scale, int causal,
                             const float* kl, const float* lse1, const float* lse2,
                             const float* dkl, void* dq2, void* dk2, void* dq1, void* dk1,
                             void* workspace, size_t ws_bytes, int* dev_status, void* stream);

/*
 * Reverse direction, KL(P2 || P1) per row. The pages define the
 * teacher-first direction KL(P1 || P2) only (gist.science technical summary,
 * "Declaracion del Problema"); the reverse one is the same computation with
 * the two distributions exchanged, so these two calls run the kernels above
 * with the argument slots swapped and add nothing else.
 *   streamkl_fwd_reverse: arguments as for streamkl_fwd; out: kl[b,h,i] =
 *        KL(P2 || P1) of row i, lse1 / lse2 the log-partition of S1 / S2
 *        exactly as from streamkl_fwd.
 *   streamkl_bwd_reverse: gradients of L = sum dkl * KL(P2 || P1), with kl,
 *        lse1, lse2 from streamkl_fwd_reverse. dq2, dk2 get the student's
 *        gradients (P1 fixed), dq1, dk1 the teacher's (P2 fixed); either pair
 *        may be NULL to skip it (at least one pair). ws_bytes >=
 *        streamkl_bwd_workspace_size(..., want_grad1 = both pairs requested).
 * Errors as for streamkl_fwd / streamkl_bwd; a message about a tensor names
 * it by its slot in the exchanged call (q1 for the q2 given here, and so on).
 */
streamkl_status streamkl_fwd_reverse(const void* q1, const void* k1, const void* q2,
                                     const void* k2, int B, int H, int NQ, int NK, int d,
                                     float scale, int causal, int num_splits, float* kl,
                                     float* lse1, float* lse2, void* workspace, size_t ws_bytes,
                                     int* dev_status, void* stream);
streamkl_status streamkl_bwd_reverse(const void* q1, const void* k1, const void* q2,
                                     const void* k2, int B, int H, int NQ, int NK, int d,
                                     float scale, int causal, const float* kl, const float* lse1,
                                     const float* lse2, const float* dkl, void* dq2, void* dk2,
                                     void* dq1, void* dk1, void* workspace, size_t ws_bytes,
                                     int* dev_status, void* stream);

/*
 * Variable-length batches (packed, token-major). The same forward as
 * streamkl_fwd for B independent sequences of different lengths, each with
 * H heads (gist.science technical summary, section 1: the streaming pass is
 * per (batch, head) row and never needs the other sequences' keys).
 *   in : q1, q2 bf16 [total_q, H, d]; k1, k2 bf16 [total_k, H, d] (16-byte
 *        aligned, d contiguous, heads next, then tokens); cu_seqlens_q,
 *        cu_seqlens_k: DEVICE int32 arrays of B+1 offsets, 0 = cu[0] <= cu[1]
 *        <= ... <= cu[B] = total: sequence b owns query rows cu_seqlens_q[b]
 *        .. cu_seqlens_q[b+1] and key rows cu_seqlens_k[b] .. cu_seqlens_k[b+1];
 *        max_seqlen_q / max_seqlen_k: upper bounds on the per-sequence lengths
 *        (they size the grid); causal: per sequence, bottom-right aligned.
 *   out: kl, lse1, lse2 fp32 [total_q, H].
 * No split-K and no workspace. Host-side errors as for streamkl_fwd; the
 * offsets live on the device, so the kernels check them and write
 * STREAMKL_ERR_INVALID_ARG into *dev_status for offsets outside [0, total],
 * a length above its max_seqlen, a sequence with query rows but no key (a
 * softmax over no key is undefined), or a causal sequence with more query
 * rows than keys (its rows of that sequence are then left unwritten). A
 * sequence without query rows contributes nothing.
 */
streamkl_status streamkl_fwd_varlen(const void* q1, const void* k1, const void* q2, const void* k2,
                                    const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                                    int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                                    int d, float scale, int causal, float* kl, float* lse1,
                                    float* lse2, int* dev_status, void* stream);

/*
 * Backward of L = sum dkl * KL for a packed variable-length batch: inputs
 * and sequence offsets as for streamkl_fwd_varlen; kl, lse1, lse2, dkl fp32
 * [total_q, H]; gradients bf16 [total_q, H, d] (dq2, dq1) and [total_k, H, d]
 * (dk2, dk1), either pair NULL to skip that configuration (at least one
 * pair). Always the separate dK/dQ kernels; no workspace. Errors as for
 * streamkl_bwd and streamkl_fwd_varlen. The dK rows of a sequence without
 * query rows are zero (no query sees those keys).
 */
streamkl_status streamkl_bwd_varlen(const void* q1, const void* k1, const void* q2, const void* k2,
                                    const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                                    int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                                    int d, float scale, int causal, const float* kl,
                                    const float* lse1, const float* lse2, const float* dkl,
                                    void* dq2, void* dk2, void* dq1, void* dk1, int* dev_status,
                                    void* stream);

/*
 * Self-test of the bounded-wait path: launches one tiny kernel that waits on
 * a barrier nothing arrives on, for timeout_us microseconds, then records
 * STREAMKL_ERR_TIMEOUT in *dev_status and returns. No other state is touched.
 * The paper has no counterpart; it exists so that the failure path of the
 * kernels' waits can be tested without hanging a GPU.
 */
streamkl_status streamkl_selftest_wait_timeout(int* dev_status, unsigned timeout_us,
                                               void* stream);

/*
 * Self-test of the debug build's range checks: launches one tiny kernel that
 * checks a TMEM column range lying past any allocation (no TMEM is allocated
 * and nothing is accessed). In the debug build (libstreamkl_debug.so) the
 * check fails and records STREAMKL_ERR_DEVICE_CHECK in *dev_status; in the
 * release build the checks are compiled out and *dev_status is left as it
 * was. The paper has no counterpart; it exists so that the report path of
 * the checks can be tested without a faulty access.
 */
streamkl_status streamkl_selftest_device_check(int* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* STREAMKL_H_ */
