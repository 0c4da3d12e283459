/*
 * dspark.h -- C ABI of the DSpark per-round hot path on one GB300 (sm_103a).
 *
 * One decoding round of DSpark speculative decoding, as the pages describe it
 * ("DSpark: Aceleração da inferência de LLM com speculative decoding [pdf]",
 * GeekNews, section "Arquitetura - dois componentes complementares"):
 *   1. draft   -- sequential Markov-head stage over the parallel backbone's
 *                 base logits: for k = 1..gamma, bias = W1[prev] . W2 is added
 *                 to base logits of position k, a tempered softmax over the
 *                 whole vocabulary is formed and token k is sampled;
 *   2. schedule-- confidence-scheduled verification lengths: prefix-survival
 *                 products, a global descending merge of all R x gamma
 *                 candidates, greedy admission against a throughput table
 *                 with early stop ("Verificação com agendamento por
 *                 confiança", "Hardware-Aware Prefix Scheduler"), or the
 *                 production lagged variant ("Aplicação prática do scheduler");
 *   3. verify  -- lossless speculative sampling: accept x_k with probability
 *                 min(1, p/q), resample the first rejection from
 *                 normalize(max(0, p - q)), or draw a bonus token when every
 *                 scheduled token is accepted ("Definição do problema").
 * The parallel backbone, confidence head and target forward pass are outside
 * this library: their outputs (base logits, confidences, target logits) are
 * inputs.
 *
 * Conventions (all entry points):
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, row-major,
 *     densely packed, at least 16-byte aligned. The library allocates no
 *     memory and keeps no pointer after a call returns.
 *   - `dtype` selects the element type of base logits, target logits, W1 and
 *     W2: DSPARK_BF16 (bf16 bit patterns) or DSPARK_FP32. Everything else is
 *     int32 / float32 / float64 as declared.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream). Only host-checkable argument errors are returned
 *     synchronously; nothing is launched in that case.
 *   - Errors found on the device (non-finite inputs, a token id out of range,
 *     a bounded wait that ran out) set a sticky status word inside the
 *     workspace; read it with dspark_device_status(). Nothing aborts, traps
 *     or prints.
 *   - Randomness: one uniform per decision, U(seed, r, k, purpose), from
 *     Philox4x64-10 (Salmon et al., SC'11) with key (seed, 0x44535041524B0000)
 *     and counter (r, k, purpose, 0), u = (2*(w0 >> 12) + 1) * 2^-53;
 *     purposes DRAFT=0 (r, k), ACCEPT=1 (r, k), RESID=2 (r, j), BONUS=3
 *     (r, L_r + 1). Same inputs and seed give bit-identical outputs.
 *   - Sampling is inverse-CDF in vocabulary order: the smallest v with
 *     u * Z < sum_{i<=v} w_i. Temperature 0 is greedy (argmax, lowest index on
 *     ties) for both the draft and the target.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st* dspark_stream_t;

typedef enum {
  DSPARK_OK = 0,
  DSPARK_ERR_INVALID_ARG = 1, /* bad shape, null pointer, unsupported combination */
  DSPARK_ERR_NONFINITE = 2,   /* NaN/Inf confidence or cost-table entry (device) */
  DSPARK_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or too small */
  DSPARK_ERR_CUDA = 4,        /* a CUDA runtime call failed */
  DSPARK_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out (device) */
  DSPARK_ERR_RANGE = 6,       /* a token id outside [0, V) was read (device) */
  DSPARK_ERR_TOO_LARGE = 7    /* problem exceeds the fixed scratch of dspark_schedule_static */
} dspark_status;

typedef enum { DSPARK_FP32 = 0, DSPARK_BF16 = 1 } dspark_dtype;

typedef enum {
  DSPARK_SCHED_CAUSAL = 0, /* greedy admission with early stop */
  DSPARK_SCHED_LAGGED = 1, /* K from lagged confidences (argmax, no early stop), top K of current */
  DSPARK_SCHED_ALL = 2     /* verify every drafted position (scheduler off) */
} dspark_sched_mode;

/* Bytes of device workspace every entry point below needs for these sizes.
 * One workspace may be reused by consecutive calls on one stream; calls that
 * may overlap on the GPU need separate workspaces. Alignment: 256 bytes. */
size_t dspark_workspace_bytes(int32_t R, int32_t gamma, int32_t V, int32_t rank,
                              int32_t dtype, int32_t n_table);

/* Clears the whole workspace (async on `stream`): the sticky status word and
 * the library's internal completion counters, which every call leaves at zero
 * again. Call once after allocating a workspace; every entry point below
 * leaves earlier errors in place (sticky) until this is called again. */
dspark_status dspark_workspace_init(void* workspace, size_t workspace_bytes,
                                    dspark_stream_t stream);

/*
 * Sequential drafting stage with the low-rank Markov head (GeekNews page,
 * "Geração semiautorregressiva": "Etapa sequencial" and "Head de Markov";
 * the anchor is the first prediction position, "Etapa paralela").
 *
 *   base_logits  [R, gamma, V] dtype   row k-1 = base logits of block position k
 *   anchor       [R] int32             the target's last sampled token
 *   W1           [V, rank] dtype       Markov factor: bias(prev) = W1[prev, :] . W2
 *   W2           [rank, V] dtype
 *   temperature  >= 0; softmax((base + bias) / T); 0 = greedy
 *   draft_tokens [R, gamma] int32 out  x_{r,k}; prev of position k>1 is x_{r,k-1}
 *   q_tok        [R, gamma] float out  Q_k(x_k), the draft probability of x_k
 *   q_stats      [R, gamma, 2] float out  (M, Z): Q_k(v) = 2^((l_v - M) log2(e)/T) / Z
 *                                         (greedy: (max l, 1))
 * Requirements: R >= 1, gamma >= 1, V >= 1, rank >= 1. The tensor-core path
 * (one cooperative launch for all gamma steps) is used when dtype = BF16,
 * rank % 64 == 0, rank <= 256, V % 8 == 0, V >= 64, base_logits, W1 and W2
 * are 16-byte aligned and the device supports cooperative launch; other
 * shapes run on CUDA cores with the same results up to rounding.
 */
dspark_status dspark_draft_sequential(int32_t R, int32_t gamma, int32_t V, int32_t rank,
                                      int32_t dtype, const void* base_logits,
                                      const int32_t* anchor, const void* W1, const void* W2,
                                      float temperature, uint64_t seed,
                                      int32_t* draft_tokens, float* q_tok, float* q_stats,
                                      void* workspace, size_t workspace_bytes,
                                      dspark_stream_t stream);

/*
 * Hardware-aware prefix scheduler (GeekNews page, "Verificação com
 * agendamento por confiança": "Hardware-Aware Prefix Scheduler" and
 * "Calibração posterior"; production variant in "Aplicação prática do
 * scheduler").
 *
 *   conf        [R, gamma] float   c_{r,k}, clamped to [0, 1]; non-finite -> DSPARK_ERR_NONFINITE
 *   conf_lagged [R, gamma] float   confidences of two rounds earlier (LAGGED only, else NULL)
 *   sps_table   [n_table] float    SPS(B) at B = i + 1 batch tokens (finite)
 *   mode        dspark_sched_mode
 *   sched_len   [R] int32 out      L_r, the verified prefix length of request r
 *   K           [1] int32 out      admitted candidates (sum of L_r)
 *   tau_theta   [2] double out     expected tokens tau and Theta = tau * SPS(R + K)
 * Arithmetic (fixed so every implementation agrees bit for bit):
 *   a_{r,j} = fl32(a_{r,j-1} * c_{r,j}), a_{r,0} = 1; candidates ordered by a
 *   descending, ties by flat index r*gamma + j - 1; after i admissions
 *   tau_i = R + S_i * 2^-40 with S_i the sum of floor(a * 2^40 + 1/2),
 *   Theta_i = tau_i * SPS[R + i - 1] (float64). CAUSAL admits candidate i+1
 *   while R + i + 1 <= n_table and Theta_{i+1} >= Theta_i. LAGGED takes K as
 *   the smallest argmax of Theta_i (lagged confidences), i <= min(R gamma,
 *   n_table - R), then admits the top K current candidates. R > n_table admits
 *   nothing (K = 0, Theta reported 0). ALL sets L_r = gamma.
 * Requirements: R * gamma <= 65536.
 */
dspark_status dspark_schedule(int32_t R, int32_t gamma, const float* conf,
                              const float* conf_lagged, const float* sps_table,
                              int32_t n_table, int32_t mode, int32_t* sched_len,
                              int32_t* K, double* tau_theta, void* workspace,
                              size_t workspace_bytes, dspark_stream_t stream);

/*
 * dspark_schedule without a workspace, for callers that cannot allocate device
 * memory. The pages describe no such entry point: it exists for
 * callers that run inside an engine which owns all device memory (a reserved
 * pool sized for weights and KV cache, with no allocator reachable from the
 * decode step), or that must not risk an allocation failing or fragmenting
 * memory in the middle of serving. It computes exactly what dspark_schedule
 * computes, bit for bit, with the same arguments except the workspace.
 *
 * Scratch: a fixed array inside the library (393,472 bytes on every GPU that
 * loads the library, kept until the process exits), so R * gamma must not
 * exceed 16384; larger problems return DSPARK_ERR_TOO_LARGE and launch
 * nothing. The call allocates nothing and calls no allocating routine.
 *   device_status [1] uint32 out, device memory, or NULL: receives this call's
 *                 device-side status (DSPARK_OK or DSPARK_ERR_NONFINITE), the
 *                 counterpart of dspark_device_status for this entry point.
 * The first call on each device looks up the scratch's device address (with
 * that device current) and caches it; make that first call before any stream
 * capture. Every call on a device shares the one array, which keeps the last
 * call's contents: calls that may overlap on the GPU (different streams
 * without ordering between them) race on it and must not be issued.
 */
dspark_status dspark_schedule_static(int32_t R, int32_t gamma, const float* conf,
                                     const float* conf_lagged, const float* sps_table,
                                     int32_t n_table, int32_t mode, int32_t* sched_len,
                                     int32_t* K, double* tau_theta, uint32_t* device_status,
                                     dspark_stream_t stream);

/*
 * Lossless speculative-sampling verification (GeekNews page, "Definição do
 * problema" and the decoding-cycle paragraph: E, F accepted, G rejected and
 * replaced by a corrected G*).
 *
 *   target_logits [R, gamma+1, V] dtype  row k = target logits after the anchor and k draft tokens
 *   base_logits, anchor, W1, W2           as for drafting (the draft distribution Q_j of the first
 *                                          rejected position is recomputed for the residual)
 *   draft_tokens, q_tok, q_stats          outputs of dspark_draft_sequential
 *   sched_len     [R] int32               L_r from dspark_schedule (0..gamma)
 *   out_tokens    [R, gamma+1] int32 out  x_1..x_{A_r} then the corrected/bonus token; -1 after
 *   accepted_len  [R] int32 out           A_r in [0, L_r]
 *   p_tok         [R, gamma] float out    P_{k-1}(x_k) for k <= L_r, 0 beyond
 * Rule: accept x_k iff u_ACCEPT < p/q (strict); at the first rejection j draw
 * from normalize(max(0, P_{j-1} - Q_j)) (from P_{j-1} if that has no mass);
 * if all L_r are accepted draw the bonus from P_{L_r}.
 */
dspark_status dspark_verify(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                            const void* target_logits, const void* base_logits,
                            const int32_t* anchor, const void* W1, const void* W2,
                            const int32_t* draft_tokens, const float* q_tok,
                            const float* q_stats, const int32_t* sched_len,
                            float temperature, uint64_t seed, int32_t* out_tokens,
                            int32_t* accepted_len, float* p_tok, void* workspace,
                            size_t workspace_bytes, dspark_stream_t stream);

/*
 * Acceptance labels of the confidence head (GeekNews page, "Confidence head"
 * and "Calibração posterior": the head predicts the probability that each
 * drafted token passes verification). For every request r and position
 * k = 1..gamma,
 *   labels[r, k-1] = 1 - (1/2) sum_v |Q_k(v) - P_{k-1}(v)|  (one minus the
 *                    total variation distance = sum_v min(P_{k-1}, Q_k)),
 * Q_k the drafter's distribution at position k given the drafted tokens
 * before it, P_{k-1} the target's row k-1, both at `temperature`; for
 * temperature 0 both are one-hot and the label is 1 where the drafted token
 * is the target row's argmax (lowest index on ties), else 0.
 *
 *   target_logits, base_logits, anchor, W1, W2   as for dspark_verify
 *   draft_tokens [R, gamma] int32, q_stats [R, gamma, 2]  outputs of dspark_draft_sequential
 *   labels       [R, gamma] float out
 * Every position is labelled, whatever a scheduler would admit. Sampled mode
 * (temperature > 0) needs the tensor-core shape: bf16 inputs, rank a multiple
 * of 64 up to 256, V a multiple of 8 and at least 64, 16-byte aligned
 * pointers, and cooperative launch; otherwise it returns
 * DSPARK_ERR_INVALID_ARG and enqueues nothing it would need. Uses the same
 * workspace as the other calls.
 */
dspark_status dspark_acceptance_labels(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                                       const void* target_logits, const void* base_logits,
                                       const int32_t* anchor, const void* W1, const void* W2,
                                       const int32_t* draft_tokens, const float* q_stats, float temperature,
                                       float* labels, void* workspace, size_t workspace_bytes,
                                       dspark_stream_t stream);

/*
 * One whole round: draft -> schedule -> verify on one stream, with no host
 * synchronisation in between (the scheduled lengths stay on the device).
 * Arguments are the union of the three calls above; the intermediate outputs
 * (draft_tokens, q_tok, q_stats, sched_len, K, tau_theta) are written too,
 * and every output equals, bit for bit, what the three calls give in turn.
 * On the tensor-core path the drafting launch itself computes the schedule
 * and, outside ALL mode, the target row statistics and acceptance chains
 * (the target tensor 16-byte aligned), leaving one launch for the residual
 * or bonus draw.
 */
dspark_status dspark_round(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                           const void* base_logits, const void* target_logits,
                           const int32_t* anchor, const void* W1, const void* W2,
                           const float* conf, const float* conf_lagged,
                           const float* sps_table, int32_t n_table, int32_t mode,
                           float temperature, uint64_t seed, int32_t* draft_tokens,
                           float* q_tok, float* q_stats, int32_t* sched_len, int32_t* K,
                           double* tau_theta, int32_t* out_tokens, int32_t* accepted_len,
                           float* p_tok, void* workspace, size_t workspace_bytes,
                           dspark_stream_t stream);

/*
 * Base logits from the parallel backbone's hidden states (GeekNews page,
 * "Etapa paralela": one backbone pass over the block gives hidden states and
 * base logits; "Comunicação de estados ocultos": only the hidden state before
 * the LM head has to travel, and the LM head runs where the logits are used).
 *
 *   hidden   [M, d] bf16      final hidden states (M = R * gamma block positions)
 *   lm_head  [d, V] bf16      the (shared) LM head
 *   logits   [M, V] bf16 out  bf16(hidden . lm_head): float32 accumulation on
 *                             the tensor cores, one rounding to nearest (ties to
 *                             even); [R, gamma, V] for dspark_draft_sequential
 * Requirements: M >= 1, d >= 64 and d % 8 == 0, V >= 64 and V % 8 == 0, the
 * three tensors 16-byte aligned. `workspace` (at least 256 bytes, 256-byte
 * aligned; any DSpark workspace) receives the device status word.
 */
dspark_status dspark_lm_head(int32_t M, int32_t d, int32_t V, const void* hidden,
                             const void* lm_head, void* logits, void* workspace,
                             size_t workspace_bytes, dspark_stream_t stream);

/*
 * Recurrent (gated) sequential head (GeekNews page, "Geração
 * semiautorregressiva": "Head RNN", the variant that keeps a recurrent state
 * of the whole prefix drafted in the block, updated through gates). The pages
 * give no equations; the reading implemented is a minimal gated recurrence
 * over the head's input, the previous token prev_k (the anchor at k = 1,
 * else x_{k-1}):
 *   s_0 = 0,  s_k = (1 - gate[prev_k]) * s_{k-1} + gate[prev_k] * W1[prev_k]
 * elementwise in float32 (each product and sum rounded once), and
 *   bias_k = bf16(s_k) . W2      (s_k rounded to bf16, ties to even).
 * gate [V, rank] (dtype, values in [0, 1]) is the update gate of each token,
 * tabulated once (a gate driven by a one-hot input is a row lookup). Gate
 * values 1 give the Markov head exactly; 0 gives bias 0.
 *
 * dspark_draft_sequential_gated, dspark_verify_gated and dspark_round_gated
 * take the arguments of dspark_draft_sequential, dspark_verify and
 * dspark_round plus `gate` (after W1), and write the same outputs;
 * verification recomputes the residual's Q_j from the state replayed over the
 * anchor and the accepted tokens. They run on the tensor-core path only:
 * dtype BF16, rank a multiple of 64 up to 256, V a multiple of 8 and at least
 * 64, every tensor 16-byte aligned, and a device with cooperative launch;
 * otherwise they return DSPARK_ERR_INVALID_ARG and enqueue nothing. The
 * workspace is the same as for the Markov head (it holds each request's
 * float32 state between steps).
 */
dspark_status dspark_draft_sequential_gated(int32_t R, int32_t gamma, int32_t V, int32_t rank,
                                            int32_t dtype, const void* base_logits,
                                            const int32_t* anchor, const void* W1, const void* gate,
                                            const void* W2, float temperature, uint64_t seed,
                                            int32_t* draft_tokens, float* q_tok, float* q_stats,
                                            void* workspace, size_t workspace_bytes,
                                            dspark_stream_t stream);
dspark_status dspark_verify_gated(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                                  const void* target_logits, const void* base_logits,
                                  const int32_t* anchor, const void* W1, const void* gate,
                                  const void* W2, const int32_t* draft_tokens, const float* q_tok,
                                  const float* q_stats, const int32_t* sched_len,
                                  float temperature, uint64_t seed, int32_t* out_tokens,
                                  int32_t* accepted_len, float* p_tok, void* workspace,
                                  size_t workspace_bytes, dspark_stream_t stream);
dspark_status dspark_round_gated(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                                 const void* base_logits, const void* target_logits,
                                 const int32_t* anchor, const void* W1, const void* gate,
                                 const void* W2, const float* conf, const float* conf_lagged,
                                 const float* sps_table, int32_t n_table, int32_t mode,
                                 float temperature, uint64_t seed, int32_t* draft_tokens,
                                 float* q_tok, float* q_stats, int32_t* sched_len, int32_t* K,
                                 double* tau_theta, int32_t* out_tokens, int32_t* accepted_len,
                                 float* p_tok, void* workspace, size_t workspace_bytes,
                                 dspark_stream_t stream);

/*
 * Sequential Temperature Scaling of the confidence head (GeekNews page,
 * "Calibração posterior — Sequential Temperature Scaling (STS)").
 *
 * dspark_sts_fit: on a held-out set of N blocks with confidences
 * conf [N, gamma] float and A = accepted [N] int32 (leading drafted tokens that
 * passed verification, every position verified), finds per-position
 * temperatures left to right: T_k is the first value of grid [n_grid] that
 * minimises the expected calibration error (n_bins equal-width bins on [0, 1],
 * sum over bins of |sum of predictions - sum of outcomes| / N) of the
 * calibrated survival prod_{i<=k} sigmoid(logit(c_i) / T_i) against the outcome
 * [A >= k], T_1..T_{k-1} fixed. Confidences are clipped to [1e-6, 1 - 1e-6]
 * before the logit. Writes temperature [gamma] and, unless NULL, the ECE curve
 * ece [gamma, n_grid]. n_bins is at most 64. scratch: device memory of
 * dspark_sts_scratch_bytes(...) bytes, 256-byte aligned, owned by the caller;
 * a non-finite confidence sets DSPARK_ERR_NONFINITE in it, read by
 * dspark_sts_status (which synchronises the stream).
 *
 * dspark_sts_apply: conf_out[r, k] = sigmoid(logit(clip(conf[r, k])) / T_k),
 * the calibrated confidences to pass to dspark_schedule (non-finite inputs
 * are passed through, for the scheduler to report).
 */
size_t dspark_sts_scratch_bytes(int32_t N, int32_t gamma, int32_t n_grid, int32_t n_bins);
dspark_status dspark_sts_fit(int32_t N, int32_t gamma, const float* conf, const int32_t* accepted,
                             int32_t n_grid, const float* grid, int32_t n_bins, float* temperature, float* ece,
                             void* scratch, size_t scratch_bytes, dspark_stream_t stream);
dspark_status dspark_sts_status(const void* scratch, dspark_stream_t stream);
dspark_status dspark_sts_apply(int32_t R, int32_t gamma, const float* conf, const float* temperature,
                               float* conf_out, dspark_stream_t stream);

/* Synchronises `stream`, then returns the workspace's sticky device status
 * (DSPARK_OK if no device-side error was recorded). */
dspark_status dspark_device_status(const void* workspace, dspark_stream_t stream);

/*
 * Host-to-device copy of the target-logit rows verification reads: rows
 * 0..sched_len[r] of every request r (dspark_verify reads no other row), one
 * cudaMemcpyAsync per request on `stream`. host_target [R, gamma+1, V] dtype
 * is HOST memory (pinned for the copies to be asynchronous), device_target
 * the device tensor of the same shape (rows past sched_len[r] are left as
 * they are), host_sched_len [R] int32 a HOST array (for instance the lengths
 * of dspark_schedule copied back). For a serving loop that receives target
 * logits from the host: the bytes sent follow the schedule, as the target's
 * verification cost does.
 */
dspark_status dspark_copy_scheduled_rows(int32_t R, int32_t gamma, int32_t V, int32_t dtype,
                                         const void* host_target, void* device_target,
                                         const int32_t* host_sched_len, dspark_stream_t stream);

/*
 * Self-test of the bounded device waits: runs one wait of the kinds the
 * kernels use on a condition nothing meets -- `which` 0 = the grid barrier,
 * 1 = an mbarrier wait, 2 = the poll on a counter another CTA of the launch
 * advances (the drafting launch's row list and per-request completion) -- so
 * that it gives up after its iteration limit
 * (about a second), records DSPARK_ERR_TIMEOUT in the workspace's status word
 * (read with dspark_device_status) and returns. Nothing traps; later calls on
 * the same context work. Uses word 16 of the workspace's status block.
 */
dspark_status dspark_wait_selftest(int32_t which, void* workspace, size_t workspace_bytes,
                                   dspark_stream_t stream);

/* Static, human-readable name of a status code. */
const char* dspark_status_string(dspark_status status);

/* Number of kernel launches the most recent call of each entry point made on
 * this thread (for launch accounting in benchmarks). */
int32_t dspark_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
