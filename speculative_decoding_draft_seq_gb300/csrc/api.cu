// C-ABI entry points of the DSpark library (declared in include/dspark.h):
// host-side argument checks, workspace sizing and kernel dispatch. Every
// launch goes to the caller's stream; nothing here synchronises except
// dspark_device_status().
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dspark {
bool draft_tc_eligible(const DraftArgs& a);
cudaError_t launch_draft_cuda_core(const DraftArgs& a, cudaStream_t s, int& launches);
cudaError_t launch_draft_persistent(const DraftArgs& a, cudaStream_t s, int& launches, bool& taken);

// bf16 shapes the tensor cores take run as one persistent cooperative launch
// (all steps); every other shape runs on CUDA cores.
cudaError_t launch_draft(const DraftArgs& a, cudaStream_t s, int& launches) {
  bool taken = false;
  cudaError_t e = launch_draft_persistent(a, s, launches, taken);
  if (taken || e != cudaSuccess) return e;
  return launch_draft_cuda_core(a, s, launches);
}
}  // namespace dspark

using namespace dspark;

static thread_local int g_last_launches = 0;

static bool dims_ok(int R, int gamma, int V, int rank, int dtype) {
  return R >= 1 && gamma >= 1 && gamma < 65535 && V >= 1 && rank >= 1 &&
         (dtype == DSPARK_FP32 || dtype == DSPARK_BF16) && (long long)R * (long long)gamma <= 65536 &&
         V <= (1 << 30) && (long long)rank * V <= (1ll << 40);
}

static bool ws_ok(const void* ws, size_t bytes, size_t need) {
  return ws != nullptr && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0 && bytes >= need;
}

static dspark_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA; }

extern "C" {

size_t dspark_workspace_bytes(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                              int32_t n_table) {
  (void)rank; (void)dtype; (void)n_table;
  if (R < 1 || gamma < 1 || V < 1) return 0;
  const size_t a = ws_layout(R, gamma, V).total;
  const size_t b = ws_layout(R, gamma, 1).total;
  return a > b ? a : b;
}

dspark_status dspark_workspace_init(void* workspace, size_t workspace_bytes, dspark_stream_t stream) {
  if (!ws_ok(workspace, workspace_bytes, 256)) return DSPARK_ERR_WORKSPACE;
  // the whole workspace: the status word and every completion counter start at zero
  return cuda_status(cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream));
}

}  // extern "C"

// Drafting with the Markov head (gate == nullptr) or the gated head.
static dspark_status draft_entry(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                                 const void* base_logits, const int32_t* anchor, const void* W1, const void* gate,
                                 const void* W2, float temperature, uint64_t seed, int32_t* draft_tokens,
                                 float* q_tok, float* q_stats, void* workspace, size_t workspace_bytes,
                                 dspark_stream_t stream) {
  g_last_launches = 0;
  if (!dims_ok(R, gamma, V, rank, dtype) || !(temperature >= 0.f) || !isfinite(temperature))
    return DSPARK_ERR_INVALID_ARG;
  if (!base_logits || !anchor || !W1 || !W2 || !draft_tokens || !q_tok || !q_stats)
    return DSPARK_ERR_INVALID_ARG;
  if (!ws_ok(workspace, workspace_bytes, ws_layout(R, gamma, V).total)) return DSPARK_ERR_WORKSPACE;
  DraftArgs a{R, gamma, V, rank, dtype, base_logits, anchor, W1, W2, temperature, seed,
              draft_tokens, q_tok, q_stats, workspace, gate};
  int n = 0;
  cudaError_t e;
  if (gate) {  // the persistent tensor-core sweep only: decide before enqueueing anything
    if (!gated_supported(a)) return DSPARK_ERR_INVALID_ARG;
    bool taken = false;
    e = launch_draft_persistent(a, (cudaStream_t)stream, n, taken);
    if (e == cudaSuccess && !taken) return DSPARK_ERR_INVALID_ARG;
  } else {
    e = launch_draft(a, (cudaStream_t)stream, n);
  }
  g_last_launches = n;
  return cuda_status(e);
}

extern "C" {

dspark_status dspark_draft_sequential(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                                      const void* base_logits, const int32_t* anchor, const void* W1,
                                      const void* W2, float temperature, uint64_t seed,
                                      int32_t* draft_tokens, float* q_tok, float* q_stats,
                                      void* workspace, size_t workspace_bytes, dspark_stream_t stream) {
  return draft_entry(R, gamma, V, rank, dtype, base_logits, anchor, W1, nullptr, W2, temperature, seed,
                     draft_tokens, q_tok, q_stats, workspace, workspace_bytes, stream);
}

dspark_status dspark_draft_sequential_gated(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                                            const void* base_logits, const int32_t* anchor, const void* W1,
                                            const void* gate, const void* W2, float temperature, uint64_t seed,
                                            int32_t* draft_tokens, float* q_tok, float* q_stats,
                                            void* workspace, size_t workspace_bytes, dspark_stream_t stream) {
  if (!gate) return DSPARK_ERR_INVALID_ARG;
  return draft_entry(R, gamma, V, rank, dtype, base_logits, anchor, W1, gate, W2, temperature, seed,
                     draft_tokens, q_tok, q_stats, workspace, workspace_bytes, stream);
}

dspark_status dspark_schedule(int32_t R, int32_t gamma, const float* conf, const float* conf_lagged,
                              const float* sps_table, int32_t n_table, int32_t mode, int32_t* sched_len,
                              int32_t* K, double* tau_theta, void* workspace, size_t workspace_bytes,
                              dspark_stream_t stream) {
  g_last_launches = 0;
  if (R < 1 || gamma < 1 || gamma >= 65535 || (long long)R * gamma > 65536 || n_table < 0)
    return DSPARK_ERR_INVALID_ARG;
  if (mode != DSPARK_SCHED_CAUSAL && mode != DSPARK_SCHED_LAGGED && mode != DSPARK_SCHED_ALL)
    return DSPARK_ERR_INVALID_ARG;
  if (!conf || !sched_len || !K || !tau_theta || (n_table > 0 && !sps_table)) return DSPARK_ERR_INVALID_ARG;
  if (mode == DSPARK_SCHED_LAGGED && !conf_lagged) return DSPARK_ERR_INVALID_ARG;
  if (!ws_ok(workspace, workspace_bytes, ws_layout(R, gamma, 1).total)) return DSPARK_ERR_WORKSPACE;
  ScheduleArgs a{R, gamma, conf, conf_lagged, sps_table, n_table, mode, sched_len, K, tau_theta, workspace};
  int n = 0;
  cudaError_t e = launch_schedule(a, (cudaStream_t)stream, n);
  g_last_launches = n;
  return cuda_status(e);
}

}  // extern "C"

// The gated head's support check for verification: its residual draw runs
// only on the tensor-core sweep, which reads the target rows with 16-byte
// copies, so the drafting conditions plus an aligned target tensor.
static bool gated_verify_supported(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                                   const void* target_logits, const void* base_logits, const int32_t* anchor,
                                   const void* W1, const void* gate, const void* W2, void* workspace) {
  DraftArgs d{R, gamma, V, rank, dtype, base_logits, anchor, W1, W2, 1.f, 0, nullptr, nullptr, nullptr,
              workspace, gate};
  return gated_supported(d) && (reinterpret_cast<uintptr_t>(target_logits) & 15) == 0;
}

static dspark_status verify_entry(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                                  const void* target_logits, const void* base_logits, const int32_t* anchor,
                                  const void* W1, const void* gate, const void* W2, const int32_t* draft_tokens,
                                  const float* q_tok, const float* q_stats, const int32_t* sched_len,
                                  float temperature, uint64_t seed, int32_t* out_tokens, int32_t* accepted_len,
                                  float* p_tok, void* workspace, size_t workspace_bytes, dspark_stream_t stream) {
  g_last_launches = 0;
  if (!dims_ok(R, gamma, V, rank, dtype) || !(temperature >= 0.f) || !isfinite(temperature))
    return DSPARK_ERR_INVALID_ARG;
  if (!target_logits || !base_logits || !anchor || !W1 || !W2 || !draft_tokens || !q_tok || !q_stats ||
      !sched_len || !out_tokens || !accepted_len || !p_tok)
    return DSPARK_ERR_INVALID_ARG;
  if (!ws_ok(workspace, workspace_bytes, ws_layout(R, gamma, V).total)) return DSPARK_ERR_WORKSPACE;
  if (gate && !gated_verify_supported(R, gamma, V, rank, dtype, target_logits, base_logits, anchor, W1, gate, W2,
                                      workspace))
    return DSPARK_ERR_INVALID_ARG;
  VerifyArgs a{R, gamma, V, rank, dtype, target_logits, base_logits, anchor, W1, W2, draft_tokens,
               q_tok, q_stats, sched_len, temperature, seed, out_tokens, accepted_len, p_tok, workspace, gate};
  int n = 0;
  cudaError_t e = launch_verify(a, (cudaStream_t)stream, n);
  g_last_launches = n;
  return cuda_status(e);
}

extern "C" {

dspark_status dspark_verify(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                            const void* target_logits, const void* base_logits, const int32_t* anchor,
                            const void* W1, const void* W2, const int32_t* draft_tokens,
                            const float* q_tok, const float* q_stats, const int32_t* sched_len,
                            float temperature, uint64_t seed, int32_t* out_tokens, int32_t* accepted_len,
                            float* p_tok, void* workspace, size_t workspace_bytes, dspark_stream_t stream) {
  return verify_entry(R, gamma, V, rank, dtype, target_logits, base_logits, anchor, W1, nullptr, W2,
                      draft_tokens, q_tok, q_stats, sched_len, temperature, seed, out_tokens, accepted_len, p_tok,
                      workspace, workspace_bytes, stream);
}

dspark_status dspark_verify_gated(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                                  const void* target_logits, const void* base_logits, const int32_t* anchor,
                                  const void* W1, const void* gate, const void* W2, const int32_t* draft_tokens,
                                  const float* q_tok, const float* q_stats, const int32_t* sched_len,
                                  float temperature, uint64_t seed, int32_t* out_tokens, int32_t* accepted_len,
                                  float* p_tok, void* workspace, size_t workspace_bytes, dspark_stream_t stream) {
  if (!gate) return DSPARK_ERR_INVALID_ARG;
  return verify_entry(R, gamma, V, rank, dtype, target_logits, base_logits, anchor, W1, gate, W2, draft_tokens,
                      q_tok, q_stats, sched_len, temperature, seed, out_tokens, accepted_len, p_tok, workspace,
                      workspace_bytes, stream);
}

}  // extern "C"

static dspark_status round_entry(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                                 const void* base_logits, const void* target_logits, const int32_t* anchor,
                                 const void* W1, const void* gate, const void* W2, const float* conf,
                                 const float* conf_lagged, const float* sps_table, int32_t n_table, int32_t mode,
                                 float temperature, uint64_t seed, int32_t* draft_tokens, float* q_tok,
                                 float* q_stats, int32_t* sched_len, int32_t* K, double* tau_theta,
                                 int32_t* out_tokens, int32_t* accepted_len, float* p_tok, void* workspace,
                                 size_t workspace_bytes, dspark_stream_t stream) {
  g_last_launches = 0;
  if (!dims_ok(R, gamma, V, rank, dtype) || !(temperature >= 0.f) || !isfinite(temperature))
    return DSPARK_ERR_INVALID_ARG;
  if (mode != DSPARK_SCHED_CAUSAL && mode != DSPARK_SCHED_LAGGED && mode != DSPARK_SCHED_ALL)
    return DSPARK_ERR_INVALID_ARG;
  if (!base_logits || !target_logits || !anchor || !W1 || !W2 || !conf || !draft_tokens || !q_tok ||
      !q_stats || !sched_len || !K || !tau_theta || !out_tokens || !accepted_len || !p_tok ||
      n_table < 0 || (n_table > 0 && !sps_table) || (mode == DSPARK_SCHED_LAGGED && !conf_lagged))
    return DSPARK_ERR_INVALID_ARG;
  if (!ws_ok(workspace, workspace_bytes, dspark_workspace_bytes(R, gamma, V, rank, dtype, n_table)))
    return DSPARK_ERR_WORKSPACE;
  if (gate && !gated_verify_supported(R, gamma, V, rank, dtype, target_logits, base_logits, anchor, W1, gate, W2,
                                      workspace))
    return DSPARK_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int n = 0;
  // The schedule's inputs do not depend on the draft, nor do the target row statistics that verification
  // needs (given the schedule): on the tensor-core path the drafting launch computes both while it sweeps,
  // and runs the acceptance chains after its last draw; else the scheduler and verification run as their
  // own launches. In ALL mode every target row is verified, more than the launch's spare CTAs can stream
  // during the sweep, and verification keeps its own launch.
  ScheduleArgs sa{R, gamma, conf, conf_lagged, sps_table, n_table, mode, sched_len, K, tau_theta, workspace};
  VerifyArgs va{R, gamma, V, rank, dtype, target_logits, base_logits, anchor, W1, W2, draft_tokens,
                q_tok, q_stats, sched_len, temperature, seed, out_tokens, accepted_len, p_tok, workspace, gate};
  bool sched_done = false, verify_done = false;
  DraftArgs da{R, gamma, V, rank, dtype, base_logits, anchor, W1, W2, temperature, seed,
               draft_tokens, q_tok, q_stats, workspace, gate, &sa, &sched_done,
               mode == DSPARK_SCHED_ALL ? nullptr : &va, &verify_done};
  cudaError_t e;
  if (gate) {
    bool taken = false;
    e = launch_draft_persistent(da, s, n, taken);
    if (e == cudaSuccess && !taken) return DSPARK_ERR_INVALID_ARG;  // nothing was enqueued
  } else {
    e = launch_draft(da, s, n);
  }
  if (e == cudaSuccess && !sched_done) e = launch_schedule(sa, s, n);
  if (e == cudaSuccess) e = verify_done ? launch_verify_tail(va, s, n) : launch_verify(va, s, n);
  g_last_launches = n;
  return cuda_status(e);
}

extern "C" {

dspark_status dspark_round(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                           const void* base_logits, const void* target_logits, const int32_t* anchor,
                           const void* W1, const void* W2, const float* conf, const float* conf_lagged,
                           const float* sps_table, int32_t n_table, int32_t mode, float temperature,
                           uint64_t seed, int32_t* draft_tokens, float* q_tok, float* q_stats,
                           int32_t* sched_len, int32_t* K, double* tau_theta, int32_t* out_tokens,
                           int32_t* accepted_len, float* p_tok, void* workspace, size_t workspace_bytes,
                           dspark_stream_t stream) {
  return round_entry(R, gamma, V, rank, dtype, base_logits, target_logits, anchor, W1, nullptr, W2, conf,
                     conf_lagged, sps_table, n_table, mode, temperature, seed, draft_tokens, q_tok, q_stats,
                     sched_len, K, tau_theta, out_tokens, accepted_len, p_tok, workspace, workspace_bytes, stream);
}

dspark_status dspark_round_gated(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                                 const void* base_logits, const void* target_logits, const int32_t* anchor,
                                 const void* W1, const void* gate, const void* W2, const float* conf,
                                 const float* conf_lagged, const float* sps_table, int32_t n_table, int32_t mode,
                                 float temperature, uint64_t seed, int32_t* draft_tokens, float* q_tok,
                                 float* q_stats, int32_t* sched_len, int32_t* K, double* tau_theta,
                                 int32_t* out_tokens, int32_t* accepted_len, float* p_tok, void* workspace,
                                 size_t workspace_bytes, dspark_stream_t stream) {
  if (!gate) return DSPARK_ERR_INVALID_ARG;
  return round_entry(R, gamma, V, rank, dtype, base_logits, target_logits, anchor, W1, gate, W2, conf,
                     conf_lagged, sps_table, n_table, mode, temperature, seed, draft_tokens, q_tok, q_stats,
                     sched_len, K, tau_theta, out_tokens, accepted_len, p_tok, workspace, workspace_bytes, stream);
}

dspark_status dspark_acceptance_labels(int32_t R, int32_t gamma, int32_t V, int32_t rank, int32_t dtype,
                                       const void* target_logits, const void* base_logits,
                                       const int32_t* anchor, const void* W1, const void* W2,
                                       const int32_t* draft_tokens, const float* q_stats, float temperature,
                                       float* labels, void* workspace, size_t workspace_bytes,
                                       dspark_stream_t stream) {
  g_last_launches = 0;
  if (!dims_ok(R, gamma, V, rank, dtype) || !(temperature >= 0.f) || !isfinite(temperature))
    return DSPARK_ERR_INVALID_ARG;
  if (!target_logits || !base_logits || !anchor || !W1 || !W2 || !draft_tokens || !q_stats || !labels)
    return DSPARK_ERR_INVALID_ARG;
  if (!ws_ok(workspace, workspace_bytes, ws_layout(R, gamma, V).total)) return DSPARK_ERR_WORKSPACE;
  if (temperature > 0.f) {  // decide support before enqueueing anything
    DraftArgs d{R, gamma, V, rank, dtype, base_logits, anchor, W1, W2, temperature, 0,
                nullptr, nullptr, nullptr, workspace};
    int dev = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (!draft_tc_eligible(d) || (reinterpret_cast<uintptr_t>(target_logits) & 15) != 0 || !coop)
      return DSPARK_ERR_INVALID_ARG;
  }
  LabelArgs a{R, gamma, V, rank, dtype, target_logits, base_logits, anchor, W1, W2, draft_tokens, q_stats,
              temperature, labels, workspace};
  int n = 0;
  bool supported = true;
  cudaError_t e = launch_labels(a, (cudaStream_t)stream, n, supported);
  g_last_launches = n;
  if (e == cudaSuccess && !supported) return DSPARK_ERR_INVALID_ARG;
  return cuda_status(e);
}

dspark_status dspark_copy_scheduled_rows(int32_t R, int32_t gamma, int32_t V, int32_t dtype, const void* host_target,
                                        void* device_target, const int32_t* host_sched_len,
                                        dspark_stream_t stream) {
  if (R < 1 || gamma < 1 || V < 1 || (dtype != DSPARK_FP32 && dtype != DSPARK_BF16) || !host_target ||
      !device_target || !host_sched_len)
    return DSPARK_ERR_INVALID_ARG;
  const size_t e = dtype == DSPARK_BF16 ? 2 : 4;
  const size_t row = (size_t)V * e, req = (size_t)(gamma + 1) * row;
  for (int r = 0; r < R; ++r) {
    const int L = host_sched_len[r] < 0 ? 0 : (host_sched_len[r] > gamma ? gamma : host_sched_len[r]);
    const size_t off = (size_t)r * req;
    if (cudaMemcpyAsync(static_cast<char*>(device_target) + off, static_cast<const char*>(host_target) + off,
                        (size_t)(L + 1) * row, cudaMemcpyHostToDevice, (cudaStream_t)stream) != cudaSuccess)
      return DSPARK_ERR_CUDA;
  }
  return DSPARK_OK;
}

dspark_status dspark_device_status(const void* workspace, dspark_stream_t stream) {
  if (!workspace) return DSPARK_ERR_WORKSPACE;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return DSPARK_ERR_CUDA;
  return (dspark_status)word;
}

const char* dspark_status_string(dspark_status status) {
  switch (status) {
    case DSPARK_OK: return "ok";
    case DSPARK_ERR_INVALID_ARG: return "invalid argument";
    case DSPARK_ERR_NONFINITE: return "non-finite confidence or cost-table entry";
    case DSPARK_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DSPARK_ERR_CUDA: return "CUDA runtime error";
    case DSPARK_ERR_TIMEOUT: return "bounded device wait ran out";
    case DSPARK_ERR_RANGE: return "token id outside [0, V)";
    case DSPARK_ERR_TOO_LARGE: return "R * gamma exceeds the 16384 candidates of the fixed scratch";
  }
  return "unknown status";
}

int32_t dspark_last_launch_count(void) { return g_last_launches; }

}  // extern "C"
