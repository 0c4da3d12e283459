// Internal launch interface between the C-ABI layer and the kernel files.
#pragma once

#include <atomic>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dspark.h"

namespace dspark {

struct ScheduleArgs;
struct VerifyArgs;

struct DraftArgs {
  int R, gamma, V, rank, dtype;
  const void* base;
  const int32_t* anchor;
  const void* W1;
  const void* W2;
  float temperature;
  uint64_t seed;
  int32_t* tokens;
  float* q_tok;
  float* q_stats;
  void* ws;
  const void* gate = nullptr;  // gated head: gate values [V, rank] (bf16); null = Markov head
  // a round's schedule, computed by one extra CTA of the drafting launch when the tensor-core sweep
  // runs; *sched_done tells the caller whether it was
  const ScheduleArgs* sched = nullptr;
  bool* sched_done = nullptr;
  // with a schedule, the round's verification up to the residual draw (target row statistics of the
  // scheduled rows, the acceptance chains) in the same launch; *verify_done tells whether it was
  const VerifyArgs* verify = nullptr;
  bool* verify_done = nullptr;
};

struct ScheduleArgs {
  int R, gamma;
  const float* conf;
  const float* conf_lagged;
  const float* sps;
  int n_table, mode;
  int32_t* sched_len;
  int32_t* K;
  double* tau_theta;
  void* ws;
};

struct VerifyArgs {
  int R, gamma, V, rank, dtype;
  const void* target;
  const void* base;
  const int32_t* anchor;
  const void* W1;
  const void* W2;
  const int32_t* tokens;
  const float* q_tok;
  const float* q_stats;
  const int32_t* sched_len;
  float temperature;
  uint64_t seed;
  int32_t* out_tokens;
  int32_t* accepted_len;
  float* p_tok;
  void* ws;
  const void* gate = nullptr;  // gated head: gate values [V, rank] (bf16); null = Markov head
};

struct LabelArgs {
  int R, gamma, V, rank, dtype;
  const void* target;
  const void* base;
  const int32_t* anchor;
  const void* W1;
  const void* W2;
  const int32_t* tokens;
  const float* q_stats;
  float temperature;
  float* labels;
  void* ws;
};

// Each launcher enqueues its kernels on `s`, adds the number of kernel
// launches to `launches`, and returns cudaGetLastError().
// Raises a kernel's dynamic shared-memory limit, once per device (devices
// 0..63; others every call). `done` is a per-kernel bit mask of devices.
inline cudaError_t set_smem_limit_once(const void* fn, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

cudaError_t launch_draft(const DraftArgs& a, cudaStream_t s, int& launches);
// The gated head runs only on the persistent tensor-core path: bf16, rank a
// multiple of 64 up to 256, V a multiple of 8 and at least 64, 16-byte
// aligned tensors, cooperative launch.
bool gated_supported(const DraftArgs& a);
cudaError_t launch_schedule(const ScheduleArgs& a, cudaStream_t s, int& launches);
cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s, int& launches);
// Verification after the acceptance chains (the residual / bonus draw and, for the gated head, its A
// rows), for a round whose drafting launch computed the row statistics and chains.
cudaError_t launch_verify_tail(const VerifyArgs& a, cudaStream_t s, int& launches);
// Acceptance labels; `supported` is false (and nothing is launched) when the
// sampled-mode shape is outside the tensor-core path.
cudaError_t launch_labels(const LabelArgs& a, cudaStream_t s, int& launches, bool& supported);

}  // namespace dspark
