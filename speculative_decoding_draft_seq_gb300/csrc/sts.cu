// Sequential Temperature Scaling of the confidence head ("DSpark: Aceleração
// da inferência de LLM com speculative decoding [pdf]" (GeekNews), "Calibração
// posterior — Sequential Temperature Scaling (STS)"): per-position
// temperatures T_k, c'_k = sigmoid(logit(c_k) / T_k), chosen left to right on
// a held-out set by a 1-D grid search that minimises the expected calibration
// error of the calibrated survival a'_j = prod_{i<=j} c'_i against the outcome
// y_j = [A >= j] (A = leading drafted tokens that passed verification).
//
// Device plan, per position j (three launches): sts_bins_kernel evaluates
// every grid temperature on every row at once (grid x row blocks), binning
// a' into equal-width bins on [0, 1] with exact 2^-40 fixed-point sums of a'
// and of y (shared-memory then global atomics: order-free, deterministic);
// sts_select_kernel turns the sums into the ECE curve, takes the first
// minimum, clears the sums; sts_advance_kernel multiplies each row's survival
// by its calibrated c'_j. The calibrated probabilities are float64 throughout.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace dspark {

constexpr double kStsClip = 1e-6;
constexpr int kStsThreads = 256;
constexpr int kStsRowsPerThread = 4;
constexpr int kStsMaxBins = 64;

__device__ __forceinline__ double sts_logit(float c) {
  const double x = fmin(fmax((double)c, kStsClip), 1.0 - kStsClip);
  return log(x) - log1p(-x);
}
__device__ __forceinline__ double sts_sigmoid(double z, double T) { return 1.0 / (1.0 + exp(-z / T)); }

// z[n, k] = logit(clip(c[n, k])); a[n] = 1
__global__ void sts_prepare_kernel(int N, int gamma, const float* __restrict__ conf, double* __restrict__ z,
                                   double* __restrict__ a, uint32_t* status) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < (long long)N * gamma) {
    const float c = conf[i];
    if (!isfinite(c)) set_status(status, DSPARK_ERR_NONFINITE);
    z[i] = sts_logit(isfinite(c) ? c : 0.f);
  }
  if (i < N) a[i] = 1.0;
}

__device__ __forceinline__ unsigned long long fx40_d(double v) {  // round(v * 2^40), v >= 0
  return (unsigned long long)__double2ull_rn(v * 0x1p40);
}

// blockIdx.x = grid point t, blockIdx.y = block of rows
__global__ void __launch_bounds__(kStsThreads) sts_bins_kernel(int N, int gamma, int j, const double* __restrict__ z,
                                                               const double* __restrict__ a,
                                                               const int32_t* __restrict__ accepted,
                                                               const float* __restrict__ grid, int n_bins,
                                                               unsigned long long* __restrict__ sums) {
  __shared__ unsigned long long sp[kStsMaxBins], sy[kStsMaxBins];
  const int t = blockIdx.x;
  for (int b = threadIdx.x; b < n_bins; b += blockDim.x) { sp[b] = 0ull; sy[b] = 0ull; }
  __syncthreads();
  const double T = (double)grid[t];
  const int r0 = blockIdx.y * kStsThreads * kStsRowsPerThread;
#pragma unroll
  for (int u = 0; u < kStsRowsPerThread; ++u) {
    const int n = r0 + u * kStsThreads + threadIdx.x;
    if (n < N) {
      const double ap = a[n] * sts_sigmoid(z[(size_t)n * gamma + (j - 1)], T);
      const int b = min((int)(ap * n_bins), n_bins - 1);
      atomicAdd(&sp[b], fx40_d(ap));
      if (accepted[n] >= j) atomicAdd(&sy[b], 1ull << 40);
    }
  }
  __syncthreads();
  for (int b = threadIdx.x; b < n_bins; b += blockDim.x) {
    if (sp[b]) atomicAdd(&sums[((size_t)t * n_bins + b) * 2], sp[b]);
    if (sy[b]) atomicAdd(&sums[((size_t)t * n_bins + b) * 2 + 1], sy[b]);
  }
}

// One CTA: ECE curve of position j, first minimum, sums cleared for the next position.
__global__ void __launch_bounds__(kStsThreads) sts_select_kernel(int N, int gamma, int j, int n_grid, int n_bins,
                                                                 const float* __restrict__ grid,
                                                                 unsigned long long* __restrict__ sums,
                                                                 float* __restrict__ temperature,
                                                                 float* __restrict__ ece_out, int* __restrict__ pick) {
  __shared__ double sv[kStsThreads];
  __shared__ int si[kStsThreads];
  double best = INFINITY;
  int besti = 0x7fffffff;
  for (int t = threadIdx.x; t < n_grid; t += blockDim.x) {
    double e = 0.0;
    for (int b = 0; b < n_bins; ++b) {
      unsigned long long* s = sums + ((size_t)t * n_bins + b) * 2;
      const long long d = (long long)(s[0] - s[1]);  // |sum a' - sum y| in 2^-40 units
      e += (double)(d < 0 ? -d : d) * 0x1p-40;
      s[0] = 0ull;
      s[1] = 0ull;
    }
    e /= (double)N;
    if (ece_out) ece_out[(size_t)(j - 1) * n_grid + t] = (float)e;
    if (e < best || (e == best && t < besti)) { best = e; besti = t; }
  }
  sv[threadIdx.x] = best;
  si[threadIdx.x] = besti;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < (int)blockDim.x; ++i)
      if (sv[i] < best || (sv[i] == best && si[i] < besti)) { best = sv[i]; besti = si[i]; }
    *pick = besti;
    temperature[j - 1] = grid[besti];
  }
}

__global__ void sts_advance_kernel(int N, int gamma, int j, const double* __restrict__ z, double* __restrict__ a,
                                   const float* __restrict__ grid, const int* __restrict__ pick) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n < N) a[n] = a[n] * sts_sigmoid(z[(size_t)n * gamma + (j - 1)], (double)grid[*pick]);
}

__global__ void sts_apply_kernel(int R, int gamma, const float* __restrict__ conf, const float* __restrict__ T,
                                 float* __restrict__ out) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)R * gamma) return;
  const int k = (int)(i % gamma);
  const float c = conf[i];
  out[i] = isfinite(c) ? (float)sts_sigmoid(sts_logit(c), (double)T[k]) : c;  // non-finite stays for the scheduler
}

// Scratch: status u32[64] | z double[N * gamma] | a double[N] | sums u64[n_grid * n_bins * 2] | pick int
struct StsLayout {
  size_t status, z, a, sums, pick, total;
};
inline StsLayout sts_layout(int N, int gamma, int n_grid, int n_bins) {
  StsLayout L;
  size_t o = 0;
  L.status = o; o = align256(o + 64 * sizeof(uint32_t));
  L.z = o;      o = align256(o + (size_t)N * gamma * sizeof(double));
  L.a = o;      o = align256(o + (size_t)N * sizeof(double));
  L.sums = o;   o = align256(o + (size_t)n_grid * n_bins * 2 * sizeof(unsigned long long));
  L.pick = o;   o = align256(o + sizeof(int));
  L.total = o;
  return L;
}

}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_sts_scratch_bytes(int32_t N, int32_t gamma, int32_t n_grid, int32_t n_bins) {
  if (N < 1 || gamma < 1 || n_grid < 1 || n_bins < 1 || n_bins > kStsMaxBins) return 0;
  return sts_layout(N, gamma, n_grid, n_bins).total;
}

extern "C" dspark_status dspark_sts_fit(int32_t N, int32_t gamma, const float* conf, const int32_t* accepted,
                                        int32_t n_grid, const float* grid, int32_t n_bins, float* temperature,
                                        float* ece, void* scratch, size_t scratch_bytes, dspark_stream_t stream) {
  if (N < 1 || gamma < 1 || n_grid < 1 || n_bins < 1 || n_bins > kStsMaxBins || !conf || !accepted || !grid ||
      !temperature)
    return DSPARK_ERR_INVALID_ARG;
  const StsLayout L = sts_layout(N, gamma, n_grid, n_bins);
  if (!scratch || scratch_bytes < L.total || (reinterpret_cast<uintptr_t>(scratch) & 255) != 0)
    return DSPARK_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  char* base = static_cast<char*>(scratch);
  uint32_t* status = reinterpret_cast<uint32_t*>(base + L.status);
  double* z = reinterpret_cast<double*>(base + L.z);
  double* a = reinterpret_cast<double*>(base + L.a);
  unsigned long long* sums = reinterpret_cast<unsigned long long*>(base + L.sums);
  int* pick = reinterpret_cast<int*>(base + L.pick);
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (cudaMemsetAsync(sums, 0, (size_t)n_grid * n_bins * 2 * sizeof(unsigned long long), s) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  const long long nz = (long long)N * gamma;
  sts_prepare_kernel<<<(int)ceil_div(std::max<long long>(nz, N), 256), 256, 0, s>>>(N, gamma, conf, z, a, status);
  const dim3 bgrid((unsigned)n_grid, (unsigned)ceil_div(N, kStsThreads * kStsRowsPerThread));
  for (int j = 1; j <= gamma; ++j) {
    sts_bins_kernel<<<bgrid, kStsThreads, 0, s>>>(N, gamma, j, z, a, accepted, grid, n_bins, sums);
    sts_select_kernel<<<1, kStsThreads, 0, s>>>(N, gamma, j, n_grid, n_bins, grid, sums, temperature, ece, pick);
    sts_advance_kernel<<<ceil_div(N, 256), 256, 0, s>>>(N, gamma, j, z, a, grid, pick);
  }
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

extern "C" dspark_status dspark_sts_status(const void* scratch, dspark_stream_t stream) {
  if (!scratch) return DSPARK_ERR_WORKSPACE;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return DSPARK_ERR_CUDA;
  return (dspark_status)word;
}

extern "C" dspark_status dspark_sts_apply(int32_t R, int32_t gamma, const float* conf, const float* temperature,
                                          float* conf_out, dspark_stream_t stream) {
  if (R < 1 || gamma < 1 || !conf || !temperature || !conf_out) return DSPARK_ERR_INVALID_ARG;
  const long long n = (long long)R * gamma;
  sts_apply_kernel<<<(int)ceil_div(n, 256), 256, 0, (cudaStream_t)stream>>>(R, gamma, conf, temperature, conf_out);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}
