// Hardware-aware prefix scheduler ("DSpark: Aceleração da inferência de LLM com
// speculative decoding [pdf]" (GeekNews), "Verificação com agendamento por
// confiança": cumulative prefix survival a_{r,j} = prod c_{r,i}; all R x gamma
// candidates merged by a in descending order and admitted greedily against the
// steps-per-second table SPS(B), stopping at the first admission that lowers
// Theta = tau * SPS(B); production variant in "Aplicação prática do scheduler":
// K from the confidences of two steps earlier by an unconstrained search, then
// the top K of the current ranking).
//
// Two forms. Up to 4,096 candidates, schedule_small_kernel: up to one CTA per
// SM, each building every survival key and ranking its own candidates by
// counting (below). Larger problems, schedule_kernel: schedule_block
// (sched_common.cuh) in one CTA of 1024 threads -- survival products per
// request in float32, a stable LSD radix sort of 32-bit keys (4-bit digits,
// per-thread contiguous segments, counts scanned in digit-major order) with
// the flat candidate index as payload, an exact fixed-point (2^-40) inclusive
// scan of the sorted survivals, and the Theta_i comparisons in float64 with the
// operation order fixed by the C ABI. Inside dspark_round on the tensor-core
// path, one extra CTA of the drafting launch runs schedule_block instead.
#include "common.cuh"
#include "internal.h"
#include "sched_common.cuh"

#include <algorithm>

namespace dspark {

constexpr int kSchedThreads = 1024;
constexpr size_t kSchedSmemMax = (size_t)kDigits * kSchedThreads * sizeof(uint32_t) +
                                  4 * (size_t)kSmemKeys * sizeof(uint32_t);

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(
    int R, int gamma, const float* __restrict__ conf, const float* __restrict__ conf_lag,
    const float* __restrict__ sps, int n_table, int mode, int32_t* __restrict__ L,
    int32_t* __restrict__ Kout, double* __restrict__ tau_theta, uint32_t* key0, uint32_t* key1,
    uint32_t* idx0, uint32_t* idx1, unsigned long long* fx, uint32_t* status) {
  extern __shared__ uint32_t cnt[];  // kDigits * blockDim.x, then the keys when they fit
  __shared__ unsigned long long shu[32];
  __shared__ int shi[32];
  __shared__ double shd[32];
  __shared__ int sBad;
  const BlockSchedScratch sc{cnt, R * gamma <= kSmemKeys ? cnt + kDigits * blockDim.x : nullptr, shu, shi, shd,
                             &sBad};
  schedule_block(R, gamma, conf, conf_lag, sps, n_table, mode, L, Kout, tau_theta, key0, key1, idx0, idx1, fx,
                 status, sc);
}

// ---------------------------------------------------------------------------
// Small problems (R * gamma <= kRankMaxKeys): one launch of up to one CTA per
// SM instead of one CTA.
//
// Every CTA forms all the survival keys and their running fixed-point row
// sums in shared memory (column-major tables, conflict-free for a warp). Warp
// w of CTA b takes candidates 8 b + w, 8 (b + grid) + w, ...: its 32 lanes
// count over the rows both the candidates before it in the ascending key
// order (ties by flat index: the radix sort's order) and the fixed-point sum
// of their survivals. So the warp knows the candidate's sorted position p and
// the exact prefix sums S_p (before it) and S_p + f (with it), and evaluates
// the admission rule at that position:
//   CAUSAL: admitting position p stops the scheduler iff B = R + p + 1 >
//     n_table or Theta(S_p + f, SPS[B - 1]) < Theta(S_p, SPS[B - 2]); the
//     smallest stopping position is K, gathered by an atomic max of n - p;
//   LAGGED: Theta_{p+1} on the lagged order, written for the argmax;
//   ALL: nothing (every candidate is admitted; the sum of all survivals is
//     the sum of the rows' last running sums).
// The last CTA to finish (a counter in the status block; it resets every
// counter it used) reads K (LAGGED: the smallest argmax of the Theta_i),
// the prefix at K of the current order, and counts L_r = #{j : p(r, j) < K}
// (the order is prefix-closed within a request).
constexpr int kRankThreads = 256;
constexpr int kRankWarps = kRankThreads / 32;
constexpr int kRankMaxKeys = 4096;
constexpr int kRankStageMax = kRankMaxKeys * 3 / 2;  // R (gamma | 1) <= 3/2 R gamma

// Byte offsets of the tables in dynamic shared memory (the lagged ones empty
// unless LAGGED), and their total.
struct SmallLayout {
  int Rs, m;
  size_t fxv, fxl, key, keyl, stg, stgl, spsv, bytes;
};
inline __host__ __device__ SmallLayout small_layout(int R, int gamma, int n_table, bool lagged) {
  SmallLayout L;
  L.Rs = sched_col_stride(R, gamma, kRankMaxKeys);
  L.m = sched_sps_count(R, gamma, n_table);
  const size_t T = (size_t)L.Rs * gamma, S = (size_t)R * sched_stage_stride(gamma), nl = lagged ? 1 : 0;
  L.fxv = 0;
  L.fxl = L.fxv + 8 * T;
  L.key = L.fxl + nl * 8 * T;
  L.keyl = L.key + 4 * T;
  L.stg = L.keyl + nl * 4 * T;
  L.stgl = L.stg + 4 * S;
  L.spsv = L.stgl + nl * 4 * S;
  L.bytes = L.spsv + 4 * (size_t)L.m;
  return L;
}
constexpr size_t kSmallSmemMax =
    2 * (size_t)kRankMaxKeys * 12 + 2 * 4 * (size_t)kRankStageMax + 4 * ((size_t)kRankMaxKeys + 1);

__global__ void __launch_bounds__(kRankThreads) schedule_small_kernel(
    int R, int gamma, const float* __restrict__ conf, const float* __restrict__ conf_lag,
    const float* __restrict__ sps, int n_table, int mode, uint32_t* pos_g, unsigned long long* prefix_g,
    unsigned long long* theta_lag_g, int32_t* __restrict__ L, int32_t* __restrict__ Kout,
    double* __restrict__ tau_theta, uint32_t* status) {
  extern __shared__ __align__(16) unsigned char sm_raw[];
  const bool lagged = mode == DSPARK_SCHED_LAGGED;
  const SmallLayout Ly = small_layout(R, gamma, n_table, lagged);
  unsigned long long* fxv = reinterpret_cast<unsigned long long*>(sm_raw + Ly.fxv);
  unsigned long long* fxl = reinterpret_cast<unsigned long long*>(sm_raw + Ly.fxl);
  uint32_t* key = reinterpret_cast<uint32_t*>(sm_raw + Ly.key);
  uint32_t* keyl = reinterpret_cast<uint32_t*>(sm_raw + Ly.keyl);
  uint32_t* stg = reinterpret_cast<uint32_t*>(sm_raw + Ly.stg);
  uint32_t* stgl = reinterpret_cast<uint32_t*>(sm_raw + Ly.stgl);
  const float* spsv = reinterpret_cast<const float*>(sm_raw + Ly.spsv);
  __shared__ int sLast;
  __shared__ unsigned long long sMax[kRankWarps];
  __shared__ int sMaxI[kRankWarps];
  unsigned int* done = status + 2;
  unsigned int* stop_enc = status + 6;
  unsigned int* bad_table = status + 8;
  const int tid = threadIdx.x, T = blockDim.x, warp = tid >> 5, lane = tid & 31;
  const int n = R * gamma, Rs = Ly.Rs;
  bool badv = false;
  {  // this CTA's slice of the cost table must be finite (loads in flight with the staging's)
    const int per = ceil_div(n_table, (int)gridDim.x);
    const int j0 = (int)blockIdx.x * per, j1 = min(j0 + per, n_table);
    for (int j = j0 + tid; j < j1; j += T) badv |= !isfinite(__ldg(sps + j));
  }
  stage_sched_inputs(conf, lagged ? conf_lag : nullptr, sps, R, gamma, Ly.m, stg, stgl,
                     reinterpret_cast<float*>(sm_raw + Ly.spsv), tid, T);
  if (badv) atomicOr(bad_table, 1u);
  __syncthreads();
  survival_tables(stg, R, gamma, Rs, key, fxv, status, tid, T);
  if (lagged) survival_tables(stgl, R, gamma, Rs, keyl, fxl, status, tid, T);
  __syncthreads();
  const bool table_ok = R <= n_table;
  if (mode != DSPARK_SCHED_ALL) {
    for (int i = (int)blockIdx.x * kRankWarps + warp; i < n; i += (int)gridDim.x * kRankWarps) {  // warp-uniform
      const int r = i / gamma, j = i - r * gamma;
      int p;
      unsigned long long Sb;
      rank_and_prefix(key, fxv, R, gamma, Rs, r, j, lane, p, Sb);
      if (lane == 0) {
        const unsigned long long f = cand_fx(fxv, Rs, r, j);
        pos_g[i] = (uint32_t)p;
        prefix_g[p] = Sb + f;  // inclusive prefix at sorted position p
        if (mode == DSPARK_SCHED_CAUSAL && table_ok) {  // SPS(B) = spsv[B - R]
          const int B = R + p + 1;
          bool st = B > n_table;
          if (!st) st = theta_of(R, Sb + f, spsv[p + 1]) < theta_of(R, Sb, spsv[p]);
          if (st) atomicMax(stop_enc, (unsigned)(n - p));
        }
      }
      if (lagged) {
        int pl;
        unsigned long long Sl;
        rank_and_prefix(keyl, fxl, R, gamma, Rs, r, j, lane, pl, Sl);
        if (lane == 0 && table_ok && pl + 1 <= min(n, n_table - R))  // Theta_{pl+1} of the lagged order
          theta_lag_g[pl] = ordered_bits(theta_of(R, Sl + cand_fx(fxl, Rs, r, j), spsv[pl + 1]));
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    sLast = atomicAdd(done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!sLast) return;
  __threadfence();

  // admission (last CTA)
  const unsigned int enc = __ldcg(stop_enc);
  const unsigned int bad = __ldcg(bad_table);
  __syncthreads();
  if (tid == 0) {  // every counter back to zero for the next call
    *done = 0u;
    *stop_enc = 0u;
    *bad_table = 0u;
  }
  if (bad) {
    if (tid == 0) {
      set_status(status, DSPARK_ERR_NONFINITE);
      *Kout = 0;
      tau_theta[0] = (double)R;
      tau_theta[1] = 0.0;
    }
    for (int r = tid; r < R; r += T) L[r] = 0;
    return;
  }
  if (mode == DSPARK_SCHED_ALL) {
    const unsigned long long total = survival_total(fxv, R, gamma, Rs, sMax, tid, T, [] { __syncthreads(); });
    for (int r = tid; r < R; r += T) L[r] = gamma;
    if (tid == 0) {
      *Kout = n;
      tau_theta[0] = __dadd_rn((double)R, __dmul_rn(__ull2double_rn(total), 0x1p-40));
      tau_theta[1] = R + n <= n_table ? theta_of(R, total, spsv[n]) : 0.0;
    }
    return;
  }
  if (!table_ok) {
    for (int r = tid; r < R; r += T) L[r] = 0;
    if (tid == 0) {
      *Kout = 0;
      tau_theta[0] = (double)R;
      tau_theta[1] = 0.0;
    }
    return;
  }
  int K;
  if (lagged) {  // smallest argmax of Theta_i, i = 0..imax (Theta_0 = Theta(R, 0))
    const int imax = min(n, n_table - R);
    unsigned long long best = 0ull;
    int besti = 0x7fffffff;
    for (int j = tid; j <= imax; j += T) {
      const unsigned long long th =
          j == 0 ? ordered_bits(theta_of(R, 0ull, spsv[0])) : __ldcg(theta_lag_g + (j - 1));
      if (th > best || (th == best && j < besti)) { best = th; besti = j; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, besti, o);
      if (ob > best || (ob == best && oi < besti)) { best = ob; besti = oi; }
    }
    if ((tid & 31) == 0) { sMax[tid >> 5] = best; sMaxI[tid >> 5] = besti; }
    __syncthreads();
    best = 0ull;
    besti = 0x7fffffff;
    for (int w = 0; w < T / 32; ++w)
      if (sMax[w] > best || (sMax[w] == best && sMaxI[w] < besti)) { best = sMax[w]; besti = sMaxI[w]; }
    K = besti;
  } else {
    K = enc ? n - (int)enc : n;
  }
  // the prefix at K (thread 0) and the positions (every thread) are fetched together
  unsigned long long S = 0ull;
  float sps_K = 0.f;
  if (tid == 0) {
    S = K ? __ldcg(prefix_g + (K - 1)) : 0ull;
    sps_K = spsv[K];  // SPS(R + K)
  }
  uint32_t* srank = key;  // the positions, staged over the key array
  stage_smem(srank, pos_g, n);
  if (tid == 0) {
    *Kout = K;
    tau_theta[0] = __dadd_rn((double)R, __dmul_rn(__ull2double_rn(S), 0x1p-40));
    tau_theta[1] = theta_of(R, S, sps_K);
  }
  __syncthreads();
  for (int r = tid; r < R; r += T) {
    int cnt = 0;
    for (int j = 0; j < gamma; ++j) cnt += srank[r * gamma + j] < (uint32_t)K;
    L[r] = cnt;
  }
}

// Both scheduler forms behind one call: the many-CTA rank kernel (admission
// in its last CTA) for small problems, the single-CTA radix sort otherwise.
// Scratch: key0/key1/idx0/idx1 (u32[n] each), fx (u64[n]), for the small form
// fx2 (u64[n]); status[0] is the sticky status word, status[2], [6] and [8]
// the small form's completion counter, stop word and cost-table flag (zero
// between calls).
cudaError_t schedule_launch(const ScheduleArgs& a, uint32_t* key0, uint32_t* key1, uint32_t* idx0, uint32_t* idx1,
                            unsigned long long* fx, unsigned long long* fx2, uint32_t* status, cudaStream_t s,
                            int& launches) {
  const long long n = (long long)a.R * a.gamma;
  if (n <= kRankMaxKeys) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // at most one CTA per SM: every CTA builds the whole tables
    const int grid = std::min(ceil_div(n, kRankWarps), std::max(sms, 1));
    const size_t smem = small_layout(a.R, a.gamma, a.n_table, a.mode == DSPARK_SCHED_LAGGED).bytes;
    static std::atomic<unsigned long long> attr{0};
    e = set_smem_limit_once((const void*)schedule_small_kernel, (int)kSmallSmemMax, attr);
    if (e != cudaSuccess) return e;
    schedule_small_kernel<<<grid, kRankThreads, smem, s>>>(a.R, a.gamma, a.conf, a.conf_lagged, a.sps, a.n_table,
                                                           a.mode, key0, fx, fx2, a.sched_len, a.K, a.tau_theta,
                                                           status);
    launches += 1;
    return cudaGetLastError();
  }
  const size_t smem = (size_t)kDigits * kSchedThreads * 4 + (n <= kSmemKeys ? 4 * (size_t)kSmemKeys * 4 : 0);
  static std::atomic<unsigned long long> attr{0};
  {
    cudaError_t e = set_smem_limit_once((const void*)schedule_kernel, (int)kSchedSmemMax, attr);
    if (e != cudaSuccess) return e;
  }
  schedule_kernel<<<1, kSchedThreads, smem, s>>>(a.R, a.gamma, a.conf, a.conf_lagged, a.sps, a.n_table, a.mode,
                                                 a.sched_len, a.K, a.tau_theta, key0, key1, idx0, idx1, fx, status);
  launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_schedule(const ScheduleArgs& a, cudaStream_t s, int& launches) {
  const WsLayout L = ws_layout(a.R, a.gamma, 1);
  void* ws = a.ws;
  return schedule_launch(a, ws_at<uint32_t>(ws, L.skey0), ws_at<uint32_t>(ws, L.skey1), ws_at<uint32_t>(ws, L.sidx0),
                         ws_at<uint32_t>(ws, L.sidx1), ws_at<unsigned long long>(ws, L.fx),
                         ws_at<unsigned long long>(ws, L.fx2), ws_at<uint32_t>(ws, L.status), s, launches);
}

}  // namespace dspark

// ---------------------------------------------------------------------------
// Scheduler entry point that allocates nothing (dspark_schedule_static).
//
// Its scratch is the file-scope array below instead of a caller-provided
// workspace: a status word, the radix-sort ping-pong buffers and the
// fixed-point prefix sums for at most kStaticMaxCandidates = R * gamma
// candidates (393,472 bytes, held by every GPU that loads the library until
// the process exits). Host code cannot use the array's name as a device
// address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it.
namespace dspark {

constexpr int kStaticMaxCandidates = 16384;
constexpr size_t kStaticStatusOff = 0;
constexpr size_t kStaticKey0Off = 256;
constexpr size_t kStaticKey1Off = kStaticKey0Off + (size_t)kStaticMaxCandidates * 4;
constexpr size_t kStaticIdx0Off = kStaticKey1Off + (size_t)kStaticMaxCandidates * 4;
constexpr size_t kStaticIdx1Off = kStaticIdx0Off + (size_t)kStaticMaxCandidates * 4;
constexpr size_t kStaticFxOff = kStaticIdx1Off + (size_t)kStaticMaxCandidates * 4;
constexpr size_t kStaticScratchBytes = kStaticFxOff + (size_t)kStaticMaxCandidates * 8;

static __device__ __align__(256) unsigned char g_schedule_scratch[kStaticScratchBytes];

constexpr int kStaticMaxDevices = 64;
static void* g_schedule_scratch_ptr[kStaticMaxDevices] = {};

}  // namespace dspark

extern "C" dspark_status dspark_schedule_static(int32_t R, int32_t gamma, const float* conf,
                                                const float* conf_lagged, const float* sps_table,
                                                int32_t n_table, int32_t mode, int32_t* sched_len,
                                                int32_t* K, double* tau_theta, uint32_t* device_status,
                                                dspark_stream_t stream) {
  using namespace dspark;
  if (R < 1 || gamma < 1 || n_table < 0) return DSPARK_ERR_INVALID_ARG;
  if (mode != DSPARK_SCHED_CAUSAL && mode != DSPARK_SCHED_LAGGED && mode != DSPARK_SCHED_ALL)
    return DSPARK_ERR_INVALID_ARG;
  if (!conf || !sched_len || !K || !tau_theta || (n_table > 0 && !sps_table)) return DSPARK_ERR_INVALID_ARG;
  if (mode == DSPARK_SCHED_LAGGED && !conf_lagged) return DSPARK_ERR_INVALID_ARG;
  if ((long long)R * (long long)gamma > kStaticMaxCandidates) return DSPARK_ERR_TOO_LARGE;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kStaticMaxDevices) return DSPARK_ERR_CUDA;
  if (g_schedule_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_schedule_scratch) != cudaSuccess || p == nullptr) return DSPARK_ERR_CUDA;
    g_schedule_scratch_ptr[dev] = p;
  }
  char* base = static_cast<char*>(g_schedule_scratch_ptr[dev]);
  uint32_t* status = reinterpret_cast<uint32_t*>(base + kStaticStatusOff);
  cudaStream_t s = (cudaStream_t)stream;
  // The status word is the only scratch that must start at zero; every other
  // byte a call reads it has written first.
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return DSPARK_ERR_CUDA;
  // the small form's second survival array shares the key0/key1 bytes, which
  // that form leaves unused (it keeps its ranks in idx0)
  const ScheduleArgs a{R, gamma, conf, conf_lagged, sps_table, n_table, mode, sched_len, K, tau_theta, nullptr};
  int launches = 0;
  const bool small = (long long)R * gamma <= kRankMaxKeys;
  uint32_t* key0 = reinterpret_cast<uint32_t*>(base + kStaticKey0Off);
  uint32_t* key1 = reinterpret_cast<uint32_t*>(base + kStaticKey1Off);
  uint32_t* idx0 = reinterpret_cast<uint32_t*>(base + kStaticIdx0Off);
  uint32_t* idx1 = reinterpret_cast<uint32_t*>(base + kStaticIdx1Off);
  if (schedule_launch(a, small ? idx0 : key0, key1, small ? key0 : idx0, idx1,
                      reinterpret_cast<unsigned long long*>(base + kStaticFxOff),
                      reinterpret_cast<unsigned long long*>(base + kStaticKey0Off), status, s,
                      launches) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  if (device_status != nullptr &&
      cudaMemcpyAsync(device_status, status, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}
