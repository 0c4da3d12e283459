// Hardware-aware prefix scheduler ("DSpark: Aceleração da inferência de LLM com
// speculative decoding [pdf]" (GeekNews), "Verificação com agendamento por
// confiança": cumulative prefix survival a_{r,j} = prod c_{r,i}; all R x gamma
// candidates merged by a in descending order and admitted greedily against the
// steps-per-second table SPS(B), stopping at the first admission that lowers
// Theta = tau * SPS(B); production variant in "Aplicação prática do scheduler":
// K from the confidences of two steps earlier by an unconstrained search, then
// the top K of the current ranking).
//
// One CTA of 1024 threads (the problem is at most 65536 keys and latency
// bound): survival products per request in float32, a stable LSD radix sort of
// 32-bit keys (4-bit digits, per-thread contiguous segments, counts scanned in
// digit-major order) with the flat candidate index as payload, an exact
// fixed-point (2^-40) inclusive scan of the sorted survivals, and the
// Theta_i comparisons in float64 with the operation order fixed by the C ABI.
#include "common.cuh"
#include "internal.h"
#include "sched_common.cuh"

namespace dspark {

constexpr int kSchedThreads = 1024;
constexpr int kDigits = 16;
// Up to this many candidates the sort keys and indices live in shared memory.
constexpr int kSmemKeys = 8192;
constexpr size_t kCntBytes = (size_t)kDigits * kSchedThreads * sizeof(uint32_t);
constexpr size_t kSchedSmemMax = kCntBytes + 4 * (size_t)kSmemKeys * sizeof(uint32_t);

// Exclusive scan of one unsigned 64-bit value per thread; returns the total.
__device__ __forceinline__ unsigned long long block_exscan_u64(unsigned long long v,
                                                               unsigned long long* sh,
                                                               unsigned long long& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  unsigned long long ex = __shfl_up_sync(0xffffffffu, x, 1);
  if (lane == 0) ex = 0;
  __syncthreads();
  if (lane == 31) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    unsigned long long s = lane < nw ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) sh[lane] = s;
  }
  __syncthreads();
  total = sh[nw - 1];
  const unsigned long long res = (w > 0 ? sh[w - 1] : 0ull) + ex;
  __syncthreads();
  return res;
}

// Survival keys of one confidence matrix; flags non-finite entries.
// `stage` (n words) receives the confidences in one coalesced pass first.
__device__ void build_keys(const float* conf, int R, int gamma, uint32_t* key, uint32_t* idx,
                           uint32_t* stage, uint32_t* status) {
  const int n = R * gamma;
  stage_smem(stage, reinterpret_cast<const uint32_t*>(conf), n);
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    float acc = 1.f;
    for (int j = 0; j < gamma; ++j) {
      float c = __uint_as_float(stage[(size_t)r * gamma + j]);
      if (!isfinite(c)) {
        set_status(status, DSPARK_ERR_NONFINITE);
        c = 0.f;
      }
      c = c > 0.f ? fminf(c, 1.f) : 0.f;
      acc = __fmul_rn(acc, c);
      key[(size_t)r * gamma + j] = survival_key(acc);
      idx[(size_t)r * gamma + j] = (uint32_t)(r * gamma + j);
    }
  }
  __syncthreads();
}

// Stable LSD radix sort of (key, idx), 8 passes of 4 bits; result in key0/idx0.
__device__ void radix_sort(uint32_t* key0, uint32_t* idx0, uint32_t* key1, uint32_t* idx1, int n,
                           uint32_t* cnt, unsigned long long* shu) {
  const int T = blockDim.x, tid = threadIdx.x;
  const int seg = ceil_div(n, T);
  const int s0 = min(n, tid * seg), s1 = min(n, s0 + seg);
  uint32_t *kin = key0, *iin = idx0, *kout = key1, *iout = idx1;
  for (int shift = 0; shift < 32; shift += 4) {
    for (int d = 0; d < kDigits; ++d) cnt[d * T + tid] = 0;
    for (int i = s0; i < s1; ++i) cnt[((kin[i] >> shift) & 15u) * T + tid] += 1;
    __syncthreads();
    uint32_t loc[kDigits];
    unsigned long long sum = 0;
#pragma unroll
    for (int j = 0; j < kDigits; ++j) {
      loc[j] = cnt[kDigits * tid + j];
      sum += loc[j];
    }
    unsigned long long tot;
    unsigned long long run = block_exscan_u64(sum, shu, tot);
#pragma unroll
    for (int j = 0; j < kDigits; ++j) {
      cnt[kDigits * tid + j] = (uint32_t)run;
      run += loc[j];
    }
    __syncthreads();
    for (int i = s0; i < s1; ++i) {
      const uint32_t k = kin[i];
      const uint32_t slot = ((k >> shift) & 15u) * T + tid;
      const uint32_t pos = cnt[slot];
      cnt[slot] = pos + 1;
      kout[pos] = k;
      iout[pos] = iin[i];
    }
    __syncthreads();
    uint32_t* t;
    t = kin; kin = kout; kout = t;
    t = iin; iin = iout; iout = t;
  }
}

// fx[i] = sum of fixed_point(a) over sorted positions 0..i.
__device__ void fixed_prefix(const uint32_t* key, int n, unsigned long long* fx, unsigned long long* shu) {
  const int T = blockDim.x, tid = threadIdx.x;
  const int seg = ceil_div(n, T);
  const int s0 = min(n, tid * seg), s1 = min(n, s0 + seg);
  unsigned long long loc = 0;
  for (int i = s0; i < s1; ++i) loc += fixed_point(key_survival(key[i]));
  unsigned long long tot;
  unsigned long long run = block_exscan_u64(loc, shu, tot);
  for (int i = s0; i < s1; ++i) {
    run += fixed_point(key_survival(key[i]));
    fx[i] = run;
  }
  __syncthreads();
}

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
  const int tid = threadIdx.x, T = blockDim.x;
  const int n = R * gamma;
  if (n <= kSmemKeys) {  // sort in shared memory
    uint32_t* sk = cnt + kDigits * kSchedThreads;
    key0 = sk;
    key1 = sk + kSmemKeys;
    idx0 = sk + 2 * kSmemKeys;
    idx1 = sk + 3 * kSmemKeys;
  }

  if (tid == 0) sBad = 0;
  __syncthreads();
  for (int i = tid; i < n_table; i += T)
    if (!isfinite(sps[i])) sBad = 1;
  for (int r = tid; r < R; r += T) L[r] = (mode == DSPARK_SCHED_ALL) ? gamma : 0;
  __syncthreads();
  if (sBad) {
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
    build_keys(conf, R, gamma, key0, idx0, key1, status);
    unsigned long long loc = 0;
    for (int i = tid; i < n; i += T) loc += fixed_point(key_survival(key0[i]));
    unsigned long long tot;
    block_exscan_u64(loc, shu, tot);
    if (tid == 0) {
      *Kout = n;
      tau_theta[0] = __dadd_rn((double)R, __dmul_rn(__ull2double_rn(tot), 0x1p-40));
      tau_theta[1] = (R + n >= 1 && R + n <= n_table) ? theta_of(R, tot, sps[R + n - 1]) : 0.0;
    }
    return;
  }

  if (R > n_table) {
    if (tid == 0) {
      *Kout = 0;
      tau_theta[0] = (double)R;
      tau_theta[1] = 0.0;
    }
    return;
  }

  int K = 0;
  if (mode == DSPARK_SCHED_LAGGED) {
    build_keys(conf_lag, R, gamma, key0, idx0, key1, status);
    radix_sort(key0, idx0, key1, idx1, n, cnt, shu);
    fixed_prefix(key0, n, fx, shu);
    const int imax = min(n, n_table - R);
    // smallest argmax of Theta_i, i = 0..imax
    double best = -INFINITY;
    int besti = 0x7fffffff;
    for (int i = tid; i <= imax; i += T) {
      const unsigned long long S = i ? fx[i - 1] : 0ull;
      const double th = theta_of(R, S, sps[R + i - 1]);
      if (th > best || (th == best && i < besti)) { best = th; besti = i; }
    }
    // block (value, index) argmax in float64
    const int lane = tid & 31, w = tid >> 5, nw = T >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, besti, o);
      if (ob > best || (ob == best && oi < besti)) { best = ob; besti = oi; }
    }
    __syncthreads();
    if (lane == 0) { shd[w] = best; shi[w] = besti; }
    __syncthreads();
    best = lane < nw ? shd[lane] : -INFINITY;
    besti = lane < nw ? shi[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, besti, o);
      if (ob > best || (ob == best && oi < besti)) { best = ob; besti = oi; }
    }
    K = besti;
    __syncthreads();
  }

  build_keys(conf, R, gamma, key0, idx0, key1, status);
  radix_sort(key0, idx0, key1, idx1, n, cnt, shu);
  fixed_prefix(key0, n, fx, shu);

  if (mode == DSPARK_SCHED_CAUSAL) {
    const int seg = ceil_div(n, T);
    const int s0 = min(n, tid * seg), s1 = min(n, s0 + seg);
    int stop = 0x7fffffff;
    for (int i = s0; i < s1; ++i) {
      const int B = R + i + 1;
      bool st = B > n_table;
      if (!st) {
        const double th_next = theta_of(R, fx[i], sps[B - 1]);
        const double th_prev = theta_of(R, i ? fx[i - 1] : 0ull, sps[B - 2]);
        st = th_next < th_prev;
      }
      if (st) { stop = i; break; }
    }
    K = block_min_i(stop, shi);
    if (K == 0x7fffffff) K = n;
  }

  for (int i = tid; i < K; i += T) atomicAdd(&L[idx0[i] / (uint32_t)gamma], 1);
  if (tid == 0) {
    const unsigned long long S = K ? fx[K - 1] : 0ull;
    *Kout = K;
    tau_theta[0] = __dadd_rn((double)R, __dmul_rn(__ull2double_rn(S), 0x1p-40));
    tau_theta[1] = theta_of(R, S, sps[R + K - 1]);
  }
}

// ---------------------------------------------------------------------------
// Small problems (R * gamma <= kRankMaxKeys): one launch of many CTAs instead
// of one CTA.
//
// Every CTA forms all the survival keys and their fixed-point values in
// shared memory. For each of its own kRankKeysPerCta candidates, kRankSplit
// threads count over interleaved slices of the keys both the candidates
// before it in the ascending key order (ties by flat index: the radix sort's
// order) and the fixed-point sum of their survivals. So the CTA knows the
// candidate's sorted position p and the exact prefix sums S_p (before it) and
// S_p + f (with it), and evaluates the admission rule at that position:
//   CAUSAL: admitting position p stops the scheduler iff B = R + p + 1 >
//     n_table or Theta(S_p + f, SPS[B - 1]) < Theta(S_p, SPS[B - 2]); the
//     smallest stopping position is K, gathered by an atomic max of n - p;
//   LAGGED: Theta_{p+1} on the lagged order, written for the argmax;
//   ALL: the survivals' sum, gathered by an atomic add.
// The last CTA to finish (a counter in the status block; it resets every
// counter it used) reads K (LAGGED: the smallest argmax of the Theta_i),
// the prefix at K of the current order, and counts L_r = #{j : p(r, j) < K}
// (the order is prefix-closed within a request).
constexpr int kRankThreads = 256;
constexpr int kRankKeysPerCta = kRankThreads / kRankSplit;
constexpr int kRankMaxKeys = 4096;
// keys + fixed-point survivals, current and lagged
constexpr size_t kSmallSmem = 2 * (size_t)kRankMaxKeys * (sizeof(uint32_t) + sizeof(unsigned long long));

__global__ void __launch_bounds__(kRankThreads) schedule_small_kernel(
    int R, int gamma, const float* __restrict__ conf, const float* __restrict__ conf_lag,
    const float* __restrict__ sps, int n_table, int mode, uint32_t* pos_g, unsigned long long* prefix_g,
    unsigned long long* theta_lag_g, int32_t* __restrict__ L, int32_t* __restrict__ Kout,
    double* __restrict__ tau_theta, uint32_t* status) {
  extern __shared__ __align__(16) unsigned char sm_raw[];
  unsigned long long* fxv = reinterpret_cast<unsigned long long*>(sm_raw);
  unsigned long long* fxl = fxv + kRankMaxKeys;
  uint32_t* key = reinterpret_cast<uint32_t*>(fxl + kRankMaxKeys);
  uint32_t* keyl = key + kRankMaxKeys;
  __shared__ int sLast;
  __shared__ unsigned long long sMax[kRankThreads / 32];
  __shared__ int sMaxI[kRankThreads / 32];
  unsigned int* done = status + 2;
  unsigned long long* all_sum = reinterpret_cast<unsigned long long*>(status + 4);
  unsigned int* stop_enc = status + 6;
  unsigned int* bad_table = status + 8;
  const int tid = threadIdx.x, T = blockDim.x;
  const int n = R * gamma;
  const bool lagged = mode == DSPARK_SCHED_LAGGED;
  {  // this CTA's slice of the cost table must be finite
    const int per = ceil_div(n_table, (int)gridDim.x);
    const int j0 = (int)blockIdx.x * per, j1 = min(j0 + per, n_table);
    bool badv = false;
    for (int j = j0 + tid; j < j1; j += T) badv |= !isfinite(__ldg(sps + j));
    if (badv) atomicOr(bad_table, 1u);
  }

  auto sync_all = [] { __syncthreads(); };
  survival_keys_smem(conf, R, gamma, key, fxv, status, tid, T, sync_all);
  if (lagged) survival_keys_smem(conf_lag, R, gamma, keyl, fxl, status, tid, T, sync_all);
  __syncthreads();
  const int i = blockIdx.x * kRankKeysPerCta + tid / kRankSplit;
  const int s = tid % kRankSplit;
  const bool mine = s == 0 && i < n;
  const bool table_ok = R <= n_table;
  if (mode == DSPARK_SCHED_ALL) {  // the sum is order-free: each CTA adds its own candidates
    unsigned long long v = mine ? cand_fx(fxv, gamma, i) : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((tid & 31) == 0 && v) atomicAdd(all_sum, v);
  } else {
    int p;
    unsigned long long Sb;
    rank_and_prefix(key, fxv, R, gamma, i, s, p, Sb);
    if (mine) {
      pos_g[i] = (uint32_t)p;
      prefix_g[p] = Sb + cand_fx(fxv, gamma, i);  // inclusive prefix at sorted position p
      if (mode == DSPARK_SCHED_CAUSAL && table_ok) {
        const int B = R + p + 1;
        bool st = B > n_table;
        if (!st) st = theta_of(R, Sb + cand_fx(fxv, gamma, i), sps[B - 1]) < theta_of(R, Sb, sps[B - 2]);
        if (st) atomicMax(stop_enc, (unsigned)(n - p));
      }
    }
    if (lagged) {
      int pl;
      unsigned long long Sl;
      rank_and_prefix(keyl, fxl, R, gamma, i, s, pl, Sl);
      if (mine && table_ok && pl + 1 <= min(n, n_table - R))  // Theta_{pl+1} of the lagged order
        theta_lag_g[pl] = ordered_bits(theta_of(R, Sl + cand_fx(fxl, gamma, i), sps[R + pl]));
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
  const unsigned long long total = __ldcg(all_sum);
  const unsigned int enc = __ldcg(stop_enc);
  const unsigned int bad = __ldcg(bad_table);
  __syncthreads();
  if (tid == 0) {  // every counter back to zero for the next call
    *done = 0u;
    *all_sum = 0ull;
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
    for (int r = tid; r < R; r += T) L[r] = gamma;
    if (tid == 0) {
      *Kout = n;
      tau_theta[0] = __dadd_rn((double)R, __dmul_rn(__ull2double_rn(total), 0x1p-40));
      tau_theta[1] = (R + n >= 1 && R + n <= n_table) ? theta_of(R, total, sps[R + n - 1]) : 0.0;
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
          j == 0 ? ordered_bits(theta_of(R, 0ull, sps[R - 1])) : __ldcg(theta_lag_g + (j - 1));
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
    sps_K = __ldg(sps + R + K - 1);
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
// fx2 (u64[n]); status[0] is the sticky status word, status[2], [4..5], [6]
// and [8] the small form's completion counter, sum, stop word and cost-table
// flag (zero between calls).
cudaError_t schedule_launch(const ScheduleArgs& a, uint32_t* key0, uint32_t* key1, uint32_t* idx0, uint32_t* idx1,
                            unsigned long long* fx, unsigned long long* fx2, uint32_t* status, cudaStream_t s,
                            int& launches) {
  const long long n = (long long)a.R * a.gamma;
  if (n <= kRankMaxKeys) {
    const int grid = (int)ceil_div(n, kRankKeysPerCta);
    static std::atomic<unsigned long long> attr{0};
    {
      cudaError_t e = set_smem_limit_once((const void*)schedule_small_kernel, (int)kSmallSmem, attr);
      if (e != cudaSuccess) return e;
    }
    schedule_small_kernel<<<grid, kRankThreads, kSmallSmem, s>>>(a.R, a.gamma, a.conf, a.conf_lagged, a.sps,
                                                                 a.n_table, a.mode, key0, fx, fx2, a.sched_len, a.K,
                                                                 a.tau_theta, status);
    launches += 1;
    return cudaGetLastError();
  }
  const size_t smem = kCntBytes + (n <= kSmemKeys ? 4 * (size_t)kSmemKeys * 4 : 0);
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
