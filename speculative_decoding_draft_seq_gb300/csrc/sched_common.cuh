// The prefix scheduler's device code, shared by its own kernels (schedule.cu)
// and by the scheduler CTA of the drafting launch (draft_persistent.cu):
// survival keys, the exact 2^-40 fixed-point survivals, Theta = tau * SPS(B)
// in float64, the counting rank of one candidate (many-CTA form) and the
// whole scheduler in one thread block ("DSpark: Aceleração da inferência de LLM com
// speculative decoding [pdf]" (GeekNews), "Verificação com agendamento por
// confiança").
#pragma once

#include "common.cuh"

namespace dspark {

// Threads per candidate in the counting rank: one warp.
constexpr int kRankSplit = 32;

// Coalesced copy of n words from global (L2) to shared memory with eight loads
// in flight per thread (a load-then-store loop would wait out one memory round
// trip per iteration).
// Threads t = 0..nt-1 of the participating group take part.
template <class T>
__device__ void stage_smem(T* dst, const T* src, int n, int t, int nt) {
  constexpr int kU = 8;
  for (int base = t; base < n; base += kU * nt) {
    T v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int j = base + u * nt;
      v[u] = j < n ? __ldcg(src + j) : T();
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int j = base + u * nt;
      if (j < n) dst[j] = v[u];
    }
  }
}
template <class T>
__device__ void stage_smem(T* dst, const T* src, int n) { stage_smem(dst, src, n, (int)threadIdx.x, (int)blockDim.x); }

// a in [0, 1] -> ascending sort key (descending a); bits of +0.0 .. 1.0.
__device__ __forceinline__ uint32_t survival_key(float a) { return 0x3F800000u - __float_as_uint(a); }
__device__ __forceinline__ float key_survival(uint32_t key) { return __uint_as_float(0x3F800000u - key); }

// floor(a * 2^40 + 1/2) for a float32 a in [0, 1], with integer operations
// (equal to the same expression evaluated exactly in float64).
__device__ __forceinline__ unsigned long long fixed_point(float a) {
  const uint32_t b = __float_as_uint(a);
  const int e = (int)((b >> 23) & 0xFFu);
  if (e == 0) return 0ull;  // zero or subnormal: below 2^-41
  const unsigned long long m = (unsigned long long)((b & 0x7FFFFFu) | 0x800000u);
  const int sh = e - 110;  // a * 2^40 = m * 2^(e - 110)
  if (sh >= 0) return m << sh;
  const int s = -sh;
  if (s > 40) return 0ull;
  return (m + (1ull << (s - 1))) >> s;
}

__device__ __forceinline__ double theta_of(int R, unsigned long long S, float sps) {
  const double tau = __dadd_rn((double)R, __dmul_rn(__ull2double_rn(S), 0x1p-40));
  return __dmul_rn(tau, (double)sps);
}

// Shared-memory layout of the rank form. The survival keys and the running
// fixed-point row sums are column-major -- entry (r, j) at j * Rs + r -- with
// Rs = R rounded up to a multiple of 32 when Rs * gamma fits `cap` entries
// (else R): the 32 lanes of a warp that read one column at rows lane,
// lane + 32, ... then hit 32 distinct banks. The confidences are staged with
// the odd row stride gamma | 1, so that threads reading entry j of
// consecutive rows hit distinct banks too.
__host__ __device__ __forceinline__ int sched_col_stride(int R, int gamma, int cap) {
  const int Rp = (R + 31) & ~31;
  return (long long)Rp * gamma <= cap ? Rp : R;
}
__host__ __device__ __forceinline__ int sched_stage_stride(int gamma) { return gamma | 1; }
// The cost-table entries the schedule reads, SPS(R) .. SPS(R + m - 1) (the
// batch sizes from no admitted candidate to all of them, within the table):
// m of them, staged as spsv[t] = sps[R - 1 + t].
__host__ __device__ __forceinline__ int sched_sps_count(int R, int gamma, int n_table) {
  if (R > n_table) return 0;
  const int n = R * gamma, room = n_table - R;
  return (n < room ? n : room) + 1;
}

// One coalesced pass over the schedule's inputs, eight loads of each in
// flight per thread: the confidences (and the lagged ones, when conf_lag is
// not null) into rows of stride gamma | 1, and m cost-table entries from
// SPS(R) on. Threads t = 0..nt-1 of the group take part.
__device__ __forceinline__ void stage_sched_inputs(const float* conf, const float* conf_lag, const float* sps, int R,
                                                   int gamma, int m, uint32_t* stg, uint32_t* stgl, float* spsv,
                                                   int t, int nt) {
  constexpr int kU = 8;
  const int n = R * gamma, gs = sched_stage_stride(gamma), total = max(n, m);
  const uint32_t* c32 = reinterpret_cast<const uint32_t*>(conf);
  const uint32_t* l32 = reinterpret_cast<const uint32_t*>(conf_lag);
  for (int base = t; base < total; base += kU * nt) {
    uint32_t c[kU], cl[kU];
    float sv[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int j = base + u * nt;
      c[u] = j < n ? __ldcg(c32 + j) : 0u;
      cl[u] = (l32 != nullptr && j < n) ? __ldcg(l32 + j) : 0u;
      sv[u] = j < m ? __ldcg(sps + (R - 1) + j) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int j = base + u * nt;
      if (j < n) {
        const int r = j / gamma, o = r * gs + (j - r * gamma);
        stg[o] = c[u];
        if (l32 != nullptr) stgl[o] = cl[u];
      }
      if (j < m) spsv[j] = sv[u];
    }
  }
}

// Each request's survivals a_{r,j} = fl32(a_{r,j-1} c_{r,j}) from the staged
// confidences (clamped to [0, 1]; a non-finite one sets
// DSPARK_ERR_NONFINITE and counts as 0), written as keys, and the running
// sum along the row of fixed_point(a) (inclusive), both column-major with
// stride Rs. A row's survivals never increase along j (c <= 1), so each row
// of keys is sorted. Threads t = 0..nt-1 take part, one row each at a time.
__device__ __forceinline__ void survival_tables(const uint32_t* stg, int R, int gamma, int Rs, uint32_t* key,
                                                unsigned long long* fxc, uint32_t* status, int t, int nt) {
  constexpr int kU = 8;
  const int gs = sched_stage_stride(gamma);
  for (int r = t; r < R; r += nt) {
    const uint32_t* row = stg + r * gs;
    float acc = 1.f;
    unsigned long long run = 0ull;
    for (int j0 = 0; j0 < gamma; j0 += kU) {
      uint32_t cv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) cv[u] = j0 + u < gamma ? row[j0 + u] : 0u;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = j0 + u;
        if (j < gamma) {
          float c = __uint_as_float(cv[u]);
          if (!isfinite(c)) {
            set_status(status, DSPARK_ERR_NONFINITE);
            c = 0.f;
          }
          c = c > 0.f ? fminf(c, 1.f) : 0.f;
          acc = __fmul_rn(acc, c);
          key[j * Rs + r] = survival_key(acc);
          run += fixed_point(acc);
          fxc[j * Rs + r] = run;
        }
      }
    }
  }
}

// fixed_point(a) of candidate (r, j), from the running row sums.
__device__ __forceinline__ unsigned long long cand_fx(const unsigned long long* fxc, int Rs, int r, int j) {
  return fxc[j * Rs + r] - (j ? fxc[(j - 1) * Rs + r] : 0ull);
}

// Sorted position of candidate (r, j) (ascending key, ties by flat index
// r gamma + j) and the fixed-point sum of the survivals before it; every lane
// of the calling warp gets both. The rows are sorted, so row r' contributes
// the count of its entries before the candidate -- j for r' = r, else keys
// <= the candidate's for the rows before r (their equal keys have smaller
// flat indices) and keys < it for the rows after -- and the running sum of
// that many entries. Lane l counts rows l, l + 32, ..., four at a time, each
// with a branch-free binary search (steps of the powers of two up to gamma,
// the four rows' probes issued together); R log(gamma) steps per candidate.
__device__ __forceinline__ void rank_and_prefix(const uint32_t* key, const unsigned long long* fxc, int R, int gamma,
                                                int Rs, int r, int j, int lane, int& pos,
                                                unsigned long long& before_sum) {
  constexpr int kRows = 4;
  const uint32_t ki = key[j * Rs + r];
  const int top = 1 << (31 - __clz(gamma));
  int cnt = 0;
  unsigned long long sum = 0ull;
  for (int r0 = lane; r0 < R; r0 += 32 * kRows) {
    int c[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u) c[u] = 0;
    for (int step = top; step > 0; step >>= 1) {
      uint32_t kv[kRows];
#pragma unroll
      for (int u = 0; u < kRows; ++u) {
        const int rr = r0 + 32 * u, probe = c[u] + step;
        kv[u] = (rr < R && probe <= gamma) ? key[(probe - 1) * Rs + rr] : 0xFFFFFFFFu;
      }
#pragma unroll
      for (int u = 0; u < kRows; ++u) {
        const int rr = r0 + 32 * u, probe = c[u] + step;
        if (rr < R && probe <= gamma && (kv[u] < ki || (kv[u] == ki && rr < r))) c[u] = probe;
      }
    }
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const int rr = r0 + 32 * u;
      if (rr < R) {
        const int cc = rr == r ? j : c[u];
        cnt += cc;
        sum += cc ? fxc[(cc - 1) * Rs + rr] : 0ull;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    sum += __shfl_xor_sync(0xffffffffu, sum, o);
  }
  pos = cnt;
  before_sum = sum;
}

// Sum of every candidate's fixed-point survival (the rows' last running
// sums), reduced over the calling group (nt a multiple of 32) and returned to
// each of its threads. `red` holds one word per warp of the group;
// `group_sync` synchronises the group.
template <class Sync>
__device__ __forceinline__ unsigned long long survival_total(const unsigned long long* fxc, int R, int gamma, int Rs,
                                                             unsigned long long* red, int t, int nt,
                                                             Sync group_sync) {
  unsigned long long v = 0ull;
  for (int r = t; r < R; r += nt) v += fxc[(gamma - 1) * Rs + r];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  group_sync();
  if ((t & 31) == 0) red[t >> 5] = v;
  group_sync();
  v = 0ull;
  for (int w = 0; w < nt / 32; ++w) v += red[w];
  return v;
}

// ---------------------------------------------------------------------------
// The scheduler in one thread block (any block size that is a multiple of 32,
// up to 1024): survival keys, a stable LSD radix sort of (key, flat index)
// -- ties keep the flat order --, the exact fixed-point inclusive scan in
// sorted order, and the admission rule of the mode. Runs as its own launch
// for large problems and as one extra CTA of the drafting launch.

constexpr int kDigits = 16;
// Up to this many candidates the sort keys and indices live in shared memory.
constexpr int kSmemKeys = 8192;

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

// The one-block scheduler's sequential loops over a thread's segment read
// kBatch elements ahead of the dependent work: when the arrays live in the
// workspace (global memory, generic pointers the compiler cannot separate
// from the shared counters) each batch costs one memory round trip instead
// of one per element.
constexpr int kBatch = 8;

// Survival keys of one confidence matrix; flags non-finite entries.
// `stage` (n words) receives the confidences in one coalesced pass first.
inline __device__ void build_keys(const float* conf, int R, int gamma, uint32_t* key, uint32_t* idx,
                                  uint32_t* stage, uint32_t* status) {
  const int n = R * gamma;
  stage_smem(stage, reinterpret_cast<const uint32_t*>(conf), n);
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    float acc = 1.f;
    const size_t row = (size_t)r * gamma;
    for (int j0 = 0; j0 < gamma; j0 += kBatch) {
      uint32_t cb[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) cb[u] = j0 + u < gamma ? stage[row + j0 + u] : 0u;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = j0 + u;
        if (j < gamma) {
          float c = __uint_as_float(cb[u]);
          if (!isfinite(c)) {
            set_status(status, DSPARK_ERR_NONFINITE);
            c = 0.f;
          }
          c = c > 0.f ? fminf(c, 1.f) : 0.f;
          acc = __fmul_rn(acc, c);
          key[row + j] = survival_key(acc);
          idx[row + j] = (uint32_t)(row + j);
        }
      }
    }
  }
  __syncthreads();
}

// Stable LSD radix sort of (key, idx), 8 passes of 4 bits; result in key0/idx0.
inline __device__ void radix_sort(uint32_t* key0, uint32_t* idx0, uint32_t* key1, uint32_t* idx1, int n,
                                  uint32_t* cnt, unsigned long long* shu) {
  const int T = blockDim.x, tid = threadIdx.x;
  const int seg = ceil_div(n, T);
  const int s0 = min(n, tid * seg), s1 = min(n, s0 + seg);
  uint32_t *kin = key0, *iin = idx0, *kout = key1, *iout = idx1;
  for (int shift = 0; shift < 32; shift += 4) {
    for (int d = 0; d < kDigits; ++d) cnt[d * T + tid] = 0;
    for (int i0 = s0; i0 < s1; i0 += kBatch) {
      uint32_t kb[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) kb[u] = i0 + u < s1 ? kin[i0 + u] : 0u;
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (i0 + u < s1) cnt[((kb[u] >> shift) & 15u) * T + tid] += 1;
    }
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
    for (int i0 = s0; i0 < s1; i0 += kBatch) {
      uint32_t kb[kBatch], ib[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        kb[u] = i0 + u < s1 ? kin[i0 + u] : 0u;
        ib[u] = i0 + u < s1 ? iin[i0 + u] : 0u;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (i0 + u < s1) {
          const uint32_t slot = ((kb[u] >> shift) & 15u) * T + tid;
          const uint32_t pos = cnt[slot];
          cnt[slot] = pos + 1;
          kout[pos] = kb[u];
          iout[pos] = ib[u];
        }
      }
    }
    __syncthreads();
    uint32_t* t;
    t = kin; kin = kout; kout = t;
    t = iin; iin = iout; iout = t;
  }
}

// fx[i] = sum of fixed_point(a) over sorted positions 0..i.
inline __device__ void fixed_prefix(const uint32_t* key, int n, unsigned long long* fx,
                                    unsigned long long* shu) {
  const int T = blockDim.x, tid = threadIdx.x;
  const int seg = ceil_div(n, T);
  const int s0 = min(n, tid * seg), s1 = min(n, s0 + seg);
  unsigned long long loc = 0;
  for (int i0 = s0; i0 < s1; i0 += kBatch) {
    uint32_t kb[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) kb[u] = i0 + u < s1 ? key[i0 + u] : 0x3F800000u;  // survival 0
#pragma unroll
    for (int u = 0; u < kBatch; ++u) loc += fixed_point(key_survival(kb[u]));
  }
  unsigned long long tot;
  unsigned long long run = block_exscan_u64(loc, shu, tot);
  for (int i0 = s0; i0 < s1; i0 += kBatch) {
    uint32_t kb[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) kb[u] = i0 + u < s1 ? key[i0 + u] : 0x3F800000u;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      run += fixed_point(key_survival(kb[u]));
      if (i0 + u < s1) fx[i0 + u] = run;
    }
  }
  __syncthreads();
}

// Shared-memory scratch of schedule_block: kDigits * blockDim.x radix
// counters; the four key / index arrays (4 * kSmemKeys words) when
// R * gamma <= kSmemKeys, else null (they are then the global buffers
// passed in); 32-entry reduction scratch; one flag word.
struct BlockSchedScratch {
  uint32_t* cnt;
  uint32_t* keys;
  unsigned long long* shu;
  int* shi;
  double* shd;
  int* flag;
};

// Every thread of the block calls it. key0/key1/idx0/idx1 (u32[n]) are used
// when the keys do not fit shared memory; fx (u64[n]) receives the sorted
// prefix sums; status[0] the sticky status word.
inline __device__ void schedule_block(int R, int gamma, const float* __restrict__ conf,
                                      const float* __restrict__ conf_lag, const float* __restrict__ sps, int n_table,
                                      int mode, int32_t* __restrict__ L, int32_t* __restrict__ Kout,
                                      double* __restrict__ tau_theta, uint32_t* key0, uint32_t* key1, uint32_t* idx0,
                                      uint32_t* idx1, unsigned long long* fx, uint32_t* status,
                                      const BlockSchedScratch& sc) {
  uint32_t* cnt = sc.cnt;
  unsigned long long* shu = sc.shu;
  int* shi = sc.shi;
  double* shd = sc.shd;
  volatile int& sBad = *sc.flag;
  const int tid = threadIdx.x, T = blockDim.x;
  const int n = R * gamma;
  if (sc.keys != nullptr) {  // sort in shared memory
    uint32_t* sk = sc.keys;
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
    for (int i0 = s0; i0 < s1 && stop == 0x7fffffff; i0 += kBatch) {
      // prefix sums S_{i0-1} .. S_{i0+kBatch-1} and SPS(R + i0) .. SPS(R + i0 + kBatch), read together
      unsigned long long fb[kBatch + 1];
      float tb[kBatch + 1];
#pragma unroll
      for (int u = 0; u <= kBatch; ++u) {
        const int i = i0 + u - 1, B = R + i + 1;  // fb[u] = S_i, tb[u] = SPS[B - 1]
        fb[u] = (i >= 0 && i < s1) ? fx[i] : 0ull;
        tb[u] = (i < s1 && B >= 1 && B <= n_table) ? sps[B - 1] : 0.f;
      }
#pragma unroll
      for (int u = 1; u <= kBatch; ++u) {
        const int i = i0 + u - 1, B = R + i + 1;
        if (i < s1 && stop == 0x7fffffff) {
          bool st = B > n_table;
          if (!st) st = theta_of(R, fb[u], tb[u]) < theta_of(R, fb[u - 1], tb[u - 1]);
          if (st) stop = i;
        }
      }
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

// float64 bits -> unsigned key with the same order
__device__ __forceinline__ unsigned long long ordered_bits(double x) {
  const unsigned long long b = (unsigned long long)__double_as_longlong(x);
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

}  // namespace dspark
