// Device helpers of the prefix scheduler shared by its own kernels
// (schedule.cu) and by the scheduling phase that the drafting sweep runs at
// the end of a round (draft_persistent.cu): survival keys, the exact 2^-40
// fixed-point survivals, Theta = tau * SPS(B) in float64, and the counting
// rank of one candidate ("DSpark: Aceleração da inferência de LLM com
// speculative decoding [pdf]" (GeekNews), "Verificação com agendamento por
// confiança").
#pragma once

#include "common.cuh"

namespace dspark {

// Threads per candidate in the counting rank.
constexpr int kRankSplit = 16;

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

// The confidences are staged in `key` by one coalesced pass, then each row's
// running product overwrites them in place; fxc receives each row's running
// sum of fixed_point(a) (inclusive, along j). A row's survivals never increase
// along j (a_j = fl32(a_{j-1} c_j), c_j <= 1), so each row of keys is sorted.
// Threads t = 0..nt-1 take part; `group_sync` synchronises them.
template <class Sync>
__device__ void survival_keys_smem(const float* conf, int R, int gamma, uint32_t* key, unsigned long long* fxc,
                                   uint32_t* status, int t, int nt, Sync group_sync) {
  const int n = R * gamma;
  stage_smem(key, reinterpret_cast<const uint32_t*>(conf), n, t, nt);
  group_sync();
  for (int r = t; r < R; r += nt) {
    float acc = 1.f;
    unsigned long long run = 0ull;
    for (int j = 0; j < gamma; ++j) {
      float c = __uint_as_float(key[r * gamma + j]);
      if (!isfinite(c)) {
        set_status(status, DSPARK_ERR_NONFINITE);
        c = 0.f;
      }
      c = c > 0.f ? fminf(c, 1.f) : 0.f;
      acc = __fmul_rn(acc, c);
      key[r * gamma + j] = survival_key(acc);
      run += fixed_point(acc);
      fxc[r * gamma + j] = run;
    }
  }
}

// fixed_point(a) of candidate i, from the running row sums.
__device__ __forceinline__ unsigned long long cand_fx(const unsigned long long* fxc, int gamma, int i) {
  return fxc[i] - (i % gamma ? fxc[i - 1] : 0ull);
}

// Sorted position of candidate i = r gamma + j (ascending key, ties by flat
// index) and the fixed-point sum of the survivals before it; every thread of
// the kRankSplit-lane group that holds i gets both. The rows are sorted, so
// row r' contributes the count of its entries before i -- j for r' = r, else
// a binary search: keys <= i's for the rows before r (their equal keys have
// smaller flat indices), keys < i's for the rows after -- and the running sum
// of that many entries. R log(gamma) steps per candidate instead of R gamma.
__device__ __forceinline__ void rank_and_prefix(const uint32_t* key, const unsigned long long* fxc, int R, int gamma,
                                                int i, int s, int& pos, unsigned long long& before_sum) {
  i = min(i, R * gamma - 1);
  const int r = i / gamma, j = i - r * gamma;
  const uint32_t ki = key[i];
  int cnt = 0;
  unsigned long long sum = 0ull;
  for (int rr = s; rr < R; rr += kRankSplit) {
    int c = j;
    if (rr != r) {
      const uint32_t* row = key + rr * gamma;
      int lo = 0, hi = gamma;
      if (rr < r) {
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (row[mid] <= ki) lo = mid + 1;
          else hi = mid;
        }
      } else {
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (row[mid] < ki) lo = mid + 1;
          else hi = mid;
        }
      }
      c = lo;
    }
    cnt += c;
    sum += c ? fxc[rr * gamma + c - 1] : 0ull;
  }
#pragma unroll
  for (int o = kRankSplit / 2; o > 0; o >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    sum += __shfl_xor_sync(0xffffffffu, sum, o);
  }
  pos = cnt;
  before_sum = sum;
}

// float64 bits -> unsigned key with the same order
__device__ __forceinline__ unsigned long long ordered_bits(double x) {
  const unsigned long long b = (unsigned long long)__double_as_longlong(x);
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

}  // namespace dspark
