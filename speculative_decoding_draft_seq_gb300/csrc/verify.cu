// Lossless speculative-sampling verification ("DSpark: Aceleração da inferência
// de LLM com speculative decoding [pdf]" (GeekNews), "Definição do problema":
// the target checks the drafted block in one pass and rejection sampling keeps
// the longest prefix consistent with the target distribution; decoding-cycle
// paragraph: E and F accepted, G rejected, corrected token G* emitted).
//
// Launches (inside dspark_round on the tensor-core path, outside ALL mode, the
// row statistics and chains run in the drafting launch instead, with the same
// functions: verify_common.cuh):
//   verify_rows_warp_kernel  bf16 rows of a multiple of 8 elements in a
//                  16-byte aligned tensor: one CTA of eight warps per scheduled
//                  target row (r, k <= L_r), warp w streaming the row's w-th
//                  eighth (online max / sum of 2^((t - m) log2(e) / T)); the CTA
//                  combines the eight into (M, Z, argmax), and the CTA that
//                  combines a request's last row runs its chain of ratio tests
//                  u < p / q (p_tok = P_k(x_{k+1})), records the pending
//                  residual (first rejection j = A + 1) or bonus draw (row
//                  L_r = A), and stages the A row of the residual's Q_j.
//   verify_rows_kernel  any dtype or width (and the labels' statistics): one
//                  CTA per quarter row, the last quarter combining the four,
//                  the same chain.
//   gated_stage_kernel  (recurrent head only) the A row bf16(s_j), the state
//                  replayed over the anchor and the accepted tokens.
//   the residual / bonus draw: the tensor-core sweep in residual mode
//                  (draft_persistent.cu) or, for shapes it does not take,
//   resid_partials per (64-column chunk, 32 requests): residual weights
//                  max(0, P - Q) (Q recomputed with the Markov bias of the
//                  rejected position) or bonus weights P, chunk sums, and
//   resid_locate   one CTA per request: float64 scan of chunk sums, inverse
//                  CDF, recompute of the crossing chunk, emitted token.
#include <algorithm>

#include "common.cuh"
#include "verify_common.cuh"
#include "internal.h"

namespace dspark {

cudaError_t launch_resid_persistent(const VerifyArgs& a, cudaStream_t s, int& launches, bool& taken);
bool draft_tc_eligible(const DraftArgs& a);

constexpr int kRRows = 32;
constexpr int kRKBlock = 32;

template <class Tin>
__device__ __forceinline__ float bias_dot_v(const Tin* W1, const Tin* W2, int prev, int rank, int V, int v) {
  float acc = 0.f;
  const size_t w1row = (size_t)prev * rank;
  for (int i = 0; i < rank; ++i) acc = __fmaf_rn(ld_elem(W1, w1row + i), ld_elem(W2, (size_t)i * V + v), acc);
  return acc;
}

__device__ __forceinline__ float target_weight(float t, float m, float kT) {
  return exp2f(__fmul_rn(__fsub_rn(t, m), kT));
}

struct OnlineStat {
  float m = -INFINITY, s = 0.f, am = -INFINITY;
  int ai = 0x7fffffff;
  __device__ __forceinline__ void add1(float t, int v, float kT, bool greedy) {
    if (t > am) { am = t; ai = v; }
    if (greedy) return;
    if (t > m) {
      s = __fmul_rn(s, target_weight(m, t, kT));
      m = t;
    }
    s += target_weight(t, m, kT);
  }
};

// ---------------------------------------------------------------------------
// Target row statistics and the acceptance chain in one launch (rows a6, a7).
//
// Grid (R, gamma + 1, kVsSplit): CTA (r, k, s) streams the s-th quarter of
// target row k of request r (rows past L_r return at once) and writes its
// partial (max M_s, fixed-point sum Z_s of 2^((t - M_s) log2e/T) over its
// threads, argmax) to the workspace. The last CTA of a row (a per-row counter,
// reset by that CTA) combines the quarters: M = max M_s, Z = sum of the
// quarters' sums rescaled to M (each term rounded once in float32, summed as
// 2^-40 integers), the lowest-index argmax, and p(x_{k+1}). The last row of a
// request to be combined (a per-request counter) runs the request's chain: one
// warp tests the scheduled positions at once (u < p/q in float64), a ballot
// finds the first rejection, and the accepted tokens, the pending residual or
// bonus draw, and the zeroed p of unscheduled positions are written.
constexpr int kVsThreads = 256;

// One work item: quarter sp of target row k (<= L) of request r.
template <class Tin>
__device__ __forceinline__ void verify_row_item(
    int R, int gamma, int V, const Tin* __restrict__ target, const int32_t* __restrict__ tokens,
    const int32_t* __restrict__ anchor, const float* __restrict__ q_tok, float kT, int greedy, uint64_t seed,
    float4* vsplit, unsigned int* row_cnt, unsigned int* req_cnt, float4* rowstat, float* p_tok,
    int32_t* __restrict__ out, int32_t* __restrict__ acc_len, int4* __restrict__ pend, uint32_t* status,
    const Tin* __restrict__ W1, int rank, __nv_bfloat16* astage, int stats_only, int r, int k, int sp, int L,
    float* shf, int* shi, unsigned long long* shu, volatile int& sLast) {
  const int tid = threadIdx.x;
  const size_t rowi = (size_t)r * (gamma + 1) + k;
  const size_t row = rowi * V;
  float am, Ms = 0.f, Zs = 0.f;
  int ai;
  // 8-element groups by 16-byte loads: bf16 rows of a multiple of 8 elements in a 16-byte aligned tensor
  const bool fast = sizeof(Tin) == 2 && (V & 7) == 0 && (reinterpret_cast<uintptr_t>(target) & 15) == 0;
  if (fast) {  // eight 16-byte loads in flight per thread
    RowStat st;
    const uint4* p = reinterpret_cast<const uint4*>(target + row);
    const int ng = V >> 3, T = blockDim.x;
    const int gb = (int)(((long long)sp * ng) / kVsSplit), ge = (int)(((long long)(sp + 1) * ng) / kVsSplit);
    for (int g0 = gb + tid; g0 < ge; g0 += 8 * T) {
      uint4 q[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) q[u] = (g0 + u * T < ge) ? __ldcs(p + g0 + u * T) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (g0 + u * T >= ge) continue;
        if (greedy) st.add8_greedy(q[u], (g0 + u * T) * 8);
        else st.add8_sampled(q[u], kT);
      }
    }
    am = st.m;
    ai = st.ai;
    if (greedy) {
      block_argmax(am, ai, shf, shi);
    } else {
      Ms = block_max(st.m, shf);
      const float contrib = st.s > 0.f ? __fmul_rn(st.s, ex2_approx(__fmul_rn(__fsub_rn(st.m, Ms), kT))) : 0.f;
      unsigned long long v = fx40(contrib);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      __syncthreads();
      if ((tid & 31) == 0) shu[tid >> 5] = v;
      __syncthreads();
      unsigned long long Z = 0ull;
      for (int i = 0; i < (int)(blockDim.x >> 5); ++i) Z += shu[i];
      Zs = __fmul_rn((float)Z, 0x1p-40f);
      am = Ms;
      ai = 0;
    }
  } else {  // any dtype or width: one element at a time
    OnlineStat st;
    const int vb = (int)(((long long)sp * V) / kVsSplit), ve = (int)(((long long)(sp + 1) * V) / kVsSplit);
    for (int v = vb + tid; v < ve; v += blockDim.x) st.add1(ld_elem(target, row + v), v, kT, greedy);
    am = st.am;
    ai = st.ai;
    block_argmax(am, ai, shf, shi);
    if (!greedy) {
      Ms = block_max(st.m, shf);
      const float contrib = st.s > 0.f ? __fmul_rn(st.s, target_weight(st.m, Ms, kT)) : 0.f;
      unsigned long long v = fx40(contrib);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      __syncthreads();
      if ((tid & 31) == 0) shu[tid >> 5] = v;
      __syncthreads();
      unsigned long long Z = 0ull;
      for (int i = 0; i < (int)(blockDim.x >> 5); ++i) Z += shu[i];
      Zs = __fmul_rn((float)Z, 0x1p-40f);
    }
  }
  if (tid == 0) {
    __stcg(vsplit + rowi * kVsSplit + sp, make_float4(Ms, Zs, am, __int_as_float(ai)));
    __threadfence();
    sLast = atomicAdd(row_cnt + rowi, 1u) == (unsigned)(kVsSplit - 1);
  }
  __syncthreads();
  if (!sLast) return;

  if (tid == 0) {  // combine the row's quarters
    __threadfence();
    row_cnt[rowi] = 0u;
    float4 q[kVsSplit];
#pragma unroll
    for (int i = 0; i < kVsSplit; ++i) q[i] = __ldcg(vsplit + rowi * kVsSplit + i);
    float bv = q[0].z, M = q[0].x;
    int bi = __float_as_int(q[0].w);
#pragma unroll
    for (int i = 1; i < kVsSplit; ++i) {
      const int ii = __float_as_int(q[i].w);
      if (q[i].z > bv || (q[i].z == bv && ii < bi)) { bv = q[i].z; bi = ii; }
      M = fmaxf(M, q[i].x);
    }
    // the weight formula of the streaming pass that produced the quarters (`fast` above)
    auto wgt = [&](float t, float m) {
      return fast ? ex2_approx(__fmaf_rn(t, kT, -__fmul_rn(m, kT))) : target_weight(t, m, kT);
    };
    float Zf = 1.f;
    if (!greedy) {
      unsigned long long Z = 0ull;
#pragma unroll
      for (int i = 0; i < kVsSplit; ++i)
        if (q[i].y > 0.f) Z += fx40(__fmul_rn(q[i].y, fast ? ex2_approx(__fmul_rn(__fsub_rn(q[i].x, M), kT))
                                                              : target_weight(q[i].x, M, kT)));
      Zf = __fmul_rn((float)Z, 0x1p-40f);
    } else {
      M = 0.f;
    }
    __stcg(rowstat + rowi, make_float4(M, Zf, __int_as_float(bi), 0.f));
    if (stats_only) {
      sLast = 0;  // no p, no chain: the row stats are the whole result
    } else if (k < L) {
      int x = tokens[(size_t)r * gamma + k];
      if (x < 0 || x >= V) { set_status(status, DSPARK_ERR_RANGE); x = min(max(x, 0), V - 1); }
      float pv;
      if (greedy) pv = (x == bi) ? 1.f : 0.f;
      else pv = __fdiv_rn(wgt(ld_elem(target, row + x), M), Zf);
      __stcg(p_tok + (size_t)r * gamma + k, pv);
    }
    if (!stats_only) {
      __threadfence();
      sLast = atomicAdd(req_cnt + r, 1u) == (unsigned)L;  // rows 0..L of this request are combined
    }
  }
  __syncthreads();
  if (!sLast || tid >= 32) return;

  // the request's chain (warp 0)
  const int lane = tid;
  __threadfence();
  if (lane == 0) req_cnt[r] = 0u;
  int A = L;
  for (int k0 = 1; k0 <= L; k0 += 32) {
    const int kk = k0 + lane;
    bool fail = false;
    if (kk <= L) {
      const float pv = __ldcg(p_tok + (size_t)r * gamma + kk - 1);
      const float qv = q_tok[(size_t)r * gamma + kk - 1];
      const double u = philox_uniform(seed, (uint64_t)r, (uint64_t)kk, kAccept);
      fail = !((qv <= 0.f) || (u < (double)pv / (double)qv));
    }
    const unsigned m = __ballot_sync(0xffffffffu, fail);
    if (m) {  // the first rejected position k0 + ffs - 1 keeps A = k - 1 tokens
      A = k0 + __ffs(m) - 2;
      break;
    }
  }
  for (int kk = lane; kk <= gamma; kk += 32) {
    if (kk < A) out[(size_t)r * (gamma + 1) + kk] = tokens[(size_t)r * gamma + kk];
    else if (kk > A) out[(size_t)r * (gamma + 1) + kk] = -1;
    if (kk >= L && kk < gamma) p_tok[(size_t)r * gamma + kk] = 0.f;
  }
  if (lane == 0) {
    acc_len[r] = A;
    const int prev = A ? tokens[(size_t)r * gamma + A - 1] : anchor[r];
    if (greedy) {
      out[(size_t)r * (gamma + 1) + A] = __float_as_int(__ldcg(rowstat + (size_t)r * (gamma + 1) + A).z);
      pend[r] = make_int4(kPendNone, A, prev, A);
    } else {
      pend[r] = make_int4(A < L ? kPendResid : kPendBonus, A, prev, A);
    }
  }
  // The residual pass's A row of this request (rank > 0 only when the
  // tensor-core residual pass can run: bf16, rank a multiple of 64 up to 256,
  // W1 16-byte aligned): W1[prev] for a residual draw, zeros otherwise
  // (finite, so the MMA row is finite).
  if (rank > 0 && !greedy && 8 * lane < rank) {
    const int prev = min(max(A ? tokens[(size_t)r * gamma + A - 1] : anchor[r], 0), V - 1);
    const uint4 w = A < L ? __ldg(reinterpret_cast<const uint4*>(W1 + (size_t)prev * rank) + lane)
                          : make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(astage + (size_t)r * rank)[lane] = w;
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
}

// One CTA per item. Grid (kVsSplit, R, gamma + 1): the quarters of a row are
// launched together (the row combines sooner) and the small k, which are the
// scheduled rows, first.
template <class Tin>
__global__ void __launch_bounds__(kVsThreads) verify_rows_kernel(
    int R, int gamma, int V, const Tin* __restrict__ target, const int32_t* __restrict__ tokens,
    const int32_t* __restrict__ anchor, const float* __restrict__ q_tok, const int32_t* __restrict__ sched_len,
    float kT, int greedy, uint64_t seed, float4* vsplit, unsigned int* row_cnt, unsigned int* req_cnt,
    float4* rowstat, float* p_tok, int32_t* __restrict__ out, int32_t* __restrict__ acc_len,
    int4* __restrict__ pend, uint32_t* status, const Tin* __restrict__ W1, int rank, __nv_bfloat16* astage,
    int stats_only) {
  __shared__ float shf[32];
  __shared__ int shi[32];
  __shared__ unsigned long long shu[32];
  __shared__ int sLast;
  const int sp = blockIdx.x, r = blockIdx.y, k = blockIdx.z;
  // stats only (acceptance labels): rows 0..gamma-1 of every request
  const int L = stats_only ? gamma - 1 : min(max(sched_len[r], 0), gamma);
  if (k > L) return;
  verify_row_item<Tin>(R, gamma, V, target, tokens, anchor, q_tok, kT, greedy, seed, vsplit, row_cnt, req_cnt,
                       rowstat, p_tok, out, acc_len, pend, status, W1, rank, astage, stats_only, r, k, sp, L, shf,
                       shi, shu, sLast);
}

// bf16 target rows with V % 8 == 0, 16-byte aligned: one CTA of kVwSplit
// warps per scheduled row (grid (R, gamma + 1), the low k first), warp w
// streaming piece w, thread 0 combining the pieces; the CTA that combines a
// request's last row runs the request's chain. The pieces, their combination
// and the chain are those of the drafting launch's verification work
// (verify_common.cuh), so both give the same bits.
__global__ void __launch_bounds__(32 * kVwSplit) verify_rows_warp_kernel(
    int R, int gamma, int V, const __nv_bfloat16* __restrict__ target, const int32_t* tokens,
    const int32_t* __restrict__ anchor, const float* __restrict__ q_tok, const int32_t* __restrict__ sched_len,
    float kT, int greedy, uint64_t seed, unsigned int* req_cnt, float4* rowstat, float* p_tok,
    int32_t* __restrict__ out, int32_t* __restrict__ acc_len, int4* __restrict__ pend, uint32_t* status,
    const __nv_bfloat16* __restrict__ W1, int stage_rank, __nv_bfloat16* astage) {
  __shared__ float4 sPiece[kVwSplit];
  __shared__ int sLast;
  const int r = blockIdx.x, k = blockIdx.y;
  const int L = min(max(sched_len[r], 0), gamma);
  if (k > L) return;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t rowi = (size_t)r * (gamma + 1) + k;
  const float4 part = warp_row_piece(target, rowi, V, w, kT, greedy, lane);
  if (lane == 0) sPiece[w] = part;
  __syncthreads();
  if (threadIdx.x == 0) {
    float4 q[kVwSplit];
#pragma unroll
    for (int i = 0; i < kVwSplit; ++i) q[i] = sPiece[i];
    __stcg(rowstat + rowi, combine_row_pieces(q, kT, greedy));
    __threadfence();
    sLast = atomicAdd(req_cnt + r, 1u) == (unsigned)L;  // rows 0..L of this request are combined
  }
  __syncthreads();
  if (!sLast || threadIdx.x >= 32) return;
  __threadfence();
  if (lane == 0) req_cnt[r] = 0u;
  request_chain(r, gamma, V, target, tokens, anchor, q_tok, kT, greedy, seed, rowstat, p_tok, out, acc_len, pend,
                status, W1, stage_rank, astage, L, lane);
}

// Residual (or bonus) weight of one entry, with explicit rounding so the
// partials and the locate recompute agree bit for bit.
__device__ __forceinline__ float resid_weight(int kind, float t, float MP, float ZP, float b, float bias,
                                              float MQ, float ZQ, float kT) {
  const float P = __fdiv_rn(target_weight(t, MP, kT), ZP);
  if (kind == kPendBonus) return P;
  const float Q = __fdiv_rn(draft_weight(b, bias, MQ, kT), ZQ);
  return fmaxf(0.f, __fsub_rn(P, Q));
}

template <class Tin>
__global__ void __launch_bounds__(256) resid_partials_kernel(
    int R, int gamma, int V, int rank, const Tin* __restrict__ target, const Tin* __restrict__ base,
    const Tin* __restrict__ W1, const Tin* __restrict__ W2, const float* __restrict__ q_stats,
    const float4* __restrict__ rowstat, const int4* __restrict__ pend, float kT,
    float2* __restrict__ rpart) {
  __shared__ float sW1[kRRows][kRKBlock + 1];
  __shared__ float sW2[kRKBlock][kChunk];
  __shared__ int4 sPend[kRRows];
  __shared__ float sRed[kRRows][2][2];
  __shared__ int sAny;
  const int nc = ceil_div(V, kChunk);
  const int chunk = blockIdx.x, row0 = blockIdx.y * kRRows;
  const int tid = threadIdx.x, col = tid & 63, rg = tid >> 6, half = (tid >> 5) & 1;
  const int v = chunk * kChunk + col;
  if (tid == 0) sAny = 0;
  __syncthreads();
  if (tid < kRRows) {
    const int r = row0 + tid;
    int4 pd = r < R ? pend[r] : make_int4(kPendNone, 0, 0, 0);
    sPend[tid] = pd;
    if (pd.x != kPendNone) atomicOr(&sAny, 1);
  }
  __syncthreads();
  if (!sAny) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int kb = 0; kb < rank; kb += kRKBlock) {
    for (int i = tid; i < kRRows * kRKBlock; i += 256) {
      const int rr = i / kRKBlock, kk = i % kRKBlock;
      sW1[rr][kk] = (kb + kk < rank) ? ld_elem(W1, (size_t)sPend[rr].z * rank + kb + kk) : 0.f;
    }
    for (int i = tid; i < kRKBlock * kChunk; i += 256) {
      const int kk = i / kChunk, cc = i % kChunk, vv = chunk * kChunk + cc;
      sW2[kk][cc] = (kb + kk < rank && vv < V) ? ld_elem(W2, (size_t)(kb + kk) * V + vv) : 0.f;
    }
    __syncthreads();
    const int kmax = min(kRKBlock, rank - kb);
    for (int kk = 0; kk < kmax; ++kk) {
      const float w2 = sW2[kk][col];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(sW1[rg * 8 + i][kk], w2, acc[i]);
    }
    __syncthreads();
  }
#pragma unroll 1
  for (int i = 0; i < 8; ++i) {
    const int rl = rg * 8 + i, r = row0 + rl;
    const int4 pd = sPend[rl];
    const bool valid = (r < R) && (v < V) && pd.x != kPendNone;
    float w = 0.f, pw = 0.f;
    if (valid) {
      const int A = pd.y;
      const float4 rs = rowstat[(size_t)r * (gamma + 1) + A];
      const float t = ld_elem(target, ((size_t)r * (gamma + 1) + A) * V + v);
      pw = __fdiv_rn(target_weight(t, rs.x, kT), rs.y);
      if (pd.x == kPendBonus) {
        w = pw;
      } else {
        const float b = ld_elem(base, ((size_t)r * gamma + A) * V + v);
        const float MQ = q_stats[2 * ((size_t)r * gamma + A)], ZQ = q_stats[2 * ((size_t)r * gamma + A) + 1];
        w = resid_weight(kPendResid, t, rs.x, rs.y, b, acc[i], MQ, ZQ, kT);
      }
    }
    const float sw = warp_sum(w), sp = warp_sum(pw);
    if ((tid & 31) == 0) { sRed[rl][half][0] = sw; sRed[rl][half][1] = sp; }
    __syncthreads();
    if (col == 0 && r < R && pd.x != kPendNone)
      rpart[(size_t)r * nc + chunk] = make_float2(sRed[rl][0][0] + sRed[rl][1][0], sRed[rl][0][1] + sRed[rl][1][1]);
    __syncthreads();
  }
}

template <class Tin>
__global__ void __launch_bounds__(256) resid_locate_kernel(
    int R, int gamma, int V, int rank, const Tin* __restrict__ target, const Tin* __restrict__ base,
    const Tin* __restrict__ W1, const Tin* __restrict__ W2, const float* __restrict__ q_stats,
    const float4* __restrict__ rowstat, const int4* __restrict__ pend, float kT, uint64_t seed,
    const float2* __restrict__ rpart, int32_t* __restrict__ out) {
  __shared__ int shi[32];
  __shared__ double shd[32];
  __shared__ float sW[kChunk];
  __shared__ double sExcl;
  const int r = blockIdx.x, tid = threadIdx.x;
  const int4 pd = pend[r];
  if (pd.x == kPendNone) return;
  const int nc = ceil_div(V, kChunk);
  const float2* pr = rpart + (size_t)r * nc;
  const int A = pd.y;
  const int seg = ceil_div(nc, blockDim.x);
  const int c0 = min(nc, tid * seg), c1 = min(nc, c0 + seg);

  double loc_res = 0.0;
  for (int c = c0; c < c1; ++c) loc_res += (double)pr[c].x;
  double W;
  double excl = block_exscan_d(loc_res, shd, W);
  int use_p = 0;
  if (!(W > 0.0)) {  // empty residual under rounding: draw from P instead
    use_p = 1;
    double loc_p = 0.0;
    for (int c = c0; c < c1; ++c) loc_p += (double)pr[c].y;
    excl = block_exscan_d(loc_p, shd, W);
  }
  const uint64_t purpose = pd.x == kPendResid ? kResid : kBonus;
  const double u = philox_uniform(seed, (uint64_t)r, (uint64_t)(A + 1), purpose);
  const double target_v = u * W;

  int found = 0x7fffffff, last_pos = -1;
  double run = excl, found_excl = 0.0;
  for (int c = c0; c < c1; ++c) {
    const double f = (double)(use_p ? pr[c].y : pr[c].x);
    if (f > 0.0) last_pos = c;
    if (found == 0x7fffffff) {
      if (run + f > target_v) { found = c; found_excl = run; }
      run += f;
    }
  }
  int cstar = block_min_i(found, shi);
  if (found == cstar && cstar != 0x7fffffff) sExcl = found_excl;
  bool fallback = false;
  if (cstar == 0x7fffffff) {
    cstar = max(0, block_max_i(last_pos, shi));
    fallback = true;
  }
  __syncthreads();
  const int kind = use_p ? kPendBonus : pd.x;
  const float4 rs = rowstat[(size_t)r * (gamma + 1) + A];
  if (tid < kChunk) {
    const int v = cstar * kChunk + tid;
    float w = 0.f;
    if (v < V) {
      const float t = ld_elem(target, ((size_t)r * (gamma + 1) + A) * V + v);
      if (kind == kPendBonus) {
        w = resid_weight(kPendBonus, t, rs.x, rs.y, 0.f, 0.f, 0.f, 1.f, kT);
      } else {
        const float b = ld_elem(base, ((size_t)r * gamma + A) * V + v);
        const float MQ = q_stats[2 * ((size_t)r * gamma + A)], ZQ = q_stats[2 * ((size_t)r * gamma + A) + 1];
        w = resid_weight(kPendResid, t, rs.x, rs.y, b, bias_dot_v(W1, W2, pd.z, rank, V, v), MQ, ZQ, kT);
      }
    }
    sW[tid] = w;
  }
  __syncthreads();
  if (tid == 0) {
    int xc = -1;
    if (!fallback) {
      double run2 = sExcl;
      for (int c = 0; c < kChunk; ++c) {
        run2 += (double)sW[c];
        if (run2 > target_v) { xc = c; break; }
      }
    }
    if (xc < 0) {
      for (int c = kChunk - 1; c >= 0; --c)
        if (sW[c] > 0.f) { xc = c; break; }
      if (xc < 0) xc = 0;
    }
    out[(size_t)r * (gamma + 1) + A] = min(cstar * kChunk + xc, V - 1);
  }
}

// Recurrent (gated) head: the A row of request r's residual draw at the
// first rejected position j = A + 1 is bf16(s_j), s_j the state after the
// anchor and the accepted tokens x_1..x_A (the same float32 recurrence as the
// drafting kernel); zeros for a bonus draw. One CTA per request, one thread
// per state element; the gate and W1 rows of eight positions are loaded
// together.
__global__ void __launch_bounds__(256) gated_stage_kernel(int R, int gamma, int V, int rank,
                                                          const int32_t* __restrict__ anchor,
                                                          const int32_t* __restrict__ tokens,
                                                          const __nv_bfloat16* __restrict__ W1,
                                                          const __nv_bfloat16* __restrict__ gate,
                                                          const int4* __restrict__ pend,
                                                          __nv_bfloat16* astage) {
  __shared__ int sPrev[8];
  const int r = blockIdx.x, e = threadIdx.x;
  const int4 pd = pend[r];
  const bool resid = pd.x == kPendResid;
  const int A = resid ? min(max(pd.w, 0), gamma - 1) : -1;
  float st = 0.f;
  for (int i0 = 0; i0 <= A; i0 += 8) {
    __syncthreads();
    if (e < 8 && i0 + e <= A) {
      const int t = i0 + e == 0 ? anchor[r] : tokens[(size_t)r * gamma + i0 + e - 1];
      sPrev[e] = min(max(t, 0), V - 1);
    }
    __syncthreads();
    if (e < rank) {
      float z[8], w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const bool ok = i0 + u <= A;
        const size_t o = (size_t)(ok ? sPrev[u] : 0) * rank + e;
        z[u] = ok ? ld_elem(gate, o) : 0.f;
        w[u] = ok ? ld_elem(W1, o) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + u <= A) st = __fadd_rn(__fmul_rn(__fsub_rn(1.f, z[u]), st), __fmul_rn(z[u], w[u]));
    }
  }
  if (e < rank) astage[(size_t)r * rank + e] = resid ? __float2bfloat16_rn(st) : __float2bfloat16_rn(0.f);
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The residual / bonus draw (and, for the gated head, its A rows) once the
// chains have run.
template <class Tin>
static cudaError_t launch_verify_tail_t(const VerifyArgs& a, cudaStream_t s, int& launches) {
  if (a.temperature == 0.f) return cudaGetLastError();  // greedy: the chain emitted the tokens
  const WsLayout L = ws_layout(a.R, a.gamma, a.V);
  void* ws = a.ws;
  const float kT = (float)(1.4426950408889634 / (double)a.temperature);
  if (a.gate) {
    gated_stage_kernel<<<a.R, 256, 0, s>>>(a.R, a.gamma, a.V, a.rank, a.anchor, a.tokens,
                                           static_cast<const __nv_bfloat16*>(a.W1),
                                           static_cast<const __nv_bfloat16*>(a.gate), ws_at<int4>(ws, L.pend),
                                           ws_at<__nv_bfloat16>(ws, L.astage));
    launches += 1;
  }
  bool taken = false;
  cudaError_t e = launch_resid_persistent(a, s, launches, taken);
  if (taken || e != cudaSuccess) return e == cudaSuccess ? cudaGetLastError() : e;
  // the fallback kernels below recompute the Markov bias; the gated head
  // was admitted only where the tensor-core pass runs
  if (a.gate) return cudaErrorNotSupported;
  const int nc = ceil_div(a.V, kChunk);
  const Tin* target = static_cast<const Tin*>(a.target);
  const Tin* base = static_cast<const Tin*>(a.base);
  const Tin* W1 = static_cast<const Tin*>(a.W1);
  const Tin* W2 = static_cast<const Tin*>(a.W2);
  float4* rowstat = ws_at<float4>(ws, L.rowstat);
  int4* pend = ws_at<int4>(ws, L.pend);
  float2* rpart = ws_at<float2>(ws, L.rpart);
  resid_partials_kernel<Tin><<<dim3(nc, ceil_div(a.R, kRRows)), 256, 0, s>>>(
      a.R, a.gamma, a.V, a.rank, target, base, W1, W2, a.q_stats, rowstat, pend, kT, rpart);
  resid_locate_kernel<Tin><<<a.R, 256, 0, s>>>(a.R, a.gamma, a.V, a.rank, target, base, W1, W2, a.q_stats,
                                               rowstat, pend, kT, a.seed, rpart, a.out_tokens);
  launches += 2;
  return cudaGetLastError();
}

template <class Tin>
static cudaError_t launch_verify_t(const VerifyArgs& a, cudaStream_t s, int& launches) {
  const WsLayout L = ws_layout(a.R, a.gamma, a.V);
  void* ws = a.ws;
  const int greedy = a.temperature == 0.f;
  const float kT = greedy ? 0.f : (float)(1.4426950408889634 / (double)a.temperature);
  // the chain stages W1[prev] for the Markov head; the gated head's rows come next
  const int stage_rank = (sizeof(Tin) == 2 && !a.gate && a.rank % 64 == 0 && a.rank <= 256 &&
                          (reinterpret_cast<uintptr_t>(a.W1) & 15) == 0) ? a.rank : 0;
  if (sizeof(Tin) == 2 && (a.V & 7) == 0 && (reinterpret_cast<uintptr_t>(a.target) & 15) == 0) {
    verify_rows_warp_kernel<<<dim3(a.R, a.gamma + 1), 32 * kVwSplit, 0, s>>>(
        a.R, a.gamma, a.V, static_cast<const __nv_bfloat16*>(a.target), a.tokens, a.anchor, a.q_tok, a.sched_len,
        kT, greedy, a.seed, ws_at<unsigned int>(ws, L.vcount) + (size_t)a.R * (a.gamma + 1),
        ws_at<float4>(ws, L.rowstat), a.p_tok, a.out_tokens, a.accepted_len, ws_at<int4>(ws, L.pend),
        ws_at<uint32_t>(ws, L.status), static_cast<const __nv_bfloat16*>(a.W1), stage_rank,
        ws_at<__nv_bfloat16>(ws, L.astage));
    launches += 1;
    return launch_verify_tail_t<Tin>(a, s, launches);
  }
  verify_rows_kernel<Tin><<<dim3(kVsSplit, a.R, a.gamma + 1), kVsThreads, 0, s>>>(
      a.R, a.gamma, a.V, static_cast<const Tin*>(a.target), a.tokens, a.anchor, a.q_tok, a.sched_len, kT, greedy,
      a.seed, ws_at<float4>(ws, L.vsplit), ws_at<unsigned int>(ws, L.vcount),
      ws_at<unsigned int>(ws, L.vcount) + (size_t)a.R * (a.gamma + 1), ws_at<float4>(ws, L.rowstat), a.p_tok,
      a.out_tokens, a.accepted_len, ws_at<int4>(ws, L.pend), ws_at<uint32_t>(ws, L.status),
      static_cast<const Tin*>(a.W1), stage_rank, ws_at<__nv_bfloat16>(ws, L.astage), 0);
  launches += 1;
  return launch_verify_tail_t<Tin>(a, s, launches);
}

// ---------------------------------------------------------------------------
// Acceptance labels of the confidence head ([GN] "Confidence head"): for every
// request r and position k, c*_k = 1 - TV(P_{k-1}, Q_k) = 1 - sum_v max(0,
// P_{k-1}(v) - Q_k(v)). The sampled form is one stats-only pass of
// verify_rows_kernel over target rows 0..gamma-1, the staging of each pair's
// W1[prev] row, and the sweep in label mode (tensor cores); the greedy form is
// argmax agreement (the drafted token is the drafter's argmax).

cudaError_t launch_label_persistent(const LabelArgs& a, cudaStream_t s, int& launches, bool& taken);

// One warp per (request, position) pair: W1[prev] (prev = the anchor at k = 1,
// else token k - 1) into the pair's staging row; 16 bytes per lane.
__global__ void __launch_bounds__(256) label_stage_kernel(int R, int gamma, int V, int rank,
                                                          const __nv_bfloat16* __restrict__ W1,
                                                          const int32_t* __restrict__ anchor,
                                                          const int32_t* __restrict__ tokens,
                                                          __nv_bfloat16* __restrict__ lstage, uint32_t* status) {
  const int pr = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  if (pr >= R * gamma) return;
  const int r = pr / gamma, k1 = pr - r * gamma;
  int prev = k1 == 0 ? anchor[r] : tokens[(size_t)r * gamma + k1 - 1];
  if (prev < 0 || prev >= V) {
    if (lane == 0) set_status(status, DSPARK_ERR_RANGE);
    prev = min(max(prev, 0), V - 1);
  }
  if (8 * lane < rank)
    reinterpret_cast<uint4*>(lstage + (size_t)pr * rank)[lane] =
        __ldg(reinterpret_cast<const uint4*>(W1 + (size_t)prev * rank) + lane);
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__global__ void label_greedy_kernel(int R, int gamma, const int32_t* __restrict__ tokens,
                                    const float4* __restrict__ rowstat, float* __restrict__ labels) {
  const int pr = blockIdx.x * blockDim.x + threadIdx.x;
  if (pr >= R * gamma) return;
  const int r = pr / gamma, k1 = pr - r * gamma;
  const int tgt = __float_as_int(rowstat[(size_t)r * (gamma + 1) + k1].z);
  labels[pr] = tokens[pr] == tgt ? 1.f : 0.f;
}

template <class Tin>
static cudaError_t launch_labels_t(const LabelArgs& a, cudaStream_t s, int& launches, bool& supported) {
  const WsLayout L = ws_layout(a.R, a.gamma, a.V);
  void* ws = a.ws;
  const int greedy = a.temperature == 0.f;
  supported = true;
  if (!greedy) {  // the sampled form runs on the tensor-core path only
    DraftArgs d{a.R, a.gamma, a.V, a.rank, a.dtype, a.base, a.anchor, a.W1, a.W2, a.temperature, 0,
                nullptr, nullptr, nullptr, a.ws};
    if (sizeof(Tin) != 2 || !draft_tc_eligible(d) || (reinterpret_cast<uintptr_t>(a.target) & 15) != 0) {
      supported = false;
      return cudaSuccess;
    }
  }
  const float kT = greedy ? 0.f : (float)(1.4426950408889634 / (double)a.temperature);
  uint32_t* status = ws_at<uint32_t>(ws, L.status);
  float4* rowstat = ws_at<float4>(ws, L.rowstat);
  const Tin* target = static_cast<const Tin*>(a.target);
  const Tin* W1 = static_cast<const Tin*>(a.W1);
  // row stats of target rows 0..gamma-1 (stats only: no p, no chains)
  verify_rows_kernel<Tin><<<dim3(kVsSplit, a.R, a.gamma), kVsThreads, 0, s>>>(
      a.R, a.gamma, a.V, target, a.tokens, a.anchor, nullptr, nullptr, kT, greedy, 0,
      ws_at<float4>(ws, L.vsplit), ws_at<unsigned int>(ws, L.vcount), ws_at<unsigned int>(ws, L.vcount) + (size_t)a.R * (a.gamma + 1),
      rowstat, nullptr, nullptr, nullptr, nullptr, status, W1, 0, nullptr, 1);
  launches += 1;
  const int n_pairs = a.R * a.gamma;
  if (greedy) {
    label_greedy_kernel<<<ceil_div(n_pairs, 256), 256, 0, s>>>(a.R, a.gamma, a.tokens, rowstat, a.labels);
    launches += 1;
    return cudaGetLastError();
  }
  label_stage_kernel<<<ceil_div(n_pairs, 8), 256, 0, s>>>(a.R, a.gamma, a.V, a.rank,
                                                          static_cast<const __nv_bfloat16*>(a.W1), a.anchor,
                                                          a.tokens, ws_at<__nv_bfloat16>(ws, L.lstage), status);
  launches += 1;
  bool taken = false;
  cudaError_t e = launch_label_persistent(a, s, launches, taken);
  if (e != cudaSuccess) return e;
  if (!taken) supported = false;
  return cudaGetLastError();
}

cudaError_t launch_labels(const LabelArgs& a, cudaStream_t s, int& launches, bool& supported) {
  if (a.dtype == DSPARK_BF16) return launch_labels_t<__nv_bfloat16>(a, s, launches, supported);
  return launch_labels_t<float>(a, s, launches, supported);
}

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s, int& launches) {
  if (a.dtype == DSPARK_BF16) return launch_verify_t<__nv_bfloat16>(a, s, launches);
  return launch_verify_t<float>(a, s, launches);
}

cudaError_t launch_verify_tail(const VerifyArgs& a, cudaStream_t s, int& launches) {
  if (a.dtype == DSPARK_BF16) return launch_verify_tail_t<__nv_bfloat16>(a, s, launches);
  return launch_verify_tail_t<float>(a, s, launches);
}

}  // namespace dspark
