// Sequential Markov-head drafting on CUDA cores (any dtype / rank / V).
//
// "DSpark: Aceleração da inferência de LLM com speculative decoding [pdf]"
// (GeekNews), "Geração semiautorregressiva": for block position k the
// sequential stage adds the transition bias B[prev] = W1[prev, :] . W2 of the
// low-rank Markov head to the parallel backbone's base logits, so token k is
// conditioned on the token sampled at k - 1 (the anchor at k = 1).
//
// Per step k two launches:
//   draft_partials: one CTA per (64-column chunk, 32 requests); the bias tile
//     is a float32 FMA dot product over the rank in index order; the epilogue
//     forms l = base + bias and writes per-(request, chunk) softmax partials
//     (m_c = max l, s_c = sum 2^((l - m_c) log2(e) / T)), or (max, argmax)
//     for greedy decoding.
//   draft_locate: one CTA per request; combines the chunk partials in float64
//     into Z, finds the chunk where u * Z falls, recomputes that chunk with the
//     same arithmetic and finds the token by a float64 prefix sum.
// This path serves float32 inputs and shapes the tensor-core path does not
// take; the bias dot-product order here (sequential over the rank) is also
// what the locate steps of every path recompute.
#include "common.cuh"
#include "internal.h"

namespace dspark {

constexpr int kRowsPerCta = 32;
constexpr int kKBlock = 32;

__device__ __forceinline__ int draft_prev(int k, int r, int gamma, int V, const int32_t* anchor,
                                          const int32_t* tokens, uint32_t* status) {
  int p = (k == 1) ? anchor[r] : tokens[(size_t)r * gamma + (k - 2)];
  if (p < 0 || p >= V) {
    set_status(status, DSPARK_ERR_RANGE);
    p = min(max(p, 0), V - 1);
  }
  return p;
}

// bias[v] for one previous token: float32 FMA in rank order from zero.
template <class Tin>
__device__ __forceinline__ float bias_dot(const Tin* W1, const Tin* W2, int prev, int rank, int V, int v) {
  float acc = 0.f;
  const size_t w1row = (size_t)prev * rank;
  for (int i = 0; i < rank; ++i) acc = __fmaf_rn(ld_elem(W1, w1row + i), ld_elem(W2, (size_t)i * V + v), acc);
  return acc;
}

template <class Tin>
__global__ void __launch_bounds__(256) draft_partials_kernel(
    int R, int gamma, int V, int rank, int k, const Tin* __restrict__ base,
    const int32_t* __restrict__ anchor, const int32_t* __restrict__ tokens,
    const Tin* __restrict__ W1, const Tin* __restrict__ W2, float kT, int greedy,
    float2* __restrict__ part, uint32_t* status) {
  __shared__ float sW1[kRowsPerCta][kKBlock + 1];
  __shared__ float sW2[kKBlock][kChunk];
  __shared__ int sPrev[kRowsPerCta];
  __shared__ float sRedV[kRowsPerCta][2];
  __shared__ int sRedI[kRowsPerCta][2];

  const int nc = ceil_div(V, kChunk);
  const int chunk = blockIdx.x, row0 = blockIdx.y * kRowsPerCta;
  const int tid = threadIdx.x, col = tid & 63, rg = tid >> 6, half = (tid >> 5) & 1;
  const int v = chunk * kChunk + col;

  if (tid < kRowsPerCta) {
    const int r = row0 + tid;
    sPrev[tid] = r < R ? draft_prev(k, r, gamma, V, anchor, tokens, status) : 0;
  }
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  __syncthreads();

  for (int kb = 0; kb < rank; kb += kKBlock) {
    for (int i = tid; i < kRowsPerCta * kKBlock; i += 256) {
      const int rr = i / kKBlock, kk = i % kKBlock;
      sW1[rr][kk] = (kb + kk < rank) ? ld_elem(W1, (size_t)sPrev[rr] * rank + kb + kk) : 0.f;
    }
    for (int i = tid; i < kKBlock * kChunk; i += 256) {
      const int kk = i / kChunk, cc = i % kChunk, vv = chunk * kChunk + cc;
      sW2[kk][cc] = (kb + kk < rank && vv < V) ? ld_elem(W2, (size_t)(kb + kk) * V + vv) : 0.f;
    }
    __syncthreads();
    const int kmax = min(kKBlock, rank - kb);
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
    const bool valid = (r < R) && (v < V);
    const float b = valid ? ld_elem(base, ((size_t)r * gamma + (k - 1)) * V + v) : 0.f;
    const float l = valid ? draft_logit(b, acc[i]) : -INFINITY;
    if (greedy) {
      float bv = l;
      int bi = valid ? v : 0x7fffffff;
      warp_argmax(bv, bi);
      if ((tid & 31) == 0) { sRedV[rl][half] = bv; sRedI[rl][half] = bi; }
      __syncthreads();
      if (col == 0 && r < R) {
        float v0 = sRedV[rl][0], v1 = sRedV[rl][1];
        int i0 = sRedI[rl][0], i1 = sRedI[rl][1];
        if (v1 > v0 || (v1 == v0 && i1 < i0)) { v0 = v1; i0 = i1; }
        part[(size_t)r * nc + chunk] = make_float2(v0, __int_as_float(i0));
      }
      __syncthreads();
    } else {
      const float mw = warp_max(l);
      if ((tid & 31) == 0) sRedV[rl][half] = mw;
      __syncthreads();
      const float mc = fmaxf(sRedV[rl][0], sRedV[rl][1]);
      const float w = valid ? draft_weight(b, acc[i], mc, kT) : 0.f;
      const float sw = warp_sum(w);
      __syncthreads();
      if ((tid & 31) == 0) sRedV[rl][half] = sw;
      __syncthreads();
      if (col == 0 && r < R) part[(size_t)r * nc + chunk] = make_float2(mc, sRedV[rl][0] + sRedV[rl][1]);
      __syncthreads();
    }
  }
}

// Combine the chunk partials of one request, draw the token by inverse CDF.
// Shared with the tensor-core path (same partial format).
template <class Tin>
__global__ void __launch_bounds__(256) draft_locate_kernel(
    int R, int gamma, int V, int rank, int k, const Tin* __restrict__ base,
    const int32_t* __restrict__ anchor, int32_t* __restrict__ tokens, const Tin* __restrict__ W1,
    const Tin* __restrict__ W2, float kT, int greedy, uint64_t seed,
    const float2* __restrict__ part, float* __restrict__ q_tok, float* __restrict__ q_stats,
    uint32_t* status) {
  __shared__ float shf[32];
  __shared__ int shi[32];
  __shared__ double shd[32];
  __shared__ float sW[kChunk];
  __shared__ double sExcl;
  __shared__ float sG;

  const int r = blockIdx.x, tid = threadIdx.x;
  const int nc = ceil_div(V, kChunk);
  const float2* pr = part + (size_t)r * nc;
  const size_t out = (size_t)r * gamma + (k - 1);

  if (greedy) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int c = tid; c < nc; c += blockDim.x) {
      const float2 p = pr[c];
      const int idx = __float_as_int(p.y);
      if (p.x > bv || (p.x == bv && idx < bi)) { bv = p.x; bi = idx; }
    }
    block_argmax(bv, bi, shf, shi);
    // The recorded maximum is the drafted token's logit with its bias summed in
    // float64 and rounded once, fl32(base + fl32(W1[prev] . W2[:, x])): the value
    // the greedy argmax is defined on (the float32 sums the argmax was taken over
    // can differ from it in the last bits). Every product of two float32 inputs
    // is exact in float64.
    const int x = min(max(bi, 0), V - 1);
    const int prev = draft_prev(k, r, gamma, V, anchor, tokens, status);
    double acc = 0.0;
    for (int i = tid; i < rank; i += blockDim.x)
      acc = fma((double)ld_elem(W1, (size_t)prev * rank + i), (double)ld_elem(W2, (size_t)i * V + x), acc);
    acc = warp_sum_d(acc);
    if ((tid & 31) == 0) shd[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
      double bias = 0.0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) bias += shd[w];
      tokens[out] = bi;
      q_tok[out] = 1.f;
      q_stats[2 * out] = __fadd_rn(ld_elem(base, ((size_t)r * gamma + (k - 1)) * V + x), __double2float_rn(bias));
      q_stats[2 * out + 1] = 1.f;
    }
    return;
  }

  float m = -INFINITY;
  for (int c = tid; c < nc; c += blockDim.x) m = fmaxf(m, pr[c].x);
  const float M = block_max(m, shf);

  // contiguous chunk segments per thread, float64 running sums in chunk order
  const int seg = ceil_div(nc, blockDim.x);
  const int c0 = min(nc, tid * seg), c1 = min(nc, c0 + seg);
  double local = 0.0;
  for (int c = c0; c < c1; ++c) {
    const float2 p = pr[c];
    local += (double)p.y * (double)exp2f(__fmul_rn(__fsub_rn(p.x, M), kT));
  }
  double Z;
  const double excl = block_exscan_d(local, shd, Z);
  const double u = philox_uniform(seed, (uint64_t)r, (uint64_t)k, kDraft);
  const double target = u * Z;

  int found = 0x7fffffff, last_pos = -1;
  double run = excl, found_excl = 0.0;
  float found_g = 0.f;
  for (int c = c0; c < c1; ++c) {
    const float2 p = pr[c];
    const float g = exp2f(__fmul_rn(__fsub_rn(p.x, M), kT));
    const double f = (double)p.y * (double)g;
    if (f > 0.0) last_pos = c;
    if (found == 0x7fffffff) {
      if (run + f > target) { found = c; found_excl = run; found_g = g; }
      run += f;
    }
  }
  int cstar = block_min_i(found, shi);
  if (found == cstar && cstar != 0x7fffffff) { sExcl = found_excl; sG = found_g; }
  bool fallback = false;
  if (cstar == 0x7fffffff) {  // rounding left no crossing: last chunk with mass
    cstar = max(0, block_max_i(last_pos, shi));
    fallback = true;
    if (tid == 0) {
      const float2 p = pr[cstar];
      sG = exp2f(__fmul_rn(__fsub_rn(p.x, M), kT));
      sExcl = 0.0;
    }
  }
  __syncthreads();

  const int prev = draft_prev(k, r, gamma, V, anchor, tokens, status);
  const float mc = pr[cstar].x;
  if (tid < kChunk) {
    const int v = cstar * kChunk + tid;
    float w = 0.f;
    if (v < V) {
      const float b = ld_elem(base, ((size_t)r * gamma + (k - 1)) * V + v);
      w = draft_weight(b, bias_dot(W1, W2, prev, rank, V, v), mc, kT);
    }
    sW[tid] = w;
  }
  __syncthreads();
  if (tid == 0) {
    const double g = (double)sG;
    int xc = -1;
    if (!fallback) {
      double run2 = sExcl;
      for (int c = 0; c < kChunk; ++c) {
        run2 += (double)sW[c] * g;
        if (run2 > target) { xc = c; break; }
      }
    }
    if (xc < 0) {
      for (int c = kChunk - 1; c >= 0; --c)
        if (sW[c] > 0.f) { xc = c; break; }
      if (xc < 0) xc = 0;
    }
    const int x = min(cstar * kChunk + xc, V - 1);
    tokens[out] = x;
    q_tok[out] = (float)((double)sW[xc] * g / Z);
    q_stats[2 * out] = M;
    q_stats[2 * out + 1] = (float)Z;
  }
}

template <class Tin>
static cudaError_t launch_draft_cc_t(const DraftArgs& a, cudaStream_t s, int& launches) {
  const WsLayout L = ws_layout(a.R, a.gamma, a.V);
  uint32_t* status = ws_at<uint32_t>(a.ws, L.status);
  float2* part = ws_at<float2>(a.ws, L.dpart);
  const int nc = ceil_div(a.V, kChunk);
  const int greedy = a.temperature == 0.f;
  const float kT = greedy ? 0.f : (float)(1.4426950408889634 / (double)a.temperature);
  const Tin* base = static_cast<const Tin*>(a.base);
  const Tin* W1 = static_cast<const Tin*>(a.W1);
  const Tin* W2 = static_cast<const Tin*>(a.W2);
  dim3 gp(nc, ceil_div(a.R, kRowsPerCta));
  for (int k = 1; k <= a.gamma; ++k) {
    draft_partials_kernel<Tin><<<gp, 256, 0, s>>>(a.R, a.gamma, a.V, a.rank, k, base, a.anchor,
                                                  a.tokens, W1, W2, kT, greedy, part, status);
    draft_locate_kernel<Tin><<<a.R, 256, 0, s>>>(a.R, a.gamma, a.V, a.rank, k, base, a.anchor,
                                                 a.tokens, W1, W2, kT, greedy, a.seed, part,
                                                 a.q_tok, a.q_stats, status);
    launches += 2;
  }
  return cudaGetLastError();
}

cudaError_t launch_draft_cuda_core(const DraftArgs& a, cudaStream_t s, int& launches) {
  if (a.dtype == DSPARK_BF16) return launch_draft_cc_t<__nv_bfloat16>(a, s, launches);
  return launch_draft_cc_t<float>(a, s, launches);
}

}  // namespace dspark
