// Shared device/host helpers of the DSpark GB300 library: workspace layout,
// status word, input loaders, the Philox4x64-10 uniform and block reductions.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <math.h>

#include "../../include/dspark.h"

namespace dspark {

// Columns per vocabulary chunk: the unit of the per-(row, chunk) softmax
// partials that the sampling locate step scans.
constexpr int kChunk = 64;

inline __host__ __device__ int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }
inline __host__ __device__ size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Pieces each target row is split into by the row-stats pass (one CTA each).
constexpr int kVsSplit = 4;
// Pieces per target row in the drafting launch's row statistics (a warp each).
constexpr int kVsPieceMax = 8;

// Per-request pending draw of the verifier (residual or bonus).
enum PendKind : int { kPendNone = 0, kPendResid = 1, kPendBonus = 2 };

// Byte offsets of the workspace sections.
struct WsLayout {
  size_t status;   // u32[64]: [0] sticky status, [1..] counters
  size_t dpart;    // float2 [R][n_chunks]   draft chunk partials (m, s) or (max, idx)
  size_t rowstat;  // float4 [R][gamma+1]    target row stats (M, Z, argmax, unused)
  size_t pend;     // int4   [R]             (kind, target row, prev token, accepted)
  size_t rpart;    // float2 [R][n_chunks]   residual chunk partials (sum res, sum P)
  size_t astage;   // bf16   [2][R][rank]    W1 rows of the drafted tokens, by step parity (rank <= 256)
  size_t gcarry;   // float  [R][256]        gated head: float32 state of each request between steps
  size_t vsplit;   // float4 [R][gamma+1][kVsPieceMax] target row piece stats (M_s, Z_s, max, argmax)
  size_t vlist;    // u32    [R*(gamma+1)]   the scheduled target rows, listed by the drafting launch
  size_t vcount;   // u32    [R*(gamma+1) + R] row / request completion counters (zero between calls)
  size_t lstage;   // bf16   [R*gamma][256]  acceptance labels: W1 rows of every (request, position)
  size_t lsum;     // u64    [R*gamma]       acceptance labels: 2^-40 sums of max(0, P - Q) (zero between calls)
  size_t skey0, skey1, sidx0, sidx1;  // u32 [R*gamma] radix-sort ping-pong
  size_t fx;       // u64 [R*gamma]         fixed-point survivals / prefix sums in sorted order
  size_t fx2;      // u64 [R*gamma]         the same for the lagged confidences
  size_t total;
};

// Every section whose size does not depend on V comes first, so that the
// scheduler (which lays the workspace out with V = 1) and the drafting and
// verification calls (the real V) agree on all of them; the two V-sized
// partial arrays come last.
inline __host__ __device__ WsLayout ws_layout(int R, int gamma, int V) {
  WsLayout L;
  const size_t nc = (size_t)ceil_div(V, kChunk);
  const size_t n = (size_t)R * (size_t)gamma > 0 ? (size_t)R * (size_t)gamma : 1;
  size_t o = 0;
  L.status = o;  o = align256(o + 64 * sizeof(uint32_t));
  L.vcount = o;  o = align256(o + ((size_t)R * (gamma + 1) + R) * sizeof(uint32_t));
  L.rowstat = o; o = align256(o + (size_t)R * (gamma + 1) * sizeof(float4));
  L.pend = o;    o = align256(o + (size_t)R * sizeof(int4));
  L.astage = o;  o = align256(o + (size_t)2 * R * 256 * 2);
  L.gcarry = o;  o = align256(o + (size_t)R * 256 * sizeof(float));
  L.vsplit = o;  o = align256(o + (size_t)R * (gamma + 1) * kVsPieceMax * sizeof(float4));
  L.vlist = o;   o = align256(o + (size_t)R * (gamma + 1) * sizeof(uint32_t));
  L.lstage = o;  o = align256(o + (size_t)R * gamma * 256 * 2);
  L.lsum = o;    o = align256(o + (size_t)R * gamma * sizeof(unsigned long long));
  L.skey0 = o;   o = align256(o + n * sizeof(uint32_t));
  L.skey1 = o;   o = align256(o + n * sizeof(uint32_t));
  L.sidx0 = o;   o = align256(o + n * sizeof(uint32_t));
  L.sidx1 = o;   o = align256(o + n * sizeof(uint32_t));
  L.fx = o;      o = align256(o + n * sizeof(unsigned long long));
  L.fx2 = o;     o = align256(o + n * sizeof(unsigned long long));
  L.dpart = o;   o = align256(o + (size_t)R * nc * sizeof(float2));
  L.rpart = o;   o = align256(o + (size_t)R * nc * sizeof(float2));
  L.total = o;
  return L;
}

template <class T>
inline __host__ __device__ T* ws_at(void* ws, size_t off) {
  return reinterpret_cast<T*>(reinterpret_cast<char*>(ws) + off);
}

// First device-side error wins; later ones are dropped (sticky word).
__device__ __forceinline__ void set_status(uint32_t* status, int code) {
  atomicCAS(status, 0u, (uint32_t)code);
}

// Element loaders: bf16 bit patterns or float32, returned as float (exact).
__device__ __forceinline__ float ld_elem(const float* p, size_t i) { return __ldg(p + i); }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16* p, size_t i) {
  const unsigned short b = __ldg(reinterpret_cast<const unsigned short*>(p) + i);
  return __uint_as_float(((uint32_t)b) << 16);
}

// ---------------------------------------------------------------------------
// Recurrent (gated) sequential head ("Head RNN" of the GeekNews page): state
// s_k = (1 - z[prev_k]) * s_{k-1} + z[prev_k] * W1[prev_k] elementwise, s_0 = 0,
// in float32 with each operation rounded once (z * w of two bf16 values is
// exact); the operand row of position k is s_k rounded to bf16 (to nearest,
// ties to even). Eight elements per call, packed as 16 bytes of bf16 pairs
// (element 2e in the low half of word e).
__device__ __forceinline__ void gated_update8(float s[8], const uint4& z, const uint4& w) {
  const uint32_t zz[4] = {z.x, z.y, z.z, z.w}, ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float z0 = __uint_as_float(zz[e] << 16), z1 = __uint_as_float(zz[e] & 0xffff0000u);
    const float w0 = __uint_as_float(ww[e] << 16), w1 = __uint_as_float(ww[e] & 0xffff0000u);
    s[2 * e] = __fadd_rn(__fmul_rn(__fsub_rn(1.f, z0), s[2 * e]), __fmul_rn(z0, w0));
    s[2 * e + 1] = __fadd_rn(__fmul_rn(__fsub_rn(1.f, z1), s[2 * e + 1]), __fmul_rn(z1, w1));
  }
}
__device__ __forceinline__ uint4 pack_bf16x8(const float s[8]) {
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    o[e] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(s[2 * e])) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(s[2 * e + 1])) << 16);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------------------------
// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11): 10 rounds of the 4x64
// round function with the generator's published multipliers and Weyl key
// increments; u = (2 * (w0 >> 12) + 1) * 2^-53 is an exact double in (0, 1).
enum Purpose : uint64_t { kDraft = 0, kAccept = 1, kResid = 2, kBonus = 3 };

// The odd integer 2 * (w0 >> 12) + 1 < 2^53 of U(seed, r, k, purpose):
// u = philox_odd53(...) * 2^-53 exactly.
__device__ __forceinline__ uint64_t philox_odd53(uint64_t seed, uint64_t r, uint64_t k, uint64_t purpose) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
  uint64_t c0 = r, c1 = k, c2 = purpose, c3 = 0;
  uint64_t k0 = seed, k1 = 0x44535041524B0000ull;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint64_t hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
    const uint64_t hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
    const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    k0 += W0; k1 += W1;
  }
  return 2ull * (c0 >> 12) + 1ull;
}

// floor(u * Z) for u = odd53 * 2^-53 and an integer Z < 2^64 (exact, 128-bit product).
__device__ __forceinline__ unsigned long long scale_u53(uint64_t odd53, unsigned long long Z) {
  const unsigned long long hi = __umul64hi(odd53, Z), lo = odd53 * Z;
  return (hi << 11) | (lo >> 53);
}

// floor(f * 2^40) for a float f: f * 2^40 is exact in float32 (a power-of-two
// scaling, no overflow below 2^88), and the truncating conversion to u64 is
// the floor for f >= 0; negative, NaN and subnormal-range inputs give 0.
__device__ __forceinline__ unsigned long long fx40(float f) { return __float2ull_rz(__fmul_rn(f, 0x1p40f)); }

__device__ __forceinline__ double philox_uniform(uint64_t seed, uint64_t r, uint64_t k, uint64_t purpose) {
  return (double)philox_odd53(seed, r, k, purpose) * 0x1p-53;
}

// ---------------------------------------------------------------------------
// Warp / block reductions with a fixed combination order (deterministic).

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// (value, index) argmax with the lowest index on ties.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
}
__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide reductions for blockDim.x a multiple of 32 (<= 1024); `sh` needs
// 32 slots. All threads receive the result.
__device__ __forceinline__ float block_max(float v, float* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) sh[w] = v;
  __syncthreads();
  v = lane < nw ? sh[lane] : -INFINITY;
  return warp_max(v);
}
__device__ __forceinline__ int block_min_i(int v, int* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_min_i(v);
  __syncthreads();
  if (lane == 0) sh[w] = v;
  __syncthreads();
  v = lane < nw ? sh[lane] : 0x7fffffff;
  return warp_min_i(v);
}
__device__ __forceinline__ int block_max_i(int v, int* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max_i(v);
  __syncthreads();
  if (lane == 0) sh[w] = v;
  __syncthreads();
  v = lane < nw ? sh[lane] : -0x7fffffff;
  return warp_max_i(v);
}
__device__ __forceinline__ void block_argmax(float& v, int& i, float* shv, int* shi) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  warp_argmax(v, i);
  __syncthreads();
  if (lane == 0) { shv[w] = v; shi[w] = i; }
  __syncthreads();
  v = lane < nw ? shv[lane] : -INFINITY;
  i = lane < nw ? shi[lane] : 0x7fffffff;
  warp_argmax(v, i);
}
// Exclusive scan of one double per thread (thread order); returns the total.
// The exclusive value is read from the neighbouring lane's inclusive sum
// rather than formed by subtraction.
__device__ __forceinline__ double block_exscan_d(double v, double* sh, double& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  double x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  double ex = __shfl_up_sync(0xffffffffu, x, 1);
  if (lane == 0) ex = 0.0;
  __syncthreads();
  if (lane == 31) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    double s = lane < nw ? sh[lane] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) sh[lane] = s;
  }
  __syncthreads();
  total = sh[nw - 1];
  const double before_warp = w > 0 ? sh[w - 1] : 0.0;
  const double res = before_warp + ex;
  __syncthreads();
  return res;
}

// Draft / target weight of one vocabulary entry relative to a chunk maximum,
// fixed to explicit round-to-nearest operations so every kernel that forms it
// (partials, locate, residual) produces identical bits:
//   d = (base - m) + bias,  w = 2^(d * log2(e) / T).
__device__ __forceinline__ float draft_weight(float base, float bias, float m, float kT) {
  const float d = __fadd_rn(__fsub_rn(base, m), bias);
  return exp2f(__fmul_rn(d, kT));
}
__device__ __forceinline__ float draft_logit(float base, float bias) { return __fadd_rn(base, bias); }

}  // namespace dspark
