// Target-distribution row statistics and the acceptance chain ("DSpark:
// Aceleração da inferência de LLM com speculative decoding [pdf]"
// (GeekNews), "Definição do problema": the target checks the drafted block in
// one pass, rejection sampling keeps the longest consistent prefix), shared by
// the verification kernels (verify.cu) and by the drafting launch
// (draft_persistent.cu), whose spare CTAs compute the statistics of the
// scheduled target rows while the other CTAs draft (the statistics need the
// schedule, not the drafted tokens) and whose CTAs run every request's chain
// once the last token is drawn. Both places cut a row into the same pieces
// and combine them in the same order, so they produce the same bits.
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace dspark {

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed helpers: the larger of each bf16 half; two float32 in one 64-bit
// register and an fma on both halves (sm_100 and later).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f32x2_pack(float lo, float hi) {
  unsigned long long d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f32x2_unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f32x2_fma(unsigned long long a, unsigned long long b,
                                                        unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// A group of eight bf16 -inf: the filler of a chunk's missing groups.
__device__ __forceinline__ uint4 neg_inf_group() { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }

// Streaming row statistics of 8 consecutive bf16 values (one 16-byte load):
// sampled mode keeps (max m, sum of 2^(t kT - m kT)) with a running rescale,
// greedy mode keeps (max, lowest index of the max).
struct RowStat {
  float m = -INFINITY, s = 0.f;
  int ai = 0x7fffffff;
  __device__ __forceinline__ void add8_sampled(const uint4& q, float kT) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    float t[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      t[2 * e] = __uint_as_float(w[e] << 16);
      t[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
    const float gm = fmaxf(max3(t[0], t[1], t[2]), max3(t[3], t[4], max3(t[5], t[6], t[7])));
    if (gm > m) {
      s = m == -INFINITY ? 0.f : __fmul_rn(s, ex2_approx(__fmul_rn(__fsub_rn(m, gm), kT)));
      m = gm;
    }
    const float mk = __fmul_rn(m, kT);
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      a0 += ex2_approx(__fmaf_rn(t[i], kT, -mk));
      a1 += ex2_approx(__fmaf_rn(t[i + 1], kT, -mk));
    }
    s += a0 + a1;
  }
  __device__ __forceinline__ void add8_greedy(const uint4& q, int v0) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    float t[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      t[2 * e] = __uint_as_float(w[e] << 16);
      t[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
    const float gm = fmaxf(max3(t[0], t[1], t[2]), max3(t[3], t[4], max3(t[5], t[6], t[7])));
    if (gm > m) {  // strict: the first index of a tie across groups stays
      m = gm;
      int i = 7;
#pragma unroll
      for (int j = 6; j >= 0; --j) i = t[j] == gm ? j : i;
      ai = v0 + i;
    }
  }
  // A lane's share of one chunk at once. Sampled mode: the groups past the
  // chunk's end must hold bf16 -inf (neg_inf_group()), so that they add nothing.
  // The chunk's maximum comes first, on the packed bf16 pairs (exact: bf16 to
  // float32 is exact and keeps the order); the running sum is rescaled at most
  // once; then the 64 terms 2^(t kT - m kT) are formed and added in float32
  // pairs (fma.rn.f32x2: each half rounds as the scalar instruction would; the
  // sum as an fma by 1.0), in four independent accumulators combined in a
  // fixed tree. Greedy mode keeps the lowest index of the maximum, the groups
  // being g0, g0 + 32, ... in order (only the first nv).
  __device__ __forceinline__ void add_chunk_sampled(const uint4 (&q)[8], float kT) {
    uint32_t mx = 0xFF80FF80u;
#pragma unroll
    for (int u = 0; u < 8; ++u) mx = bf16x2_max(mx, bf16x2_max(bf16x2_max(q[u].x, q[u].y), bf16x2_max(q[u].z, q[u].w)));
    const float cm = fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xffff0000u));
    if (cm == -INFINITY) return;  // nothing in this chunk (and m may still be -inf)
    if (cm > m) {
      s = m == -INFINITY ? 0.f : __fmul_rn(s, ex2_approx(__fmul_rn(__fsub_rn(m, cm), kT)));
      m = cm;
    }
    const float mk = __fmul_rn(m, kT);
    const unsigned long long k2 = f32x2_pack(kT, kT), nmk2 = f32x2_pack(-mk, -mk), one2 = f32x2_pack(1.f, 1.f);
    unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a0, a1;
        f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u)), k2, nmk2),
                     a0, a1);
        acc[u & 3] = f32x2_fma(f32x2_pack(ex2_approx(a0), ex2_approx(a1)), one2, acc[u & 3]);
      }
    }
    float r[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) f32x2_unpack(acc[i], r[2 * i], r[2 * i + 1]);
    s += ((r[0] + r[1]) + (r[2] + r[3])) + ((r[4] + r[5]) + (r[6] + r[7]));
  }
  __device__ __forceinline__ void add_chunk_greedy(const uint4 (&q)[8], int nv, int g0) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (u < nv) add8_greedy(q[u], (g0 + 32 * u) * 8);
  }
};

// ---------------------------------------------------------------------------
// Row statistics by warps, for bf16 target rows with V % 8 == 0 (16-byte
// aligned rows). A row is cut into kVwSplit pieces; one warp streams a piece
// (evict-first: the rows are read once and must not push other data out of
// L2). The piece's statistics (M_s, Z_s, max, argmax) are a fixed function of
// its values, whichever warp computes them.
constexpr int kVwSplit = kVsPieceMax;

// The pieces are read in chunks of kVwChunk groups; lane l holds the chunk's
// groups l, l + 32, ..., l + 224 (at most eight) and adds them at once
// (RowStat::add_chunk_*), so a lane's arithmetic depends only on the piece's
// values and the chunk boundaries, not on how the chunk reached it.
constexpr int kVwChunk = 256;

__device__ __forceinline__ float4 warp_row_piece(const __nv_bfloat16* __restrict__ target, size_t rowi, int V, int sp,
                                                 float kT, int greedy, int lane) {
  RowStat st;
  const int ng = V >> 3;
  const int gb = (int)(((long long)sp * ng) / kVwSplit), ge = (int)(((long long)(sp + 1) * ng) / kVwSplit);
  const uint4* src = reinterpret_cast<const uint4*>(target + rowi * (size_t)V) + gb;
  const int len = ge - gb;
  uint4 cur[8], nxt[8];
  auto load = [&](uint4 (&q)[8], int c0) {
    const int cnt = min(kVwChunk, len - c0);
#pragma unroll
    for (int u = 0; u < 8; ++u) q[u] = lane + 32 * u < cnt ? __ldcs(src + c0 + lane + 32 * u) : neg_inf_group();
  };
  if (len > 0) load(cur, 0);
  for (int c0 = 0; c0 < len; c0 += kVwChunk) {
    if (c0 + kVwChunk < len) load(nxt, c0 + kVwChunk);  // the next chunk in flight while this one is added
    const int cnt = min(kVwChunk, len - c0);
    const int nv = cnt > lane ? (cnt - lane + 31) / 32 : 0;
    if (greedy) st.add_chunk_greedy(cur, nv, gb + c0 + lane);
    else st.add_chunk_sampled(cur, kT);
#pragma unroll
    for (int u = 0; u < 8; ++u) cur[u] = nxt[u];
  }
  if (greedy) {
    float am = st.m;
    int ai = st.ai;
    warp_argmax(am, ai);
    return make_float4(0.f, 0.f, am, __int_as_float(ai));
  }
  const float Ms = warp_max(st.m);
  const float contrib = st.s > 0.f ? __fmul_rn(st.s, ex2_approx(__fmul_rn(__fsub_rn(st.m, Ms), kT))) : 0.f;
  unsigned long long z = fx40(contrib);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  return make_float4(Ms, __fmul_rn((float)z, 0x1p-40f), Ms, __int_as_float(0));
}

// The same piece streamed through the warp's ring of shared-memory slots by
// bulk copies (kVwSlots chunks of kVwChunk groups in flight, read once: L2
// evict-first), so that a warp keeps 16 KB of the row in flight without
// holding it in registers. Lane l takes the same groups in the same order as
// warp_row_piece, so the result is the same. `n_issued` / `n_done` count the
// warp's chunks across calls (chunk n uses slot n % kVwSlots, phase
// (n / kVwSlots) & 1). False if a wait ran out (DSPARK_ERR_TIMEOUT recorded,
// the warp's copies in flight drained).
constexpr int kVwSlots = 4;
constexpr uint32_t kVwRingBytes = (uint32_t)kVwSlots * kVwChunk * 16;

__device__ __forceinline__ bool warp_row_piece_ring(const __nv_bfloat16* __restrict__ target, size_t rowi, int V,
                                                    int sp, float kT, int greedy, int lane, unsigned char* ring,
                                                    uint64_t* bars, uint32_t& n_issued, uint32_t& n_done,
                                                    uint64_t policy, uint32_t* status, float4& result) {
  RowStat st;
  const int ng = V >> 3;
  const int gb = (int)(((long long)sp * ng) / kVwSplit), ge = (int)(((long long)(sp + 1) * ng) / kVwSplit);
  const uint4* src = reinterpret_cast<const uint4*>(target + rowi * (size_t)V) + gb;
  const int len = ge - gb, nch = (len + kVwChunk - 1) / kVwChunk;
  int next = 0;
  auto issue = [&]() {  // warp-uniform
    if (lane == 0) {
      const int slot = (int)(n_issued % kVwSlots);
      const uint32_t bytes = (uint32_t)min(kVwChunk, len - next * kVwChunk) * 16u;
      fence_proxy_async_smem();  // the slot's earlier generic reads before the copy's writes
      mbar_expect_tx(bars + slot, bytes);
      bulk_load_hint(ring + (size_t)slot * kVwChunk * 16, src + (size_t)next * kVwChunk, bytes, bars + slot, policy);
    }
    ++n_issued;
    ++next;
  };
  while (next < nch && n_issued - n_done < (uint32_t)kVwSlots) issue();
  for (int j = 0; j < nch; ++j) {
    const int slot = (int)(n_done % kVwSlots);
    const uint32_t parity = (n_done / kVwSlots) & 1u;
    bool ready = false;
    for (uint32_t i = 0; i < kSpinLimit && !ready; ++i) ready = mbar_try_wait(bars + slot, parity);
    if (!__all_sync(0xffffffffu, ready)) {
      if (lane == 0) atomicCAS(status, 0u, (uint32_t)DSPARK_ERR_TIMEOUT);
      for (; n_done < n_issued; ++n_done) mbar_wait_drain(bars + n_done % kVwSlots, (n_done / kVwSlots) & 1u, status);
      return false;
    }
    const uint4* c4 = reinterpret_cast<const uint4*>(ring + (size_t)slot * kVwChunk * 16);
    const int cnt = min(kVwChunk, len - j * kVwChunk);
    const int nv = cnt > lane ? (cnt - lane + 31) / 32 : 0;
    uint4 q[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) q[u] = u < nv ? c4[lane + 32 * u] : neg_inf_group();
    if (greedy) st.add_chunk_greedy(q, nv, gb + j * kVwChunk + lane);
    else st.add_chunk_sampled(q, kT);
    ++n_done;
    __syncwarp();
    if (next < nch) issue();
  }
  if (greedy) {
    float am = st.m;
    int ai = st.ai;
    warp_argmax(am, ai);
    result = make_float4(0.f, 0.f, am, __int_as_float(ai));
    return true;
  }
  const float Ms = warp_max(st.m);
  const float contrib = st.s > 0.f ? __fmul_rn(st.s, ex2_approx(__fmul_rn(__fsub_rn(st.m, Ms), kT))) : 0.f;
  unsigned long long z = fx40(contrib);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  result = make_float4(Ms, __fmul_rn((float)z, 0x1p-40f), Ms, __int_as_float(0));
  return true;
}

// The row's statistics from its kVwSplit pieces: M = max M_s, Z = sum of the
// pieces' sums rescaled to M (each term rounded once in float32, summed as
// 2^-40 integers), the lowest-index argmax; greedy rows keep (0, 1, argmax).
__device__ __forceinline__ float4 combine_row_pieces(const float4 (&q)[kVwSplit], float kT, int greedy) {
  float bv = q[0].z, M = q[0].x;
  int bi = __float_as_int(q[0].w);
#pragma unroll
  for (int i = 1; i < kVwSplit; ++i) {
    const int ii = __float_as_int(q[i].w);
    if (q[i].z > bv || (q[i].z == bv && ii < bi)) { bv = q[i].z; bi = ii; }
    M = fmaxf(M, q[i].x);
  }
  if (greedy) return make_float4(0.f, 1.f, __int_as_float(bi), 0.f);
  unsigned long long Z = 0ull;
#pragma unroll
  for (int i = 0; i < kVwSplit; ++i)
    if (q[i].y > 0.f) Z += fx40(__fmul_rn(q[i].y, ex2_approx(__fmul_rn(__fsub_rn(q[i].x, M), kT))));
  return make_float4(M, __fmul_rn((float)Z, 0x1p-40f), __int_as_float(bi), 0.f);
}

// The buffers of the row-statistics work queue and of the chains.
struct RowWork {
  const __nv_bfloat16* target;  // [R, gamma + 1, V]
  const uint32_t* list;         // scheduled rows r (gamma + 1) + k, k <= L_r
  int n_items;                  // rows in the list * kVwSplit
  float4* pieces;               // [R (gamma + 1)][kVwSplit]
  unsigned int* row_cnt;        // [R (gamma + 1)] pieces done (zero between calls)
  unsigned int* req_cnt;        // [R] rows combined (zero between calls)
  float4* rowstat;              // [R (gamma + 1)] (M, Z, argmax, -)
  unsigned int* queue;          // next item (zero at launch)
  int gamma, V, greedy;
  float kT;
};

// Item i * kVwSplit + sp of the queue: piece sp of list row i, streamed by
// one warp through its ring (`ring`: kVwRingBytes of shared memory, `bars`:
// kVwSlots mbarriers initialised by the caller; `n_issued` / `n_done` carry
// the ring's chunk counts between items). The warp that completes a row's
// last piece combines the row and counts it for its request. False if a wait
// ran out.
__device__ __forceinline__ bool row_item(const RowWork& w, unsigned int item, int lane, unsigned char* ring,
                                         uint64_t* bars, uint32_t& n_issued, uint32_t& n_done, uint64_t policy,
                                         uint32_t* status) {
  const uint32_t rowi = __ldcg(w.list + item / kVwSplit);
  const int sp = (int)(item % kVwSplit);
  float4 part;
  if (!warp_row_piece_ring(w.target, rowi, w.V, sp, w.kT, w.greedy, lane, ring, bars, n_issued, n_done, policy, status,
                           part))
    return false;
  if (lane == 0) {
    __stcg(w.pieces + (size_t)rowi * kVwSplit + sp, part);
    __threadfence();
    if (atomicAdd(w.row_cnt + rowi, 1u) == (unsigned int)(kVwSplit - 1)) {
      __threadfence();
      w.row_cnt[rowi] = 0u;
      float4 q[kVwSplit];
#pragma unroll
      for (int i = 0; i < kVwSplit; ++i) q[i] = __ldcg(w.pieces + (size_t)rowi * kVwSplit + i);
      __stcg(w.rowstat + rowi, combine_row_pieces(q, w.kT, w.greedy));
      __threadfence();
      atomicAdd(w.req_cnt + rowi / (uint32_t)(w.gamma + 1), 1u);
    }
  }
  return true;
}

// One warp takes items from the queue, one at a time, until it is empty.
__device__ __forceinline__ bool row_items_warp(const RowWork& w, int lane, unsigned char* ring, uint64_t* bars,
                                               uint32_t* status) {
  const uint64_t policy = l2_policy_evict_first();
  uint32_t n_issued = 0u, n_done = 0u;
  for (;;) {
    unsigned int item = 0u;
    if (lane == 0) item = atomicAdd(w.queue, 1u);
    item = __shfl_sync(0xffffffffu, item, 0);
    if (item >= (unsigned int)w.n_items) return true;
    if (!row_item(w, item, lane, ring, bars, n_issued, n_done, policy, status)) return false;
  }
}

// Request r's verification once its rows 0..L are combined (one warp):
// p_k = P_k(x_{k+1}) for k < L (0 for the unscheduled positions), the chain
// of ratio tests u < p/q in float64 (the first failure at position j keeps
// A = j - 1 tokens), the emitted tokens, A, the pending residual or bonus
// draw, and, when stage_rank > 0, the residual pass's A row W1[prev] (zeros
// for a bonus draw). Greedy: p = 1 where x is the target argmax, and the
// emitted token at A is the argmax of row A.
__device__ __forceinline__ void request_chain(int r, int gamma, int V, const __nv_bfloat16* __restrict__ target,
                                              const int32_t* tokens, const int32_t* __restrict__ anchor,
                                              const float* __restrict__ q_tok, float kT, int greedy, uint64_t seed,
                                              const float4* rowstat, float* p_tok, int32_t* __restrict__ out,
                                              int32_t* __restrict__ acc_len, int4* __restrict__ pend,
                                              uint32_t* status, const __nv_bfloat16* __restrict__ W1, int stage_rank,
                                              __nv_bfloat16* astage, int L, int lane) {
  // lane k of each block of 32 positions: the token, p and q of position k together, then the ratio test
  // of position k + 1 on the values in registers (no round trip through p_tok)
  const size_t rb = (size_t)r * (gamma + 1), tb = (size_t)r * gamma;
  int A = L, x0 = 0;  // x0: this lane's drafted token of block 0 (positions 0..31), as stored
  bool found = false;
  for (int k0 = 0; k0 < gamma; k0 += 32) {
    const int k = k0 + lane;
    float pv = 0.f, qv = 1.f;
    int xr = 0;
    if (k < L) {
      xr = __ldcg(tokens + tb + k);
      int x = xr;
      if (x < 0 || x >= V) { set_status(status, DSPARK_ERR_RANGE); x = min(max(x, 0), V - 1); }
      const float4 rs = __ldcg(rowstat + rb + k);
      qv = __ldcg(q_tok + tb + k);
      if (greedy) {
        pv = x == __float_as_int(rs.z) ? 1.f : 0.f;
      } else {
        const float t = __bfloat162float(target[(rb + k) * (size_t)V + x]);
        pv = __fdiv_rn(ex2_approx(__fmaf_rn(t, kT, -__fmul_rn(rs.x, kT))), rs.y);
      }
    }
    if (k < gamma) __stcg(p_tok + tb + k, pv);
    if (k0 == 0) x0 = xr;
    bool fail = false;
    if (k < L) {
      const double u = philox_uniform(seed, (uint64_t)r, (uint64_t)(k + 1), kAccept);
      fail = !((qv <= 0.f) || (u < (double)pv / (double)qv));
    }
    const unsigned m = __ballot_sync(0xffffffffu, fail);
    if (!found && m) {  // the first rejected position k + 1 keeps A = k tokens
      A = k0 + __ffs(m) - 1;
      found = true;
    }
  }
  for (int kk = lane; kk <= gamma; kk += 32) {
    if (kk < A) out[rb + kk] = kk < 32 ? x0 : __ldcg(tokens + tb + kk);
    else if (kk > A) out[rb + kk] = -1;
  }
  int prev_raw;
  if (A == 0) prev_raw = anchor[r];
  else if (A <= 32) prev_raw = __shfl_sync(0xffffffffu, x0, A - 1);
  else prev_raw = __ldcg(tokens + tb + A - 1);
  if (lane == 0) {
    acc_len[r] = A;
    if (greedy) {
      out[rb + A] = __float_as_int(__ldcg(rowstat + rb + A).z);
      pend[r] = make_int4(kPendNone, A, prev_raw, A);
    } else {
      pend[r] = make_int4(A < L ? kPendResid : kPendBonus, A, prev_raw, A);
    }
  }
  if (stage_rank > 0 && !greedy && 8 * lane < stage_rank) {
    const int prev = min(max(prev_raw, 0), V - 1);
    const uint4 w = A < L ? __ldg(reinterpret_cast<const uint4*>(W1 + (size_t)prev * stage_rank) + lane)
                          : make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(astage + (size_t)r * stage_rank)[lane] = w;
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
}

}  // namespace dspark
