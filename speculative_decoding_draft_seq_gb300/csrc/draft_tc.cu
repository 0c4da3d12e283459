// Tensor-core drafting step for bf16 inputs (tcgen05 MMA into TMEM, TMA-fed).
//
// "DSpark: Aceleração da inferência de LLM com speculative decoding [pdf]"
// (GeekNews), "Etapa sequencial" / "Head de Markov": at step k every request
// adds bias = W1[prev, :] . W2 (rank r) to its base logits of position k and
// samples token k from the tempered softmax over the vocabulary.
//
// One step is the GEMM [128 requests x r] x [r x V] fused with the softmax
// partials, so neither the bias nor the logits ever reach HBM:
//   * A = the gathered rows W1[prev_r, :], written by the threads into shared
//     memory in the 128-byte-swizzled K-major layout (64 KB for r = 256);
//   * B = W2 tiles [64 K-rows x 64 columns], loaded by TMA (MN-major operand),
//     kept in L2 with an evict-last hint (W2 is re-read at every step);
//   * D = fp32 accumulators in TMEM, two 256-column buffers so the MMA of the
//     next vocabulary tile overlaps the epilogue of the current one;
//   * base logits [128 requests x 64 columns] per chunk, loaded by TMA with an
//     evict-first hint (read once).
// Warp roles: warp 0 issues the W2 loads, warp 2 the base loads, one thread
// of warp 1 issues the MMAs; warps 3..10 run the epilogue (two warps per TMEM
// lane quarter, alternating 64-column chunks): l = base + bias, per-chunk
// max, sum of 2^((l - max) log2(e) / T) -- or (max, argmax) when greedy --
// written as the per-(request, chunk) partials the locate step consumes.
// Each CTA owns a contiguous range of 64-column chunks of the vocabulary
// (balanced to within one chunk) and one 128-request M tile; one CTA per SM.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace dspark {

constexpr int kTcM = 128;
constexpr int kTcKC = 64;   // K rows per W2 stage
constexpr int kTcBStages = 3;
constexpr int kTcBaseStages = 2;  // per epilogue half: each half owns its own ring
constexpr int kTcEpiWarps = 8;
constexpr int kTcWarps = 3 + kTcEpiWarps;
constexpr int kTcThreads = 32 * kTcWarps;
constexpr uint32_t kAChunkBytes = 128 * 128;              // 128 rows x 64 bf16 (one K chunk)
constexpr uint32_t kABytes = 4 * kAChunkBytes;            // rank <= 256
constexpr uint32_t kBBoxBytes = kTcKC * 128;              // 64 K rows x 64 columns
constexpr uint32_t kBStageBytes = 4 * kBBoxBytes;         // up to 4 boxes (256 columns)
constexpr uint32_t kBaseBoxBytes = 128 * 128;             // up to 128 rows x 64 columns
constexpr uint32_t kTcSmemBytes =
    1024 + kABytes + kTcBStages * kBStageBytes + 2 * kTcBaseStages * kBaseBoxBytes + 1024;

struct TcParams {
  int R, gamma, V, rank, k;
  int nc;        // 64-column chunks of the vocabulary
  int n_cta_v;   // CTAs along the vocabulary
  int box_rows;  // rows of one base box (min(128, R))
  float kT;
  int greedy;
  const __nv_bfloat16* W1;
  const int32_t* anchor;
  const int32_t* tokens;
  float2* part;
  uint32_t* status;
};

// Weight of a logit relative to a maximum m (mk = fl(m * kT)); shared by the
// epilogue and the locate step.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float tc_weight(float l, float kT, float mk) { return ex2_approx(__fmaf_rn(l, kT, -mk)); }

__global__ void __launch_bounds__(kTcThreads, 1)
    draft_tc_partials_kernel(const __grid_constant__ CUtensorMap mapW2, const __grid_constant__ CUtensorMap mapBase,
                             TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sA = smem;
  unsigned char* sB = sA + kABytes;
  unsigned char* sBase = sB + kTcBStages * kBStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sBase + 2 * kTcBaseStages * kBaseBoxBytes);
  uint64_t* bFull = bars;
  uint64_t* bEmpty = bars + kTcBStages;
  uint64_t* baseFull = bars + 2 * kTcBStages;        // [half][stage]
  uint64_t* baseEmpty = baseFull + 2 * kTcBaseStages;
  uint64_t* accFull = baseEmpty + 2 * kTcBaseStages;
  uint64_t* accEmpty = accFull + 2;
  uint64_t* drain = accEmpty + 2;
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* sAbort = reinterpret_cast<volatile int*>(sTmem + 1);
  int* sPrev = reinterpret_cast<int*>(sTmem + 2);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.y * kTcM;
  const int c_begin = (int)(((long long)blockIdx.x * p.nc) / p.n_cta_v);
  const int c_end = (int)(((long long)(blockIdx.x + 1) * p.nc) / p.n_cta_v);
  const int n_tiles = (c_end - c_begin + 3) / 4;
  const int nkc = (p.rank + kTcKC - 1) / kTcKC;

  if (tid == 0) {
    for (int i = 0; i < kTcBStages; ++i) { mbar_init(&bFull[i], 1); mbar_init(&bEmpty[i], 1); }
    for (int i = 0; i < 2 * kTcBaseStages; ++i) { mbar_init(&baseFull[i], 1); mbar_init(&baseEmpty[i], 4); }
    for (int i = 0; i < 2; ++i) { mbar_init(&accFull[i], 1); mbar_init(&accEmpty[i], kTcEpiWarps); }
    mbar_init(drain, 1);
    *sAbort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(sTmem, 512);
  }
  if (tid < kTcM) {
    const int r = m0 + tid;
    int prev = 0;
    if (r < p.R) {
      prev = (p.k == 1) ? p.anchor[r] : p.tokens[(size_t)r * p.gamma + (p.k - 2)];
      if (prev < 0 || prev >= p.V) {
        set_status(p.status, DSPARK_ERR_RANGE);
        prev = min(max(prev, 0), p.V - 1);
      }
    }
    sPrev[tid] = prev;
  }
  __syncthreads();
  // A: rows W1[prev] as 128-byte-swizzled K-major tiles, chunk kc holds k in [64kc, 64kc+64).
  for (int u = tid; u < kTcM * 32; u += kTcThreads) {
    const int m = u >> 5, j = u & 31, kc = j >> 3, uu = j & 7;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (m0 + m < p.R && 8 * j < p.rank)
      val = __ldg(reinterpret_cast<const uint4*>(p.W1 + (size_t)sPrev[m] * p.rank + 8 * j));
    *reinterpret_cast<uint4*>(sA + kc * kAChunkBytes + m * 128 + ((uu ^ (m & 7)) << 4)) = val;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;

  if (warp == 0) {
    if (lane == 0) {  // W2 producer
      prefetch_tensormap(&mapW2);
      const uint64_t pol = l2_policy_evict_last();
      int n = 0;  // stage fills issued so far: stage n % S, phase (n / S) & 1
      for (int t = 0; t < n_tiles && !*sAbort; ++t) {
        const int c0 = c_begin + 4 * t, nbox = min(4, c_end - c0);
        for (int kc = 0; kc < nkc; ++kc) {
          const int stage = n % kTcBStages;
          if (!mbar_wait(&bEmpty[stage], ((n / kTcBStages) & 1) ^ 1, sAbort, p.status)) break;
          mbar_expect_tx(&bFull[stage], nbox * kBBoxBytes);
          for (int j = 0; j < nbox; ++j)
            tma_load_2d(sB + stage * kBStageBytes + j * kBBoxBytes, &mapW2, (c0 + j) * 64, kc * kTcKC,
                        &bFull[stage], pol);
          ++n;
        }
      }
      // let the last fills of every stage land before the CTA can exit
      for (int i = 1; i <= kTcBStages && n - i >= 0; ++i)
        mbar_wait_drain(&bFull[(n - i) % kTcBStages], ((n - i) / kTcBStages) & 1, p.status);
    }
  } else if (warp == 2) {
    if (lane == 0) {  // base-logit producer
      prefetch_tensormap(&mapBase);
      const uint64_t pol = l2_policy_evict_first();
      const uint32_t bytes = (uint32_t)p.box_rows * 128;
      // Chunk j of a tile goes to epilogue half j & 1. Each half has its own
      // ring, so every ring has one consumer group that waits on every phase
      // in order (a parity wait cannot tell phase n from phase n + 2).
      int nh[2] = {0, 0};
      bool stop = false;
      for (int t = 0; t < n_tiles && !stop && !*sAbort; ++t) {
        const int c0 = c_begin + 4 * t, nbox = min(4, c_end - c0);
        for (int j = 0; j < nbox; ++j) {
          const int h = j & 1, n = nh[h], slot = h * kTcBaseStages + n % kTcBaseStages;
          if (!mbar_wait(&baseEmpty[slot], ((n / kTcBaseStages) & 1) ^ 1, sAbort, p.status)) { stop = true; break; }
          mbar_expect_tx(&baseFull[slot], bytes);
          tma_load_3d(sBase + slot * kBaseBoxBytes, &mapBase, (c0 + j) * 64, p.k - 1, m0, &baseFull[slot], pol);
          nh[h] = n + 1;
        }
      }
      for (int h = 0; h < 2; ++h)
        for (int i = 1; i <= kTcBaseStages && nh[h] - i >= 0; ++i) {
          const int n = nh[h] - i;
          mbar_wait_drain(&baseFull[h * kTcBaseStages + n % kTcBaseStages], (n / kTcBaseStages) & 1, p.status);
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      int stage = 0;
      uint32_t ph = 0;
      for (int t = 0; t < n_tiles && !*sAbort; ++t) {
        const int buf = t & 1;
        const uint32_t use = (uint32_t)(t >> 1);
        if (!mbar_wait(&accEmpty[buf], (use & 1) ^ 1, sAbort, p.status)) break;
        tc_fence_after();
        const int c0 = c_begin + 4 * t, nbox = min(4, c_end - c0);
        const uint32_t idesc = idesc_bf16_f32(kTcM, (uint32_t)(64 * nbox), 1);
        const uint32_t d = tmem + (uint32_t)(buf * 256);
        bool ok = true;
        for (int kc = 0; kc < nkc; ++kc) {
          if (!mbar_wait(&bFull[stage], ph, sAbort, p.status)) { ok = false; break; }
          tc_fence_after();
          for (int kk = 0; kk < 4 && kc * kTcKC + kk * 16 < p.rank; ++kk) {
            const uint64_t a_desc = smem_desc_sw128(smem_u32(sA + kc * kAChunkBytes + kk * 32), 0, 1024);
            const uint64_t b_desc = smem_desc_sw128(smem_u32(sB + stage * kBStageBytes + kk * 2048), kBBoxBytes, 1024);
            tc_mma_bf16(d, a_desc, b_desc, idesc, (kc | kk) != 0);
          }
          tc_commit(&bEmpty[stage]);
          if (++stage == kTcBStages) { stage = 0; ph ^= 1; }
        }
        if (!ok) break;
        tc_commit(&accFull[buf]);
      }
      tc_commit(drain);  // every MMA issued above has completed once this arrives
      mbar_wait_drain(drain, 0, p.status);
    }
  } else {  // epilogue warps 3..10
    const int q = warp & 3, h = (warp - 3) >> 2;
    const int row = 32 * q + lane, r = m0 + row;
    const float kT = p.kT;
    int nh = 0;  // boxes this half has consumed from its ring
    for (int t = 0; t < n_tiles; ++t) {
      const int buf = t & 1;
      const uint32_t use = (uint32_t)(t >> 1);
      const int c0 = c_begin + 4 * t, nbox = min(4, c_end - c0);
      // every lane waits, then the warp agrees (and reconverges) before the
      // warp-collective tcgen05.ld below
      const bool acc_ok = __all_sync(0xffffffffu, mbar_wait(&accFull[buf], use & 1, sAbort, p.status));
      if (!acc_ok) break;
      tc_fence_after();
      bool ok = true;
      for (int j = h; j < nbox; j += 2) {
        const int s = h * kTcBaseStages + nh % kTcBaseStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&baseFull[s], (nh / kTcBaseStages) & 1, sAbort, p.status))) {
          ok = false;
          break;
        }
        ++nh;
        const unsigned char* brow = sBase + s * kBaseBoxBytes + row * 128;
        const int vbase = (c0 + j) * 64;
        float m = -INFINITY, ssum = 0.f;
        int am = 0x7fffffff;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float acc[32];
          __syncwarp();  // tcgen05.ld is warp-collective: the warp must be converged
          tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * 256 + j * 64 + half * 32), acc);
          float l[32];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int unit = half * 4 + u;
            const uint4 x = *reinterpret_cast<const uint4*>(brow + ((unit ^ (row & 7)) << 4));
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              l[8 * u + 2 * e] = __fadd_rn(__uint_as_float(w[e] << 16), acc[8 * u + 2 * e]);
              l[8 * u + 2 * e + 1] = __fadd_rn(__uint_as_float(w[e] & 0xffff0000u), acc[8 * u + 2 * e + 1]);
            }
          }
          const int vh = vbase + half * 32;
          if (vh + 32 > p.V) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (vh + i >= p.V) l[i] = -INFINITY;
          }
          if (p.greedy) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (l[i] > m) { m = l[i]; am = vh + i; }
          } else {
            float mh = l[0];
#pragma unroll
            for (int i = 1; i < 32; ++i) mh = fmaxf(mh, l[i]);
            const float mn = fmaxf(m, mh);
            const float mk = __fmul_rn(mn, kT);
            float sh = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) sh += tc_weight(l[i], kT, mk);
            ssum = (m == -INFINITY ? 0.f : ssum * tc_weight(m, kT, mk)) + sh;
            m = mn;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&baseEmpty[s]);
        if (r < p.R) p.part[(size_t)r * p.nc + (c0 + j)] = p.greedy ? make_float2(m, __int_as_float(am)) : make_float2(m, ssum);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accEmpty[buf]);
      if (!ok) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Locate step of the tensor-core path: one CTA per request. Combines the
// chunk partials (float64), finds the chunk holding u * Z, recomputes its 64
// logits (bias as a float32 dot product split over four K quarters, summed in
// a fixed order) and finds the token by a float64 prefix sum. Greedy decoding
// reduces the (max, argmax) partials instead.
__global__ void __launch_bounds__(256) draft_tc_locate_kernel(
    int R, int gamma, int V, int rank, int k, const __nv_bfloat16* __restrict__ base,
    const int32_t* __restrict__ anchor, int32_t* __restrict__ tokens, const __nv_bfloat16* __restrict__ W1,
    const __nv_bfloat16* __restrict__ W2, float kT, int greedy, uint64_t seed,
    const float2* __restrict__ part, float* __restrict__ q_tok, float* __restrict__ q_stats,
    uint32_t* status) {
  __shared__ float shf[32];
  __shared__ int shi[32];
  __shared__ double shd[32];
  __shared__ float sW1[256];
  __shared__ float sRed[4][64];
  __shared__ float sW[64];
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
      const float2 q = pr[c];
      const int idx = __float_as_int(q.y);
      if (q.x > bv || (q.x == bv && idx < bi)) { bv = q.x; bi = idx; }
    }
    block_argmax(bv, bi, shf, shi);
    if (tid == 0) {
      tokens[out] = bi;
      q_tok[out] = 1.f;
      q_stats[2 * out] = bv;
      q_stats[2 * out + 1] = 1.f;
    }
    return;
  }

  int prev = (k == 1) ? anchor[r] : tokens[(size_t)r * gamma + (k - 2)];
  prev = min(max(prev, 0), V - 1);
  for (int i = tid; i < rank; i += blockDim.x) sW1[i] = __bfloat162float(W1[(size_t)prev * rank + i]);

  float m = -INFINITY;
  for (int c = tid; c < nc; c += blockDim.x) m = fmaxf(m, pr[c].x);
  const float M = block_max(m, shf);
  const float Mk = __fmul_rn(M, kT);
  const int seg = ceil_div(nc, blockDim.x);
  const int c0 = min(nc, tid * seg), c1 = min(nc, c0 + seg);
  double local = 0.0;
  for (int c = c0; c < c1; ++c) {
    const float2 q = pr[c];
    local += (double)q.y * (double)tc_weight(q.x, kT, Mk);
  }
  double Z;
  const double excl = block_exscan_d(local, shd, Z);
  const double u = philox_uniform(seed, (uint64_t)r, (uint64_t)k, kDraft);
  const double target = u * Z;
  int found = 0x7fffffff, last_pos = -1;
  double run = excl, found_excl = 0.0;
  float found_g = 0.f;
  for (int c = c0; c < c1; ++c) {
    const float2 q = pr[c];
    const float g = tc_weight(q.x, kT, Mk);
    const double f = (double)q.y * (double)g;
    if (f > 0.0) last_pos = c;
    if (found == 0x7fffffff) {
      if (run + f > target) { found = c; found_excl = run; found_g = g; }
      run += f;
    }
  }
  int cstar = block_min_i(found, shi);
  if (found == cstar && cstar != 0x7fffffff) { sExcl = found_excl; sG = found_g; }
  bool fallback = false;
  if (cstar == 0x7fffffff) {
    cstar = max(0, block_max_i(last_pos, shi));
    fallback = true;
    if (tid == 0) { sG = tc_weight(pr[cstar].x, kT, Mk); sExcl = 0.0; }
  }
  __syncthreads();
  {  // bias of the 64 columns of chunk cstar: column tid%64, K quarter tid/64
    const int col = tid & 63, kq = tid >> 6;
    const int v = cstar * kChunk + col;
    const int kq_len = (rank + 3) / 4, k0 = kq * kq_len, k1 = min(rank, k0 + kq_len);
    float acc = 0.f;
    if (v < V) {
#pragma unroll 8
      for (int i = k0; i < k1; ++i) acc = __fmaf_rn(sW1[i], __bfloat162float(W2[(size_t)i * V + v]), acc);
    }
    sRed[kq][col] = acc;
  }
  __syncthreads();
  const float mc = pr[cstar].x;
  const float mck = __fmul_rn(mc, kT);
  if (tid < kChunk) {
    const int v = cstar * kChunk + tid;
    float w = 0.f;
    if (v < V) {
      const float bias = __fadd_rn(__fadd_rn(sRed[0][tid], sRed[1][tid]), __fadd_rn(sRed[2][tid], sRed[3][tid]));
      const float b = __bfloat162float(base[((size_t)r * gamma + (k - 1)) * V + v]);
      w = tc_weight(__fadd_rn(b, bias), kT, mck);
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
    tokens[out] = min(cstar * kChunk + xc, V - 1);
    q_tok[out] = (float)((double)sW[xc] * g / Z);
    q_stats[2 * out] = M;
    q_stats[2 * out + 1] = (float)Z;
  }
}

static int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

bool draft_tc_eligible(const DraftArgs& a) {
  return a.dtype == DSPARK_BF16 && a.rank % 64 == 0 && a.rank <= 256 && a.V % 8 == 0 && a.V >= 64 &&
         (reinterpret_cast<uintptr_t>(a.base) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.W1) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(a.W2) & 15) == 0;
}

cudaError_t launch_draft_tc(const DraftArgs& a, cudaStream_t s, int& launches, bool& taken) {
  taken = false;
  if (!draft_tc_eligible(a)) return cudaSuccess;
  CUtensorMap mapW2, mapBase;
  {
    const uint64_t dims[2] = {(uint64_t)a.V, (uint64_t)a.rank};
    const uint64_t strides[1] = {(uint64_t)a.V * 2};
    const uint32_t box[2] = {64, (uint32_t)kTcKC};
    if (!make_tmap_bf16(&mapW2, a.W2, 2, dims, strides, box)) return cudaSuccess;
  }
  const int box_rows = a.R < kTcM ? a.R : kTcM;
  {
    const uint64_t dims[3] = {(uint64_t)a.V, (uint64_t)a.gamma, (uint64_t)a.R};
    const uint64_t strides[2] = {(uint64_t)a.V * 2, (uint64_t)a.gamma * a.V * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)box_rows};
    if (!make_tmap_bf16(&mapBase, a.base, 3, dims, strides, box)) return cudaSuccess;
  }
  taken = true;
  static std::atomic<unsigned long long> attr{0};
  {
    cudaError_t e = set_smem_limit_once((const void*)draft_tc_partials_kernel, (int)kTcSmemBytes, attr);
    if (e != cudaSuccess) return e;
  }
  const WsLayout L = ws_layout(a.R, a.gamma, a.V);
  TcParams p;
  p.R = a.R; p.gamma = a.gamma; p.V = a.V; p.rank = a.rank;
  p.nc = ceil_div(a.V, kChunk);
  p.n_cta_v = p.nc < sm_count() ? p.nc : sm_count();
  p.box_rows = box_rows;
  p.greedy = a.temperature == 0.f;
  p.kT = p.greedy ? 0.f : (float)(1.4426950408889634 / (double)a.temperature);
  p.W1 = static_cast<const __nv_bfloat16*>(a.W1);
  p.anchor = a.anchor;
  p.tokens = a.tokens;
  p.part = ws_at<float2>(a.ws, L.dpart);
  p.status = ws_at<uint32_t>(a.ws, L.status);
  const dim3 grid(p.n_cta_v, ceil_div(a.R, kTcM));
  for (int k = 1; k <= a.gamma; ++k) {
    p.k = k;
    draft_tc_partials_kernel<<<grid, kTcThreads, kTcSmemBytes, s>>>(mapW2, mapBase, p);
    draft_tc_locate_kernel<<<a.R, 256, 0, s>>>(a.R, a.gamma, a.V, a.rank, k,
                                                static_cast<const __nv_bfloat16*>(a.base), a.anchor, a.tokens,
                                                p.W1, static_cast<const __nv_bfloat16*>(a.W2), p.kT, p.greedy,
                                                a.seed, p.part, a.q_tok, a.q_stats, p.status);
    launches += 2;
  }
  return cudaGetLastError();
}

}  // namespace dspark
