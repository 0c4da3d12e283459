// Base logits from the parallel backbone's hidden states ("DSpark: Aceleração
// da inferência de LLM com speculative decoding [pdf]" (GeekNews), "Etapa
// paralela": the backbone's single pass over the block gives hidden states and
// base logits; "Comunicação de estados ocultos": only the hidden state before
// the LM head has to travel, the LM head runs where the logits are used):
// logits[M, V] = bf16(hidden[M, d] . LM[d, V]), float32 accumulation on the
// tensor cores, one rounding to bf16 (nearest, ties to even).
//
// Persistent kernel, one CTA per SM, 128 x 256 output tiles taken in M-fastest
// order, so the CTAs working at one time read the same LM-head columns (one
// DRAM read, the rest from L2) and the hidden states stay in L2. CTAs run in
// pairs (a cluster of two) on the row tiles 2i and 2i + 1 of the same columns:
// each loads half of the shared B tile and multicasts it to both, halving the
// LM-head bytes the pair pulls from L2 per FLOP.
//   warp 0      TMA producer of a 4-stage ring: A = 128 rows x 64 K of the
//               hidden states (K-major, 128-byte swizzle), B = 64 K-rows x 256
//               LM-head columns as four 64-column boxes (MN-major; two from
//               each CTA of the pair); a stage is refilled once both CTAs'
//               MMAs have released it;
//   warp 1      TMEM allocation and tcgen05.mma issue (kind::f16, M = 128,
//               N = 256, K = 16) into two 256-column accumulators;
//   warps 2..5  epilogue: tcgen05.ld of 32 columns at a time, rounding to bf16,
//               16-byte streaming stores (rows >= M and columns >= V skipped).
// Every wait is bounded: one that runs out records DSPARK_ERR_TIMEOUT, the
// roles wind down, issued copies and MMAs land, and the TMEM is freed.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace dspark {

constexpr int kHM = 128;                 // tile rows (MMA M)
constexpr int kHK = 64;                  // K per stage
constexpr int kHStages = 4;
constexpr int kHEpiWarps = 4;
constexpr int kHCluster = 2;             // CTAs sharing each B tile by multicast (2 or 4)
constexpr int kHThreads = 32 * (2 + kHEpiWarps);
constexpr uint32_t kHABytes = kHM * 128;            // 128 rows x 64 bf16
constexpr uint32_t kHBBox = kHK * 128;              // 64 K-rows x 64 bf16 columns
constexpr uint32_t kHStage = kHABytes + 4 * kHBBox;
constexpr uint32_t kHSmem = 1024 + kHStages * kHStage + 256;

struct LmParams {
  int M, d, V;
  int n_m, n_n, nk;
  int a_rows;  // rows of one A box (min(M, 128))
  __nv_bfloat16* out;
  uint32_t* status;
};

// kC CTAs of a cluster work on kC row tiles of the same columns (kC = 1: no cluster).
template <int kC>
__global__ void __launch_bounds__(kHThreads, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap mapH, const __grid_constant__ CUtensorMap mapLM,
                   LmParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kHStages * kHStage);
  uint64_t* empty = full + kHStages;
  uint64_t* accFull = empty + kHStages;
  uint64_t* accEmpty = accFull + 2;
  uint64_t* drain = accEmpty + 2;
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* sAbort = reinterpret_cast<volatile int*>(sTmem + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // work items: (row tile, column tile), or (pair of row tiles, column tile) for a pair
  constexpr bool kPair = kC > 1;
  constexpr uint16_t kMask = (uint16_t)((1u << kC) - 1u);
  const int crank = kPair ? (int)cluster_ctarank() : 0;
  const int first = (int)blockIdx.x / kC;
  const int stride = (int)gridDim.x / kC;
  const int n_rows = ceil_div(p.n_m, kC);
  const int n_items = n_rows * p.n_n;
  auto item_m = [&](int t) { return kC * (t % n_rows) + crank; };
  auto item_c0 = [&](int t) { return (t / n_rows) * 256; };
  if (tid == 0) {
    for (int i = 0; i < kHStages; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], kC); }
    for (int i = 0; i < 2; ++i) { mbar_init(&accFull[i], 1); mbar_init(&accEmpty[i], kHEpiWarps); }
    mbar_init(drain, 1);
    *sAbort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(sTmem, 512);
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();  // the peer's barriers exist before anything is multicast to them
  tc_fence_after();
  const uint32_t tmem = *sTmem;

  if (warp == 0) {
    if (lane == 0) {  // producer
      prefetch_tensormap(&mapH);
      prefetch_tensormap(&mapLM);
      const uint64_t pol_h = l2_policy_evict_last();   // re-read by every column tile
      const uint64_t pol_w = l2_policy_evict_normal();  // re-read by the row tiles running alongside
      int n = 0;
      bool stop = false;
      for (int t = first; t < n_items && !stop; t += stride) {
        const int m = item_m(t), c0 = item_c0(t);
        const int nbox = min(4, ceil_div(p.V - c0, 64));
        for (int kc = 0; kc < p.nk; ++kc, ++n) {
          const int stage = n % kHStages;
          if (!mbar_wait(&empty[stage], ((n / kHStages) & 1) ^ 1, sAbort, p.status)) { stop = true; break; }
          unsigned char* st = smem + stage * kHStage;
          // the whole B tile lands here: this CTA's boxes and the peer's multicast ones
          mbar_expect_tx(&full[stage], (uint32_t)p.a_rows * 128 + (uint32_t)nbox * kHBBox);
          tma_load_2d(st, &mapH, kc * kHK, m * kHM, &full[stage], pol_h);
          if (kPair) {
            for (int j = crank * (4 / kC); j < (crank + 1) * (4 / kC) && j < nbox; ++j)
              tma_load_2d_multicast(st + kHABytes + j * kHBBox, &mapLM, c0 + 64 * j, kc * kHK, &full[stage],
                                    kMask, pol_w);
          } else {
            for (int j = 0; j < nbox; ++j)
              tma_load_2d(st + kHABytes + j * kHBBox, &mapLM, c0 + 64 * j, kc * kHK, &full[stage], pol_w);
          }
        }
      }
      for (int i = 1; i <= kHStages && n - i >= 0; ++i)  // no copy outlives the CTA
        mbar_wait_drain(&full[(n - i) % kHStages], ((n - i) / kHStages) & 1, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      int n = 0, T = 0;
      bool stop = false;
      for (int t = first; t < n_items && !stop; t += stride, ++T) {
        const int c0 = item_c0(t);
        const int nbox = min(4, ceil_div(p.V - c0, 64));
        const int buf = T & 1;
        if (!mbar_wait(&accEmpty[buf], ((T >> 1) & 1) ^ 1, sAbort, p.status)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(kHM, (uint32_t)(64 * nbox), 1);
        const uint32_t dt = tmem + (uint32_t)(buf * 256);
        for (int kc = 0; kc < p.nk; ++kc, ++n) {
          const int stage = n % kHStages;
          if (!mbar_wait(&full[stage], (n / kHStages) & 1, sAbort, p.status)) { stop = true; break; }
          tc_fence_after();
          const unsigned char* st = smem + stage * kHStage;
#pragma unroll
          for (int kk = 0; kk < kHK / 16; ++kk) {
            const uint64_t a_desc = smem_desc_sw128(smem_u32(st + kk * 32), 0, 1024);
            const uint64_t b_desc = smem_desc_sw128(smem_u32(st + kHABytes + kk * 2048), kHBBox, 1024);
            tc_mma_bf16(dt, a_desc, b_desc, idesc, (kc | kk) != 0);
          }
          if (kPair)
            tc_commit_multicast(&empty[stage], kMask);  // every CTA's copy of the stage is free
          else
            tc_commit(&empty[stage]);
        }
        if (stop) break;
        tc_commit(&accFull[buf]);
      }
      tc_commit(drain);  // every MMA issued so far has completed
      mbar_wait_drain(drain, 0, p.status);
    }
  } else {  // epilogue warps 2..5: warp w reads TMEM lanes 32 (w mod 4) ..
    const int q = warp & 3;
    int T = 0;
    for (int t = first; t < n_items; t += stride, ++T) {
      const int m = item_m(t), c0 = item_c0(t);
      const int ncol = min(256, p.V - c0);
      const int buf = T & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&accFull[buf], (T >> 1) & 1, sAbort, p.status))) break;
      tc_fence_after();
      const int row = m * kHM + 32 * q + lane;
      __nv_bfloat16* orow = p.out + (size_t)min(row, p.M - 1) * p.V + c0;
      for (int c = 0; c < ncol; c += 32) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * 256 + c), v);
        if (row < p.M) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (c + 8 * u + 8 <= ncol) __stcs(reinterpret_cast<uint4*>(orow + c + 8 * u), pack_bf16x8(v + 8 * u));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accEmpty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (kPair) cluster_sync();  // no arrival or copy from the peer is still on its way here
}

}  // namespace dspark

using namespace dspark;

extern "C" dspark_status dspark_lm_head(int32_t M, int32_t d, int32_t V, const void* hidden, const void* lm_head,
                                        void* logits, void* workspace, size_t workspace_bytes,
                                        dspark_stream_t stream) {
  // a TMA box is never wider than its tensor: d >= 64 (one K box) and V >= 64 (one column box)
  if (M < 1 || d < 64 || d % 8 != 0 || V < 64 || V % 8 != 0 || (long long)M * V > (1ll << 40) || !hidden ||
      !lm_head || !logits)
    return DSPARK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(lm_head) |
       reinterpret_cast<uintptr_t>(logits)) & 15)
    return DSPARK_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0 || workspace_bytes < 256)
    return DSPARK_ERR_WORKSPACE;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) return DSPARK_ERR_CUDA;
  static std::atomic<unsigned long long> attr{0}, attr_pair{0};
  if (set_smem_limit_once((const void*)lm_head_kernel<1>, (int)kHSmem, attr) != cudaSuccess ||
      set_smem_limit_once((const void*)lm_head_kernel<kHCluster>, (int)kHSmem, attr_pair) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  LmParams p;
  p.M = M; p.d = d; p.V = V;
  p.n_m = ceil_div(M, kHM);
  p.n_n = ceil_div(V, 256);
  p.nk = ceil_div(d, kHK);
  p.a_rows = M < kHM ? M : kHM;
  p.out = static_cast<__nv_bfloat16*>(logits);
  p.status = static_cast<uint32_t*>(workspace);
  CUtensorMap mapH, mapLM;
  {
    const uint64_t dims[2] = {(uint64_t)d, (uint64_t)M};
    const uint64_t strides[1] = {(uint64_t)d * 2};
    const uint32_t box[2] = {(uint32_t)kHK, (uint32_t)p.a_rows};
    if (!make_tmap_bf16(&mapH, hidden, 2, dims, strides, box)) return DSPARK_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {(uint64_t)V, (uint64_t)d};
    const uint64_t strides[1] = {(uint64_t)V * 2};
    const uint32_t box[2] = {64, (uint32_t)kHK};
    if (!make_tmap_bf16(&mapLM, lm_head, 2, dims, strides, box)) return DSPARK_ERR_CUDA;
  }
  cudaStream_t s = (cudaStream_t)stream;
  // pairs of row tiles share their B tiles; a single row tile (M <= 128) runs unpaired
  int clusters = 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kHCluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kHThreads);
  cfg.dynamicSmemBytes = kHSmem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (p.n_m > 1) {
    cfg.gridDim = dim3(kHCluster * (sms / kHCluster));
    if (cudaOccupancyMaxActiveClusters(&clusters, lm_head_kernel<kHCluster>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      clusters = 0;
    }
  }
  if (clusters > 0) {
    const int items = ceil_div(p.n_m, kHCluster) * p.n_n;
    cfg.gridDim = dim3(kHCluster * std::min(clusters, items));
    if (cudaLaunchKernelEx(&cfg, lm_head_kernel<kHCluster>, mapH, mapLM, p) != cudaSuccess) return DSPARK_ERR_CUDA;
  } else {
    const int grid = std::min(p.n_m * p.n_n, sms);
    lm_head_kernel<1><<<grid, kHThreads, kHSmem, s>>>(mapH, mapLM, p);
  }
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}
