// Base logits from the parallel backbone's hidden states ("DSpark: Aceleração
// da inferência de LLM com speculative decoding [pdf]" (GeekNews), "Etapa
// paralela": the backbone's single pass over the block gives hidden states and
// base logits; "Comunicação de estados ocultos": only the hidden state before
// the LM head has to travel, the LM head runs where the logits are used):
// logits[M, V] = bf16(hidden[M, d] . LM[d, V]), float32 accumulation on the
// tensor cores, one rounding to bf16 (nearest, ties to even).
//
// Persistent kernel, one CTA per SM, 256 x 256 output tiles taken in M-fastest
// order, so the CTAs working at one time read the same LM-head columns (one
// DRAM read, the rest from L2) and the hidden states stay in L2. Each K step
// issues two M = 128 MMAs that share one B stage (rows 0..127 and 128..255 of
// the tile), so every LM-head byte brought into shared memory feeds 256 rows:
// half the L2 reads per FLOP of a 128-row tile, with no cluster.
//   warp 0      TMA producer of a 3-stage ring: A = 256 rows x 64 K of the
//               hidden states (K-major, 128-byte swizzle), B = 64 K-rows x 256
//               LM-head columns as four 64-column boxes (MN-major);
//   warp 1      TMEM allocation and tcgen05.mma issue (kind::f16, M = 128,
//               N = 256, K = 16), two accumulators of 256 columns (the tile's
//               two row halves); the next tile starts once the epilogue has
//               read them (one tile's MMAs take about 80 us at K = 7168, its
//               epilogue about 1 us);
//   warps 2..9  epilogue: warp w reads TMEM lanes 32 (w mod 4) .. + 31 of row
//               half (w - 2) / 4, 32 columns at a time, rounds to bf16 and
//               stores with 16-byte streaming stores (rows >= M and columns
//               >= V skipped).
// Every wait is bounded: one that runs out records DSPARK_ERR_TIMEOUT, the
// roles wind down, issued copies and MMAs land, and the TMEM is freed.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace dspark {

constexpr int kHM = 256;                 // tile rows (two MMAs of M = 128)
constexpr int kHK = 64;                  // K per stage
constexpr int kHStages = 3;
constexpr int kHEpiWarps = 8;
constexpr int kHThreads = 32 * (2 + kHEpiWarps);
constexpr uint32_t kHABytes = kHM * 128;            // 256 rows x 64 bf16
constexpr uint32_t kHBBox = kHK * 128;              // 64 K-rows x 64 bf16 columns
constexpr uint32_t kHStage = kHABytes + 4 * kHBBox;
constexpr uint32_t kHSmem = 1024 + kHStages * kHStage + 256;

struct LmParams {
  int M, d, V;
  int n_m, n_n, nk;
  int a_rows;  // rows of one A box (min(M, 256))
  __nv_bfloat16* out;
  uint32_t* status;
};

__global__ void __launch_bounds__(kHThreads, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap mapH, const __grid_constant__ CUtensorMap mapLM,
                   LmParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kHStages * kHStage);
  uint64_t* empty = full + kHStages;
  uint64_t* accFull = empty + kHStages;
  uint64_t* accEmpty = accFull + 1;
  uint64_t* drain = accEmpty + 1;
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* sAbort = reinterpret_cast<volatile int*>(sTmem + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = p.n_m * p.n_n;
  auto item_m = [&](int t) { return t % p.n_m; };
  auto item_c0 = [&](int t) { return (t / p.n_m) * 256; };
  if (tid == 0) {
    for (int i = 0; i < kHStages; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
    mbar_init(accFull, 1);
    mbar_init(accEmpty, kHEpiWarps);
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
      for (int t = blockIdx.x; t < n_items && !stop; t += gridDim.x) {
        const int m = item_m(t), c0 = item_c0(t);
        const int nbox = min(4, ceil_div(p.V - c0, 64));
        for (int kc = 0; kc < p.nk; ++kc, ++n) {
          const int stage = n % kHStages;
          if (!mbar_wait(&empty[stage], ((n / kHStages) & 1) ^ 1, sAbort, p.status)) { stop = true; break; }
          unsigned char* st = smem + stage * kHStage;
          mbar_expect_tx(&full[stage], (uint32_t)p.a_rows * 128 + (uint32_t)nbox * kHBBox);
          tma_load_2d(st, &mapH, kc * kHK, m * kHM, &full[stage], pol_h);
          for (int j = 0; j < nbox; ++j)
            tma_load_2d(st + kHABytes + j * kHBBox, &mapLM, c0 + 64 * j, kc * kHK, &full[stage], pol_w);
        }
      }
      for (int i = 1; i <= kHStages && n - i >= 0; ++i)  // no copy outlives the CTA
        mbar_wait_drain(&full[(n - i) % kHStages], ((n - i) / kHStages) & 1, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      int n = 0, T = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < n_items && !stop; t += gridDim.x, ++T) {
        const int m = item_m(t), c0 = item_c0(t);
        const int nbox = min(4, ceil_div(p.V - c0, 64));
        const bool lower = m * kHM + 128 < p.M;  // the tile's second row half holds rows < M
        if (!mbar_wait(accEmpty, (T & 1) ^ 1, sAbort, p.status)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)(64 * nbox), 1);
        for (int kc = 0; kc < p.nk; ++kc, ++n) {
          const int stage = n % kHStages;
          if (!mbar_wait(&full[stage], (n / kHStages) & 1, sAbort, p.status)) { stop = true; break; }
          tc_fence_after();
          const unsigned char* st = smem + stage * kHStage;
#pragma unroll
          for (int kk = 0; kk < kHK / 16; ++kk) {
            const uint64_t b_desc = smem_desc_sw128(smem_u32(st + kHABytes + kk * 2048), kHBBox, 1024);
            const uint32_t acc = (kc | kk) != 0;
            tc_mma_bf16(tmem, smem_desc_sw128(smem_u32(st + kk * 32), 0, 1024), b_desc, idesc, acc);
            if (lower)  // rows 128..255: 128 rows of 128 bytes further into the A stage
              tc_mma_bf16(tmem + 256u, smem_desc_sw128(smem_u32(st + 128 * 128 + kk * 32), 0, 1024), b_desc,
                          idesc, acc);
          }
          tc_commit(&empty[stage]);
        }
        if (stop) break;
        tc_commit(accFull);
      }
      tc_commit(drain);  // every MMA issued so far has completed
      mbar_wait_drain(drain, 0, p.status);
    }
  } else {  // epilogue warps 2..9: warp w reads TMEM lanes 32 (w mod 4) .. of row half (w - 2) / 4
    const int q = warp & 3, half = (warp - 2) >> 2;
    int T = 0;
    for (int t = blockIdx.x; t < n_items; t += gridDim.x, ++T) {
      const int m = item_m(t), c0 = item_c0(t);
      const int ncol = min(256, p.V - c0);
      if (!__all_sync(0xffffffffu, mbar_wait(accFull, T & 1, sAbort, p.status))) break;
      tc_fence_after();
      const int row = m * kHM + 128 * half + 32 * q + lane;
      if (m * kHM + 128 * half < p.M) {  // warp-uniform: the half holds rows < M
        __nv_bfloat16* orow = p.out + (size_t)min(row, p.M - 1) * p.V + c0;
        for (int c = 0; c < ncol; c += 32) {
          float v[32];
          tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(256 * half + c), v);
          if (row < p.M) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (c + 8 * u + 8 <= ncol) __stcs(reinterpret_cast<uint4*>(orow + c + 8 * u), pack_bf16x8(v + 8 * u));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accEmpty);
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
  static std::atomic<unsigned long long> attr{0};
  if (set_smem_limit_once((const void*)lm_head_kernel, (int)kHSmem, attr) != cudaSuccess) return DSPARK_ERR_CUDA;
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
  const int grid = std::min(p.n_m * p.n_n, sms);
  lm_head_kernel<<<grid, kHThreads, kHSmem, s>>>(mapH, mapLM, p);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}
