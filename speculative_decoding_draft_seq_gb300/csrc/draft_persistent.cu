// Persistent tensor-core drafting: all gamma sequential steps in one
// cooperative launch (bf16 inputs).
//
// "DSpark: Aceleração da inferência de LLM com speculative decoding [pdf]"
// (GeekNews), "Etapa sequencial" / "Head de Markov": at step k each request
// adds bias = W1[prev, :] . W2 to its base logits of position k and samples
// token k from the tempered softmax over the vocabulary; prev is the token
// just sampled at k - 1 (the anchor at k = 1), so the steps are sequential.
//
// One CTA per SM, each owning a contiguous range of 64-column chunks of the
// vocabulary. Per step k:
//   1. A = W1[prev_r, :] (128 requests per M tile) arrives in 128-byte-
//      swizzled K-major shared memory by TMA from the rows the previous step's
//      draws staged in the workspace (gathered by threads at k = 1);
//   2. tcgen05 MMAs (one issuing thread) multiply A by TMA-loaded W2 tiles
//      into TMEM; the epilogue warps add the TMA-loaded base logits and write
//      per-(request, chunk) softmax partials (max, sum of 2^((l-max)log2e/T))
//      or (max, argmax) for greedy decoding;
//   3. grid barrier; the epilogue warps of CTA b draw the tokens of requests
//      r = b, b + #CTAs, ...: an exact 2^-40 fixed-point scan of the chunk
//      masses finds the crossing chunk, its 64 logits are recomputed and a
//      fixed-point warp scan finds the token, whose W1 row is staged for
//      step k + 1;
//   4. grid barrier; the tokens are visible to every CTA for step k + 1.
// The W2 and base-logit producers do not depend on the sampled tokens, so
// they keep streaming across steps: the first tiles of step k + 1 load while
// step k is being located. Inside a round the launch has CTAs past the sweep's:
// one computes the round's prefix schedule and lists the target rows
// verification reads, and the others stream those rows' statistics; after the
// last draw the sweep CTAs take the rows left and run the acceptance chains
// (side_cta_work, after_sweep_work). Every wait (mbarrier, grid barrier,
// counter poll) is bounded: when one runs out the kernel records
// DSPARK_ERR_TIMEOUT, winds down, lets issued copies and MMAs land and frees
// its TMEM.
#include "common.cuh"
#include "internal.h"
#include "sched_common.cuh"
#include "verify_common.cuh"
#include "tc_ptx.cuh"

#include <algorithm>

namespace dspark {

constexpr int kPM = 128;        // requests per M tile (MMA M)
constexpr int kPKC = 64;        // K rows per W2 stage
constexpr int kPBStages = 3;
constexpr int kPBaseStages = 2; // per epilogue half
constexpr int kPEpiWarps = 8;
constexpr int kPWarps = 3 + kPEpiWarps;
constexpr int kPThreads = 32 * kPWarps;
constexpr int kPEpiThreads = 32 * kPEpiWarps;
constexpr uint32_t kPAChunk = 128 * 128;
constexpr uint32_t kPABytes = 4 * kPAChunk;
constexpr uint32_t kPBBox = kPKC * 128;
constexpr uint32_t kPBStage = 4 * kPBBox;
constexpr uint32_t kPBaseBox = 128 * 128;
// The 1 KB block after the rings holds the mbarriers and flags (204 bytes),
// from byte 208 one scratch word per epilogue warp (the stores that hold a
// base slot's release until its values are in registers), and from byte 256
// the draft uniforms of the CTA's first request.
constexpr int kDepOffset = 208, kOddOffset = 256, kOddCap = 96;
static_assert((2 * kPBStages + 4 * kPBaseStages + 10) * 8 + 12 <= kDepOffset &&
                  kDepOffset + 4 * kPEpiWarps <= kOddOffset && kOddOffset + 8 * kOddCap <= 1024,
              "mbarriers, flags, scratch words and the uniforms table fit the 1 KB block after the rings");
constexpr uint32_t kPSmem = 1024 + kPABytes + kPBStages * kPBStage + 2 * kPBaseStages * kPBaseBox + 1024;
constexpr uint32_t kGridSpinLimit = 1u << 20;  // about 1 s of polls

// Scratch of the locate phase, carved from the A-operand region (free
// between the last MMA of a step and the next gather).
constexpr uint32_t kLsW1 = 0;         // float[256]
constexpr uint32_t kLsRed = 1024;     // float[32][64]
constexpr uint32_t kLsW = 9216;       // float[64]
constexpr uint32_t kLsF = 9472;       // float[8]
constexpr uint32_t kLsI = 9504;       // int[8]
constexpr uint32_t kLsI2 = 9536;      // int[8]
constexpr uint32_t kLsD = 9568;       // u64[8]
constexpr uint32_t kLsExcl = 9632;    // u64
constexpr uint32_t kLsG = 9640;       // float
constexpr uint32_t kLsFlag = 9644;    // int
constexpr uint32_t kLsW1Blk = 16384;  // bf16[64][rank]: W1 rows of the crossing chunk
constexpr int kCache = 8;             // chunk partials per thread kept in registers (V <= 131072)

struct PersistParams {
  int R, gamma, V, rank;
  int nc;        // 64-column chunks
  int n_cta;     // grid size (one CTA per SM)
  int n_mt;      // 128-request M tiles
  int box_rows;  // rows of one base box
  float kT;
  int greedy;
  uint64_t seed;
  const __nv_bfloat16* W1;
  const __nv_bfloat16* W2;
  const __nv_bfloat16* base;
  const int32_t* anchor;
  int32_t* tokens;
  float* q_tok;
  float* q_stats;
  float2* part;
  unsigned int* gbar;  // grid-barrier counter, zero at launch
  __nv_bfloat16* astage;  // [2][R][rank] W1 rows of the drawn tokens, by step parity
  // recurrent (gated) head: astage holds bf16(s_k) instead of W1[prev]
  const __nv_bfloat16* gate;  // [V, rank] gate values in [0, 1]; null for the Markov head
  float* gcarry;              // [R][256] float32 state s_k of each request between steps
  uint32_t* status;
  // residual / bonus pass of verification (target, rowstat, pend and out_tokens also serve the drafting
  // launch's verification work below)
  const __nv_bfloat16* target;  // [R, gamma+1, V]
  int4* pend;                   // (kind, target row A, prev token, A)
  float4* rowstat;              // target row stats (M, Z, argmax, -)
  int32_t* out_tokens;          // [R, gamma+1]
  float2* rpart;                // [R][nc] (sum max(0, P - Q), sum P)
  // acceptance labels (one pass over every (request, position) pair)
  int n_pairs;                  // R * gamma
  unsigned long long* lsum;     // [R * gamma] 2^-40 sums of max(0, P - Q), zero between calls
  float* labels;                // [R, gamma]
  int label_tma;                // label pass: target and base boxes by TMA (else per-warp row copies)
  // the round's prefix schedule, computed by one extra CTA of the drafting launch (blockIdx.x == n_cta)
  // while the others sweep: its inputs do not depend on the drafted tokens
  int sched_on;
  const float* conf;             // [R, gamma]
  const float* conf_lag;         // [R, gamma] (LAGGED)
  const float* sps;              // [n_table]
  int n_table, sched_mode;
  int32_t* sched_len;            // [R]
  int32_t* sched_K;              // [1]
  double* tau_theta;             // [2]
  uint32_t *skey0, *skey1, *sidx0, *sidx1;  // [R * gamma] sort buffers, when the keys do not fit shared memory
  unsigned long long* sched_fx;  // [R * gamma] fixed-point prefix sums in sorted order
  // verification's row statistics and chains in the same launch: the scheduler CTA lists the scheduled
  // target rows; the CTAs past it stream their statistics while the sweep runs; after its last draw each
  // sweep CTA takes the rows still queued, then runs the chains of its requests
  int vfuse;
  float4* vpieces;               // [R (gamma + 1)][kVwSplit]
  unsigned int* row_cnt;         // [R (gamma + 1)] (zero between calls)
  unsigned int* req_cnt;         // [R] (zero between calls)
  uint32_t* vlist;               // [R (gamma + 1)]
  float* p_tok;                  // [R, gamma]
  int32_t* accepted_len;         // [R]
  int stage_rank;                // rank when the chain stages the residual pass's A rows (Markov head), else 0
};
// Status words of the launch's verification work (cleared with the grid-barrier counter before the
// launch): the scheduled-row count plus one once the list is published, and the work queue's head.
constexpr int kVReadyWord = 16, kVQueueWord = 17;
// Row-statistics CTAs at most (the CTAs past the scheduler's).
constexpr int kRowCtasMax = 16;

// The scheduler CTA's shared memory: radix counters for its threads, the four key / index arrays, and the
// reduction scratch.
constexpr uint32_t kSchedCntBytes = (uint32_t)kDigits * kPThreads * 4;
constexpr uint32_t kSchedKeysBytes = 4u * kSmemKeys * 4;
static_assert(kSchedCntBytes + kSchedKeysBytes + 32 * (8 + 4 + 8) + 16 <= kPSmem - 1024,
              "the scheduler CTA's tables fit the launch's shared memory");
static_assert(kPWarps * (kVwRingBytes + 8 * kVwSlots) <= kPSmem - 1024,
              "a row-statistics CTA's rings and their mbarriers fit the launch's shared memory");
static_assert(kPEpiWarps * kVwRingBytes <= kPBStages * kPBStage + 2 * kPBaseStages * kPBaseBox &&
                  kOddOffset + kPEpiWarps * kVwSlots * 8 <= 1024,
              "after the sweep, the epilogue warps' rings fit the W2 and base rings, their mbarriers the uniforms "
              "table");

// Per-request constants of the residual pass: P(v) = 2^((t_v - M_P) log2e/T) / Z_P
// from the target row stats, Q(v) from the draft stats of the rejected position.
struct ResidRow {
  int kind, A;
  float MPk, invZP, MQk, invZQ;
};

__device__ __forceinline__ float px2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Weight of logit l relative to a maximum m, with mk = fl(m * kT).
__device__ __forceinline__ float pweight(float l, float kT, float mk) { return px2(__fmaf_rn(l, kT, -mk)); }

// Residual weight max(0, P - Q) (or P for a bonus draw) of one entry; the
// epilogue and the locate step form it with the same operations. P is
// returned through `P`.
__device__ __forceinline__ float resid_w(int kind, float t, float l, const ResidRow& rr, float kT, float& P) {
  P = __fmul_rn(pweight(t, kT, rr.MPk), rr.invZP);
  if (kind != kPendResid) return P;
  const float Q = __fmul_rn(pweight(l, kT, rr.MQk), rr.invZQ);
  return fmaxf(0.f, __fsub_rn(P, Q));
}

// --- reductions over the 8 epilogue warps (named barrier 1) --------------
__device__ __forceinline__ void eg_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ int eg_max_i(int v, int* sh, int ew, int lane) {
  v = warp_max_i(v);
  if (lane == 0) sh[ew] = v;
  eg_sync();
  int r = sh[0];
#pragma unroll
  for (int i = 1; i < kPEpiWarps; ++i) r = max(r, sh[i]);
  eg_sync();
  return r;
}
__device__ __forceinline__ void eg_argmax(float& v, int& idx, float* shf, int* shi, int ew, int lane) {
  warp_argmax(v, idx);
  if (lane == 0) { shf[ew] = v; shi[ew] = idx; }
  eg_sync();
  v = shf[0];
  idx = shi[0];
#pragma unroll
  for (int i = 1; i < kPEpiWarps; ++i)
    if (shf[i] > v || (shf[i] == v && shi[i] < idx)) { v = shf[i]; idx = shi[i]; }
  eg_sync();
}
// Exclusive scan of one unsigned 64-bit integer per epilogue thread (thread
// order) + total and this thread's inclusive value; integer adds are exact,
// so the intervals [exclusive, inclusive) tile [0, total).
__device__ __forceinline__ unsigned long long eg_exscan_u64(unsigned long long v, unsigned long long* sh,
                                                            unsigned long long& total, int ew, int lane,
                                                            unsigned long long& inclusive) {
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  unsigned long long ex = __shfl_up_sync(0xffffffffu, x, 1);
  if (lane == 0) ex = 0ull;
  if (lane == 31) sh[ew] = x;
  eg_sync();
  unsigned long long before = 0ull, tot = 0ull;
#pragma unroll
  for (int i = 0; i < kPEpiWarps; ++i) {
    if (i < ew) before += sh[i];
    tot += sh[i];
  }
  eg_sync();
  total = tot;
  inclusive = before + x;
  return before + ex;
}

// Inclusive warp scan of unsigned 64-bit integers.
__device__ __forceinline__ unsigned long long warp_inscan_u64(unsigned long long x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Grid-wide barrier among the n_cta CTAs of a cooperative launch: one
// thread per CTA calls it, after a CTA barrier that follows the writes it
// publishes. The arrival is a release add (no value awaited) and the poll an
// acquire load. Bounded: on timeout it records DSPARK_ERR_TIMEOUT, raises the
// CTA's abort flag and returns false.
__device__ bool grid_barrier(unsigned int* counter, unsigned int target, uint32_t* status,
                             volatile int* abort) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
  for (uint32_t i = 0; i < kGridSpinLimit; ++i) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
    if (v >= target) return true;
    if (*abort) return false;
    if (i > 64) __nanosleep(32);
  }
  atomicCAS(status, 0u, (uint32_t)DSPARK_ERR_TIMEOUT);
  *abort = 1;
  return false;
}

// Bounded acquire poll of a counter another CTA of the launch advances: true
// once it reaches `target`; on timeout records DSPARK_ERR_TIMEOUT and returns
// false. One thread calls it.
__device__ bool wait_count(const unsigned int* word, unsigned int target, uint32_t* status) {
  for (uint32_t i = 0; i < kGridSpinLimit; ++i) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(word) : "memory");
    if (v >= target) return true;
    if (i > 16) __nanosleep(128);
  }
  atomicCAS(status, 0u, (uint32_t)DSPARK_ERR_TIMEOUT);
  return false;
}

// The scheduled target rows r (gamma + 1) + k, k <= L_r, listed request by
// request, by every thread of the scheduler CTA after the schedule is
// written; then the count plus one is published (release) in the ready word.
__device__ void list_scheduled_rows(const PersistParams& p, unsigned long long* shu) {
  __syncthreads();
  unsigned long long run = 0ull;
  for (int b = 0; b < p.R; b += (int)blockDim.x) {  // block-uniform
    const int r = b + (int)threadIdx.x;
    const int c = r < p.R ? min(max(__ldcg(p.sched_len + r), 0), p.gamma) + 1 : 0;
    unsigned long long tot;
    const unsigned long long ex = block_exscan_u64((unsigned long long)c, shu, tot);
    for (int k = 0; k < c; ++k) p.vlist[run + ex + k] = (uint32_t)(r * (p.gamma + 1) + k);
    run += tot;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int v = (unsigned int)run + 1u;
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.status + kVReadyWord), "r"(v) : "memory");
  }
}

// A warp's row-statistics setup: initialises its ring's kVwSlots mbarriers
// (`rbars`) and waits for the row list. False on timeout.
__device__ bool row_work_setup(const PersistParams& p, int lane, uint64_t* rbars, RowWork& w) {
  if (lane == 0) {
    for (int i = 0; i < kVwSlots; ++i) mbar_init(rbars + i, 1);
    mbar_fence_init();
  }
  __syncwarp();
  unsigned int ready = 0u;
  if (lane == 0) ready = wait_count(p.status + kVReadyWord, 1u, p.status) ? __ldcg(p.status + kVReadyWord) : 0u;
  ready = __shfl_sync(0xffffffffu, ready, 0);
  __syncwarp();
  w = RowWork{p.target, p.vlist, (int)(ready ? ready - 1u : 0u) * kVwSplit, p.vpieces, p.row_cnt, p.req_cnt,
              p.rowstat, p.status + kVQueueWord, p.gamma, p.V, p.greedy, p.kT};
  return ready != 0u;
}

// A row-statistics CTA's warp: pieces from the queue one at a time until it
// is empty, streamed through `ring` (kVwRingBytes of shared memory).
__device__ bool row_stats_warp(const PersistParams& p, int lane, unsigned char* ring, uint64_t* rbars) {
  RowWork w;
  if (!row_work_setup(p, lane, rbars, w)) return false;
  return row_items_warp(w, lane, ring, rbars, p.status);
}

// The eight epilogue warps of a sweep CTA after its last draw: one atomic
// claims eight pieces (one per warp) at a time, so that the CTAs that reach
// the queue together do not all queue on its counter. Every warp takes part
// in every round's two named barriers, a warp whose wait ran out included;
// warp 0's view of the queue decides for all (sClaim: two words). False if
// the row list never came or a wait ran out.
__device__ bool row_stats_cta(const PersistParams& p, int ew, int lane, unsigned char* ring, uint64_t* rbars,
                              volatile unsigned int* sClaim) {
  RowWork w;
  bool ok = row_work_setup(p, lane, rbars, w);
  const uint64_t policy = l2_policy_evict_first();
  uint32_t n_issued = 0u, n_done = 0u;
  for (;;) {  // sClaim[0] = the round's first item, sClaim[1] = the item count, both from warp 0's view
    if (ew == 0 && lane == 0) {
      sClaim[0] = ok ? atomicAdd(w.queue, (unsigned int)kPEpiWarps) : 0u;
      sClaim[1] = ok ? (unsigned int)w.n_items : 0u;
    }
    eg_sync();
    const unsigned int base = sClaim[0], n_items = sClaim[1];
    eg_sync();
    if (base >= n_items) break;  // CTA-uniform
    const unsigned int item = base + (unsigned int)ew;
    if (ok && item < n_items) ok = row_item(w, item, lane, ring, rbars, n_issued, n_done, policy, p.status);
  }
  return ok;
}

// The CTAs past the sweep's, concurrently with it (they take part in none of its barriers). CTA n_cta is
// the scheduler ("Verificação com agendamento por confiança"): the whole prefix schedule with every thread
// of the block, then the list of the target rows verification reads. With verification in the launch, it
// and the CTAs after it then stream those rows' statistics, one piece per warp. Out of line, like
// after_sweep_work: the sweep's own code stays compact in the instruction caches.
__device__ __noinline__ void side_cta_work(const PersistParams& pg, unsigned char* smem) {
  // a local copy: the fields used stay in registers (through the parameter's address they would be read
  // again after every memory-clobbering barrier and wait)
  const PersistParams p = pg;
  if (blockIdx.x == (unsigned)p.n_cta) {
    uint32_t* cnt = reinterpret_cast<uint32_t*>(smem);
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem + kSchedCntBytes);
    unsigned long long* shu = reinterpret_cast<unsigned long long*>(smem + kSchedCntBytes + kSchedKeysBytes);
    double* shd = reinterpret_cast<double*>(shu + 32);
    int* shi = reinterpret_cast<int*>(shd + 32);
    const BlockSchedScratch sc{cnt, p.R * p.gamma <= kSmemKeys ? keys : nullptr, shu, shi, shd, shi + 32};
    schedule_block(p.R, p.gamma, p.conf, p.conf_lag, p.sps, p.n_table, p.sched_mode, p.sched_len, p.sched_K,
                   p.tau_theta, p.skey0, p.skey1, p.sidx0, p.sidx1, p.sched_fx, p.status, sc);
    if (p.vfuse) list_scheduled_rows(p, shu);
  }
  if (p.vfuse) {  // every warp streams pieces through its own ring; the mbarriers follow the rings
    const int w = (int)(threadIdx.x >> 5);
    row_stats_warp(p, (int)(threadIdx.x & 31), smem + (size_t)w * kVwRingBytes,
                   reinterpret_cast<uint64_t*>(smem + (size_t)kPWarps * kVwRingBytes) + w * kVwSlots);
  }
}

// A sweep CTA's epilogue warps after the last draw (every CTA has drawn its tokens: the step loop ended at a
// grid barrier whose verdict, the same for every warp, the caller tested). The rows still queued: warp ew's
// ring is the ew-th 16 KB of the W2 and base rings (their copies have all landed: every stage was
// consumed), its mbarriers in the uniforms table (read by the draws only), the claim words at the
// dependency scratch. Then each warp runs the verification chain of requests blockIdx.x + ew n_cta,
// blockIdx.x + (ew + 8) n_cta, ... once their rows are combined. `bars` is the 1 KB block after the rings.
__device__ __noinline__ void after_sweep_work(const PersistParams& pg, int ew, int lane, unsigned char* sB,
                                              unsigned char* bars) {
  const PersistParams p = pg;  // a local copy, as in side_cta_work
  if (!row_stats_cta(p, ew, lane, sB + (size_t)ew * kVwRingBytes,
                     reinterpret_cast<uint64_t*>(bars + kOddOffset) + ew * kVwSlots,
                     reinterpret_cast<volatile unsigned int*>(bars + kDepOffset)))
    return;
  for (int r = (int)blockIdx.x + ew * p.n_cta; r < p.R; r += kPEpiWarps * p.n_cta) {
    const int L = min(max(__ldcg(p.sched_len + r), 0), p.gamma);
    int ok = 1;
    if (lane == 0) {
      ok = wait_count(p.req_cnt + r, (unsigned int)(L + 1), p.status) ? 1 : 0;
      if (ok) p.req_cnt[r] = 0u;
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    if (!ok) break;
    request_chain(r, p.gamma, p.V, p.target, p.tokens, p.anchor, p.q_tok, p.kT, p.greedy, p.seed, p.rowstat, p.p_tok,
                  p.out_tokens, p.accepted_len, p.pend, p.status, p.W1, p.stage_rank, p.astage, L, lane);
  }
}

}  // namespace dspark

namespace dspark {

// Gated head, eight state elements per lane: s_k of request r at step k
// (k = 1: z[anchor] * W1[anchor], exact; else the state the previous step
// left in gcarry, written by this same thread).
__device__ __forceinline__ void gated_state_k(const PersistParams& p, int r, int k, int lane, float gs[8]) {
  if (k == 1) {
    const int a = min(max(__ldg(p.anchor + r), 0), p.V - 1);
    const uint4 z = __ldg(reinterpret_cast<const uint4*>(p.gate + (size_t)a * p.rank) + lane);
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(p.W1 + (size_t)a * p.rank) + lane);
#pragma unroll
    for (int e = 0; e < 8; ++e) gs[e] = 0.f;
    gated_update8(gs, z, w);
  } else {
    const float4* c = reinterpret_cast<const float4*>(p.gcarry + (size_t)r * 256) + 2 * lane;
    const float4 x = __ldcg(c), y = __ldcg(c + 1);
    gs[0] = x.x; gs[1] = x.y; gs[2] = x.z; gs[3] = x.w;
    gs[4] = y.x; gs[5] = y.y; gs[6] = y.z; gs[7] = y.w;
  }
}
__device__ __forceinline__ void store_gcarry(const PersistParams& p, int r, int lane, const float gs[8]) {
  float4* c = reinterpret_cast<float4*>(p.gcarry + (size_t)r * 256) + 2 * lane;
  __stcg(c, make_float4(gs[0], gs[1], gs[2], gs[3]));
  __stcg(c + 1, make_float4(gs[4], gs[5], gs[6], gs[7]));
}
// s_{k+1} = update(s_k, z[tok], W1[tok]); the carry and the staged bf16 row.
__device__ __forceinline__ void gated_advance(const PersistParams& p, int r, int tok, int lane, float gs[8],
                                              const uint4& wv, uint4* stage) {
  const uint4 zv = __ldg(reinterpret_cast<const uint4*>(p.gate + (size_t)tok * p.rank) + lane);
  gated_update8(gs, zv, wv);
  store_gcarry(p, r, lane, gs);
  stage[lane] = pack_bf16x8(gs);
}

// Draws token k of request r from the chunk partials (epilogue group of 256
// threads, et = thread index in the group). `ls` is the locate scratch. When a
// step k + 1 follows, the W1 row of the drawn token is staged in
// astage[k & 1][r], the A-operand row of request r for that step; the 64 W1
// rows of the crossing chunk are fetched into shared memory (bulk copy counted
// on w1Full, use number w1_use) while the chunk's logits are recomputed.
template <bool kGated>
__device__ void locate_row(const PersistParams& p, int r, int k, unsigned char* ls, int et, uint64_t* w1Full,
                           uint32_t& w1_use, const uint64_t* odd_tab) {
  const int ew = et >> 5, lane = et & 31;
  float* sW1f = reinterpret_cast<float*>(ls + kLsW1);
  float(*red)[64] = reinterpret_cast<float(*)[64]>(ls + kLsRed);
  float* sW = reinterpret_cast<float*>(ls + kLsW);
  float* shf = reinterpret_cast<float*>(ls + kLsF);
  int* shi = reinterpret_cast<int*>(ls + kLsI);
  int* shi2 = reinterpret_cast<int*>(ls + kLsI2);
  unsigned long long* shu = reinterpret_cast<unsigned long long*>(ls + kLsD);
  unsigned long long* sExclU = reinterpret_cast<unsigned long long*>(ls + kLsExcl);
  float* sG = reinterpret_cast<float*>(ls + kLsG);
  int* sFlag = reinterpret_cast<int*>(ls + kLsFlag);
  const unsigned char* sBlk = ls + kLsW1Blk;

  const int nc = p.nc;
  const float2* pr = p.part + (size_t)r * nc;
  const size_t out = (size_t)r * p.gamma + (k - 1);
  const bool stage_next = k < p.gamma;
  uint4* stage = reinterpret_cast<uint4*>(p.astage + ((size_t)(k & 1) * p.R + r) * p.rank);
  const int seg = (nc + kPEpiThreads - 1) / kPEpiThreads;
  const int c0 = min(nc, et * seg), c1 = min(nc, c0 + seg);
  // this thread's partials, kept in registers (statically indexed) when the
  // segment is short enough, else re-read from L2
  const bool cached = c1 - c0 <= kCache;
  float2 cache[kCache];
#pragma unroll
  for (int i = 0; i < kCache; ++i)
    cache[i] = (cached && i < c1 - c0) ? __ldcg(pr + c0 + i) : make_float2(-INFINITY, 0.f);

  if (p.greedy) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    if (cached) {
#pragma unroll
      for (int i = 0; i < kCache; ++i) {
        const float2 q = cache[i];
        const int idx = __float_as_int(q.y);
        if (i < c1 - c0 && (q.x > bv || (q.x == bv && idx < bi))) { bv = q.x; bi = idx; }
      }
    } else {
      for (int c = c0; c < c1; ++c) {
        const float2 q = __ldcg(pr + c);
        const int idx = __float_as_int(q.y);
        if (q.x > bv || (q.x == bv && idx < bi)) { bv = q.x; bi = idx; }
      }
    }
    eg_argmax(bv, bi, shf, shi2, ew, lane);
    const int tok = min(max(bi, 0), p.V - 1);
    if (ew == 0 && stage_next && 8 * lane < p.rank) {  // 16 bytes of the W1 row per lane
      const uint4 wv = __ldg(reinterpret_cast<const uint4*>(p.W1 + (size_t)tok * p.rank) + lane);
      if (kGated) {
        float gs[8];
        gated_state_k(p, r, k, lane, gs);
        gated_advance(p, r, tok, lane, gs, wv, stage);
      } else {
        stage[lane] = wv;
      }
      fence_proxy_async_global();
    }
    if (ew == 1) {
      // The recorded maximum is the drafted token's logit with its bias summed
      // in float64 and rounded once, fl32(base + fl32(a . W2[:, tok])), a = this
      // step's A row (W1[prev], or the gated head's bf16 state): the value the
      // greedy argmax is defined on. The tensor cores' float32 sums, which the
      // argmax was taken over, can differ from it in the last bits. Products of
      // two bf16 values are exact in float64.
      double acc = 0.0;
      const int a = min(max(__ldg(p.anchor + r), 0), p.V - 1);
      const unsigned short* arow =
          reinterpret_cast<const unsigned short*>(p.astage + ((size_t)((k - 1) & 1) * p.R + r) * p.rank);
      for (int i = lane; i < p.rank; i += 32) {
        float av;
        if (k > 1) {
          av = __uint_as_float((uint32_t)__ldcg(arow + i) << 16);
        } else {
          av = __bfloat162float(p.W1[(size_t)a * p.rank + i]);
          if (kGated) av = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__bfloat162float(p.gate[(size_t)a * p.rank + i]), av)));
        }
        acc = fma((double)av, (double)__bfloat162float(p.W2[(size_t)i * p.V + tok]), acc);
      }
      acc = warp_sum_d(acc);
      if (lane == 0)
        p.q_stats[2 * out] = __fadd_rn(__bfloat162float(p.base[((size_t)r * p.gamma + (k - 1)) * p.V + tok]),
                                       __double2float_rn(acc));
    }
    if (et == 0) {
      __stcg(p.tokens + out, tok);
      p.q_tok[out] = 1.f;
      p.q_stats[2 * out + 1] = 1.f;
    }
    fence_proxy_async_smem();  // the scratch is overwritten next by a TMA load of the A operand
    return;
  }

  // W1 row of the previous token: the anchor's at k = 1, else the row this
  // CTA staged when it drew token k - 1 of this request
  if (k == 1) {
    const int a = min(max(__ldg(p.anchor + r), 0), p.V - 1);
    for (int i = et; i < p.rank; i += kPEpiThreads) {
      const float w = __bfloat162float(p.W1[(size_t)a * p.rank + i]);
      // gated head: s_1 = z[anchor] * W1[anchor] (exact), rounded to bf16
      sW1f[i] = kGated ? __bfloat162float(__float2bfloat16_rn(__fmul_rn(__bfloat162float(p.gate[(size_t)a * p.rank + i]), w)))
                       : w;
    }
  } else {
    const __nv_bfloat16* prev_row = p.astage + ((size_t)((k - 1) & 1) * p.R + r) * p.rank;
    for (int i = et; i < p.rank; i += kPEpiThreads) {
      const unsigned short h = __ldcg(reinterpret_cast<const unsigned short*>(prev_row) + i);
      sW1f[i] = __uint_as_float((uint32_t)h << 16);
    }
  }
  // the draw's uniform: from the table filled at launch (this CTA's first request), else computed here
  const uint64_t odd = odd_tab ? odd_tab[k - 1] : philox_odd53(p.seed, (uint64_t)r, (uint64_t)k, kDraft);

  float m = -INFINITY;
  if (cached) {
#pragma unroll
    for (int i = 0; i < kCache; ++i) m = fmaxf(m, cache[i].x);
  } else {
    for (int c = c0; c < c1; ++c) m = fmaxf(m, __ldcg(pr + c).x);
  }
  // group maximum: one barrier (the slots are not written again before the
  // next row's draw, which is behind later barriers)
  m = warp_max(m);
  if (lane == 0) shf[ew] = m;
  if (et == 0) *sFlag = 1;  // "no owner" until the owner clears it
  eg_sync();
  float M = shf[0];
#pragma unroll
  for (int i = 1; i < kPEpiWarps; ++i) M = fmaxf(M, shf[i]);
  const float kT = p.kT, Mk = __fmul_rn(M, kT);
  // chunk masses f_c = s_c * 2^((m_c - M) log2e/T) (one float32 rounding),
  // summed exactly as 2^-40 fixed-point integers
  unsigned long long local = 0ull;
  int last_pos = -1;
  unsigned long long fmass[kCache];  // this thread's chunk masses, reused by the crossing search
  if (cached) {
#pragma unroll
    for (int i = 0; i < kCache; ++i) {
      fmass[i] = i < c1 - c0 ? fx40(__fmul_rn(cache[i].y, pweight(cache[i].x, kT, Mk))) : 0ull;
      if (fmass[i]) last_pos = c0 + i;
      local += fmass[i];
    }
  } else {
    for (int c = c0; c < c1; ++c) {
      const float2 q = __ldcg(pr + c);
      const unsigned long long f = fx40(__fmul_rn(q.y, pweight(q.x, kT, Mk)));
      if (f) last_pos = c;
      local += f;
    }
  }
  // exclusive scan over the group: one barrier
  const unsigned long long xin = warp_inscan_u64(local, lane);
  if (lane == 31) shu[ew] = xin;
  eg_sync();
  unsigned long long before = 0ull, Z = 0ull;
#pragma unroll
  for (int i = 0; i < kPEpiWarps; ++i) {
    if (i < ew) before += shu[i];
    Z += shu[i];
  }
  const unsigned long long incl = before + xin, excl = incl - local;
  const unsigned long long target = scale_u53(odd, Z);
  if (excl <= target && target < incl) {  // the one thread whose segment holds the crossing
    unsigned long long run = excl, found_excl = excl;
    int found = -1;
    float found_g = 0.f, found_m = 0.f;
    if (cached) {
      int fi = -1;
#pragma unroll
      for (int i = 0; i < kCache; ++i) {
        if (fi < 0 && run + fmass[i] > target) { fi = i; found_excl = run; }
        run += fmass[i];
      }
      if (fi >= 0) {
        found = c0 + fi;
        float mq = 0.f;
#pragma unroll
        for (int i = 0; i < kCache; ++i) mq = i == fi ? cache[i].x : mq;  // static indexing
        found_g = pweight(mq, kT, Mk);
        found_m = mq;
      }
    } else {
      for (int c = c0; c < c1 && found < 0; ++c) {
        const float2 q = __ldcg(pr + c);
        const float g = pweight(q.x, kT, Mk);
        const unsigned long long f = fx40(__fmul_rn(q.y, g));
        if (run + f > target) { found = c; found_excl = run; found_g = g; found_m = q.x; }
        run += f;
      }
    }
    if (found < 0) {
      found = max(c0, last_pos);
      const float2 q = __ldcg(pr + found);
      found_g = pweight(q.x, kT, Mk);
      found_m = q.x;
    }
    *sExclU = found_excl;
    *sG = found_g;
    shf[0] = found_m;
    shi2[0] = found;
    *sFlag = 0;
  }
  eg_sync();
  int cstar;
  const int fallback = *sFlag;
  if (fallback) {  // no owner (cannot happen for Z > 0): last chunk with mass
    cstar = max(0, eg_max_i(last_pos, shi, ew, lane));
    if (et == 0) {
      const float2 q = __ldcg(pr + cstar);
      *sG = pweight(q.x, kT, Mk);
      *sExclU = 0ull;
      shf[0] = q.x;
    }
    eg_sync();
  } else {
    cstar = shi2[0];
  }
  const float mck = __fmul_rn(shf[0], kT);

  const int colbase = cstar * kChunk;
  if (stage_next && et == 0) {  // the candidate W1 rows, while the chunk is recomputed
    const uint32_t bytes = (uint32_t)(min(kChunk, p.V - colbase) * p.rank * 2);
    mbar_expect_tx(w1Full, bytes);
    bulk_load(ls + kLsW1Blk, p.W1 + (size_t)colbase * p.rank, bytes, w1Full);
    if (kGated) bulk_prefetch_l2(p.gate + (size_t)colbase * p.rank, bytes);  // the candidates' gate rows
  }
  // gated head: this step's state, read while the chunk is recomputed
  float gs[8];
  if (kGated && stage_next && ew == 0 && 8 * lane < p.rank) gated_state_k(p, r, k, lane, gs);
  // bias of the 64 columns of chunk cstar: thread (row group rg, 8-column unit uc)
  float bcol = 0.f;
  if (et < kChunk && colbase + et < p.V)
    bcol = __bfloat162float(p.base[((size_t)r * p.gamma + (k - 1)) * p.V + colbase + et]);
  {
    const int uc = et & 7, rg = et >> 3;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    if (colbase + uc * 8 < p.V) {
      uint4 w[8];
#pragma unroll
      for (int it = 0; it < 8; ++it) {  // rank <= 256: at most 8 rows per thread
        const int i = rg + 32 * it;
        w[it] = i < p.rank ? __ldg(reinterpret_cast<const uint4*>(p.W2 + (size_t)i * p.V + colbase + uc * 8))
                           : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int i = rg + 32 * it;
        const float w1 = i < p.rank ? sW1f[i] : 0.f;
        const uint32_t ww[4] = {w[it].x, w[it].y, w[it].z, w[it].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[2 * e] = __fmaf_rn(w1, __uint_as_float(ww[e] << 16), acc[2 * e]);
          acc[2 * e + 1] = __fmaf_rn(w1, __uint_as_float(ww[e] & 0xffff0000u), acc[2 * e + 1]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) red[rg][uc * 8 + e] = acc[e];
  }
  eg_sync();
  if (et < kChunk) {
    const int v = colbase + et;
    float w = 0.f;
    if (v < p.V) {
      float bias = 0.f;
#pragma unroll 8
      for (int g = 0; g < 32; ++g) bias = __fadd_rn(bias, red[g][et]);
      w = pweight(__fadd_rn(bcol, bias), kT, mck);
    }
    sW[et] = w;
  }
  eg_sync();
  if (ew == 0) {  // fixed-point prefix over the 64 weights: two per lane, warp scan
    const float g = *sG;
    const unsigned long long d0 = fx40(__fmul_rn(sW[2 * lane], g));
    const unsigned long long d1 = d0 + fx40(__fmul_rn(sW[2 * lane + 1], g));
    const unsigned long long x = warp_inscan_u64(d1, lane);
    unsigned long long ex = __shfl_up_sync(0xffffffffu, x, 1);
    if (lane == 0) ex = 0ull;
    const unsigned long long base_run = *sExclU + ex;
    int c = -1;
    if (!fallback) c = (base_run + d0 > target) ? 2 * lane : ((base_run + d1 > target) ? 2 * lane + 1 : -1);
    const unsigned hit = __ballot_sync(0xffffffffu, c >= 0);
    int xc;
    if (hit) {
      xc = __shfl_sync(0xffffffffu, c, __ffs(hit) - 1);
    } else {  // no crossing inside the chunk: last entry with weight
      const int lastw = sW[2 * lane + 1] > 0.f ? 2 * lane + 1 : (sW[2 * lane] > 0.f ? 2 * lane : -1);
      xc = max(0, warp_max_i(lastw));
    }
    const int tok = min(colbase + xc, p.V - 1);
    if (stage_next) {  // copy W1[tok] from the fetched chunk rows to the staging row
      uint4 zv = make_uint4(0, 0, 0, 0);
      if (kGated && 8 * lane < p.rank) zv = __ldg(reinterpret_cast<const uint4*>(p.gate + (size_t)tok * p.rank) + lane);
      mbar_wait_drain(w1Full, w1_use & 1, p.status);
      if (8 * lane < p.rank) {
        const uint4 wv = *reinterpret_cast<const uint4*>(sBlk + (size_t)(tok - colbase) * p.rank * 2 + 16 * lane);
        if (kGated) {
          gated_update8(gs, zv, wv);
          store_gcarry(p, r, lane, gs);
          stage[lane] = pack_bf16x8(gs);
        } else {
          stage[lane] = wv;
        }
        fence_proxy_async_global();
      }
    }
    if (lane == 0) {
      const float Zf = __fmul_rn((float)Z, 0x1p-40f);
      __stcg(p.tokens + out, tok);
      p.q_tok[out] = __fdiv_rn(__fmul_rn(sW[xc], g), Zf);
      p.q_stats[2 * out] = M;
      p.q_stats[2 * out + 1] = Zf;
    }
  }
  if (stage_next) ++w1_use;
  fence_proxy_async_smem();  // the scratch is overwritten next by a TMA load of the A operand
}

}  // namespace dspark

namespace dspark {

__device__ __forceinline__ ResidRow load_resid_row(const PersistParams& p, int r) {
  ResidRow rr;
  rr.kind = kPendNone;
  rr.A = 0;
  rr.MPk = rr.invZP = rr.MQk = rr.invZQ = 0.f;
  if (r < p.R) {
    const int4 pd = __ldg(p.pend + r);
    if (pd.x == kPendResid || pd.x == kPendBonus) {
      rr.kind = pd.x;
      rr.A = min(max(pd.y, 0), p.gamma);
      const float4 rs = __ldg(p.rowstat + (size_t)r * (p.gamma + 1) + rr.A);
      rr.MPk = __fmul_rn(rs.x, p.kT);
      rr.invZP = __frcp_rn(rs.y);
      if (rr.kind == kPendResid) {
        const size_t qi = 2 * ((size_t)r * p.gamma + min(rr.A, p.gamma - 1));
        rr.MQk = __fmul_rn(__ldg(p.q_stats + qi), p.kT);
        rr.invZQ = __frcp_rn(__ldg(p.q_stats + qi + 1));
      }
    }
  }
  return rr;
}

// Acceptance-label pass: row pr is the pair (request r = pr / gamma, position
// k = pr % gamma + 1): Q from the drafting stats of position k, P from target
// row k - 1; both rows of every pair are read (kind = residual).
__device__ __forceinline__ ResidRow load_label_row(const PersistParams& p, int pr) {
  ResidRow rr;
  rr.kind = kPendNone;
  rr.A = 0;
  rr.MPk = rr.invZP = rr.MQk = rr.invZQ = 0.f;
  if (pr < p.n_pairs) {
    const int r = pr / p.gamma, k1 = pr - r * p.gamma;
    rr.kind = kPendResid;
    rr.A = k1;
    const float4 rs = __ldg(p.rowstat + (size_t)r * (p.gamma + 1) + k1);
    rr.MPk = __fmul_rn(rs.x, p.kT);
    rr.invZP = __frcp_rn(rs.y);
    const size_t qi = 2 * ((size_t)r * p.gamma + k1);
    rr.MQk = __fmul_rn(__ldg(p.q_stats + qi), p.kT);
    rr.invZQ = __frcp_rn(__ldg(p.q_stats + qi + 1));
  }
  return rr;
}

__device__ __forceinline__ float unpack_bf16(const uint4& x, int e) {
  const uint32_t w = e < 2 ? x.x : (e < 4 ? x.y : (e < 6 ? x.z : x.w));
  return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
}

// Residual-pass staging of the target and base rows. Each epilogue warp owns
// 32 requests (its TMEM lane quarter) and a 12 KB slice of the staging region
// (the base ring and the third W2 stage of the drafting layout): three
// buffers of one half-chunk (32 columns) of both rows,
// 32 rows x 64 bytes per tensor, the 16-byte unit u of row m stored at
// m * 64 + ((u ^ ((m >> 1) & 3)) << 4) so the per-row reads are free of bank
// conflicts. The copies are cp.async (16 bytes each), four per tensor and
// lane, laid out so consecutive lanes read consecutive 16 bytes of one row;
// rows without a pending draw, base rows of bonus draws and columns past V are
// zero-filled without reading global memory.
constexpr int kRsBufs = 3;  // ring of half-chunk buffers per warp: copies run two ahead
constexpr uint32_t kRsBufBytes = 4096;
constexpr uint32_t kRsWarpBytes = kRsBufs * kRsBufBytes;
constexpr uint32_t kRsTensorBytes = 2048;
static_assert(2 * kPBStage + kPEpiWarps * kRsWarpBytes <= kPBStages * kPBStage + 2 * kPBaseStages * kPBaseBox,
              "the residual layout (2 W2 stages + row staging) fits where the drafting layout keeps 3 stages "
              "and the base ring");

// Label pass with TMA rows: the 128 pairs of an M tile are consecutive flat
// (request, position) indices, so a chunk's base rows are one box of the
// base logits viewed as [R * gamma][V], and its target rows one box of the
// target logits [R][gamma + 1][V] taking gamma positions of 128 / gamma
// requests. Three slots of (target box, base box) in the staging region,
// filled by warp 2 in chunk order. Every epilogue warp reads every chunk (its
// 32-column half) in the same order and the eight release the slot, so no
// warp ever waits on a slot's barrier more than one phase ahead (a parity
// wait cannot tell a phase two ahead from a completed one).
constexpr int kLSlots = 3;
constexpr uint32_t kLSlotBytes = 2 * kPBaseBox;
static_assert(kLSlots * kLSlotBytes <= kPEpiWarps * kRsWarpBytes, "the label slots fit the staging region");

struct ResidCopyRows {  // per lane: global rows of the four (copy, row) slots it serves
  int trow[4], brow[4];   // -1: zero fill
};

__device__ __forceinline__ ResidCopyRows resid_copy_rows(const PersistParams& p, const ResidRow& rr, int r, int lane) {
  const int my_t = rr.kind != kPendNone ? r * (p.gamma + 1) + rr.A : -1;
  const int my_b = rr.kind == kPendResid ? r * p.gamma + min(rr.A, p.gamma - 1) : -1;
  ResidCopyRows cr;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int src = c * 8 + (lane >> 2);
    cr.trow[c] = __shfl_sync(0xffffffffu, my_t, src);
    cr.brow[c] = __shfl_sync(0xffffffffu, my_b, src);
  }
  return cr;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// Issues the copies of one half-chunk (columns [v0, v0 + 32)) into `buf`, and
// commits them as one group (an empty group when v0 < 0).
__device__ __forceinline__ void resid_issue(const PersistParams& p, const ResidCopyRows& cr, int v0, int lane,
                                            uint32_t buf) {
  if (v0 >= 0) {
    const int u = lane & 3;
    const int v = v0 + 8 * u;
    const bool in = v < p.V;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int m = c * 8 + (lane >> 2);
      const uint32_t off = (uint32_t)(m * 64 + ((u ^ ((m >> 1) & 3)) << 4));
      const int tr = cr.trow[c], br = cr.brow[c];
      const __nv_bfloat16* ts = p.target + (size_t)max(tr, 0) * p.V + (in ? v : 0);
      const __nv_bfloat16* bs = p.base + (size_t)max(br, 0) * p.V + (in ? v : 0);
      cp_async16(buf + off, ts, (in && tr >= 0) ? 16u : 0u);
      cp_async16(buf + kRsTensorBytes + off, bs, (in && br >= 0) ? 16u : 0u);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Residual weights of one half-chunk of row m: the bias from TMEM (32
// columns), the target and base values from the staged buffer. Branch-free
// per element (residual and bonus rows share a warp): for a bonus draw Q is
// formed against a maximum of +inf, so it is exactly 0 and max(0, P - Q) = P,
// the same value resid_w returns; columns past V are masked to 0.
__device__ __forceinline__ void resid_half(const PersistParams& p, const ResidRow& rr, int v0, uint32_t taddr,
                                           const unsigned char* buf, int m, float (&sw)[4], float (&sp)[4]) {
  float acc[32];
  __syncwarp();
  tmem_ld32(taddr, acc);
  if (rr.kind == kPendNone) return;
  const bool res = rr.kind == kPendResid;
  const float kT = p.kT, MPk = rr.MPk, invZP = rr.invZP;
  const float MQk = res ? rr.MQk : INFINITY, invZQ = res ? rr.invZQ : 0.f;
  const int nvalid = p.V - v0;  // columns col < nvalid exist
#pragma unroll
  for (int u = 0; u < 4; ++u) {  // unit u feeds accumulator pair u: four independent chains
    const uint32_t off = (uint32_t)(m * 64 + ((u ^ ((m >> 1) & 3)) << 4));
    const uint4 tv = *reinterpret_cast<const uint4*>(buf + off);
    const uint4 bv = *reinterpret_cast<const uint4*>(buf + kRsTensorBytes + off);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int col = 8 * u + e;
      const float t = unpack_bf16(tv, e);
      const float l = __fadd_rn(unpack_bf16(bv, e), acc[col]);
      const float P = __fmul_rn(pweight(t, kT, MPk), invZP);
      const float Q = __fmul_rn(pweight(l, kT, MQk), invZQ);
      const bool in = col < nvalid;
      sw[u] += in ? fmaxf(0.f, __fsub_rn(P, Q)) : 0.f;
      sp[u] += in ? P : 0.f;
    }
  }
}

// The same weights for the label pass when its rows arrive by TMA: one slot
// holds a chunk's target box (128 pairs x 64 columns, 128-byte swizzle: the
// 16-byte unit u of row m at m * 128 + ((u ^ (m & 7)) << 4)) followed by its
// base box in the same layout; half hh is units 4 hh .. 4 hh + 3.
__device__ __forceinline__ void label_half_tma(const PersistParams& p, const ResidRow& rr, int v0, uint32_t taddr,
                                               const unsigned char* slot, int m, int hh, float (&sw)[4]) {
  float acc[32];
  __syncwarp();
  tmem_ld32(taddr, acc);
  if (rr.kind == kPendNone) return;
  const float kT = p.kT, MPk = rr.MPk, invZP = rr.invZP, MQk = rr.MQk, invZQ = rr.invZQ;
  const int nvalid = p.V - v0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint32_t off = (uint32_t)(m * 128 + (((4 * hh + u) ^ (m & 7)) << 4));
    const uint4 tv = *reinterpret_cast<const uint4*>(slot + off);
    const uint4 bv = *reinterpret_cast<const uint4*>(slot + kPBaseBox + off);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int col = 8 * u + e;
      const float t = unpack_bf16(tv, e);
      const float l = __fadd_rn(unpack_bf16(bv, e), acc[col]);
      const float P = __fmul_rn(pweight(t, kT, MPk), invZP);
      const float Q = __fmul_rn(pweight(l, kT, MQk), invZQ);
      sw[u] += col < nvalid ? fmaxf(0.f, __fsub_rn(P, Q)) : 0.f;
    }
  }
}

// Draws the corrected (first rejection) or bonus token of request r from the
// residual chunk sums: inverse CDF over the chunks, recompute of the crossing
// chunk, float64 prefix within it. Falls back to P when the residual has no
// mass.
__device__ void locate_resid_row(const PersistParams& p, int r, unsigned char* ls, int et, const uint64_t* odd_tab) {
  const int ew = et >> 5, lane = et & 31;
  float* sW1f = reinterpret_cast<float*>(ls + kLsW1);
  float(*red)[64] = reinterpret_cast<float(*)[64]>(ls + kLsRed);
  float* sW = reinterpret_cast<float*>(ls + kLsW);
  int* shi = reinterpret_cast<int*>(ls + kLsI);
  unsigned long long* shd = reinterpret_cast<unsigned long long*>(ls + kLsD);
  unsigned long long* sExcl = reinterpret_cast<unsigned long long*>(ls + kLsExcl);
  int* sFlag = reinterpret_cast<int*>(ls + kLsFlag);

  // the chunk sums, the request's pending record and the staged A row (W1[prev], or bf16(s_j) for the
  // gated head; rank <= 256, one element per thread) are independent loads: all issued first, the A row
  // kept in a register until the crossing chunk's bias needs it
  const int nc = p.nc;
  const float2* pr = p.rpart + (size_t)r * nc;
  unsigned long long* shu = shd;
  unsigned long long* sExclU = sExcl;
  const int seg = (nc + kPEpiThreads - 1) / kPEpiThreads;
  const int c0 = min(nc, et * seg), c1 = min(nc, c0 + seg);
  const bool cached = c1 - c0 <= kCache;
  float2 cache[kCache];
#pragma unroll
  for (int i = 0; i < kCache; ++i)
    cache[i] = (cached && i < c1 - c0) ? __ldcg(pr + c0 + i) : make_float2(0.f, 0.f);
  const uint32_t a_bits =
      et < p.rank ? (uint32_t)__ldcg(reinterpret_cast<const unsigned short*>(p.astage + (size_t)r * p.rank) + et) : 0u;
  const ResidRow rr = load_resid_row(p, r);
  if (rr.kind == kPendNone) return;  // same for every thread of the group
  auto getp = [&](int i) -> float2 { return cached ? cache[i] : __ldcg(pr + c0 + i); };
  unsigned long long lres = 0ull, lp = 0ull;
  if (cached) {
#pragma unroll
    for (int i = 0; i < kCache; ++i) { lres += fx40(cache[i].x); lp += fx40(cache[i].y); }
  } else {
    for (int c = c0; c < c1; ++c) {
      const float2 q = __ldcg(pr + c);
      lres += fx40(q.x);
      lp += fx40(q.y);
    }
  }
  unsigned long long W, incl;
  unsigned long long excl = eg_exscan_u64(lres, shu, W, ew, lane, incl);
  const bool use_p = W == 0ull;  // group-uniform: empty residual under rounding
  if (use_p) excl = eg_exscan_u64(lp, shu, W, ew, lane, incl);
  const int kind = use_p ? kPendBonus : rr.kind;
  const uint64_t purpose = rr.kind == kPendResid ? kResid : kBonus;
  const unsigned long long target =
      scale_u53(odd_tab ? *odd_tab : philox_odd53(p.seed, (uint64_t)r, (uint64_t)(rr.A + 1), purpose), W);
  if (et == 0) *sFlag = 1;
  if (rr.kind == kPendResid && et < p.rank) sW1f[et] = __uint_as_float(a_bits << 16);
  eg_sync();
  int last_pos = -1;
  if (cached) {
#pragma unroll
    for (int i = 0; i < kCache; ++i)
      if (i < c1 - c0 && fx40(use_p ? cache[i].y : cache[i].x)) last_pos = c0 + i;
  } else {
    for (int c = c0; c < c1; ++c)
      if (fx40(use_p ? __ldcg(pr + c).y : __ldcg(pr + c).x)) last_pos = c;
  }
  if (excl <= target && target < incl) {  // the one owner of the crossing
    unsigned long long run = excl, found_excl = excl;
    int found = -1;
    if (cached) {
#pragma unroll
      for (int i = 0; i < kCache; ++i)
        if (i < c1 - c0) {
          const unsigned long long f = fx40(use_p ? cache[i].y : cache[i].x);
          if (found < 0 && run + f > target) { found = c0 + i; found_excl = run; }
          run += f;
        }
    } else {
      for (int c = c0; c < c1 && found < 0; ++c) {
        const float2 q = getp(c - c0);
        const unsigned long long f = fx40(use_p ? q.y : q.x);
        if (run + f > target) { found = c; found_excl = run; }
        run += f;
      }
    }
    if (found < 0) found = max(c0, last_pos);
    *sExclU = found_excl;
    shi[0] = found;
    *sFlag = 0;
  }
  eg_sync();
  const int fallback = *sFlag;
  int cstar;
  if (fallback) {
    cstar = max(0, eg_max_i(last_pos, shi, ew, lane));
    if (et == 0) *sExclU = 0ull;
    eg_sync();
  } else {
    cstar = shi[0];
  }
  eg_sync();

  const int colbase = cstar * kChunk;
  float tcol = 0.f, bcol = 0.f;
  if (et < kChunk && colbase + et < p.V) {
    tcol = __bfloat162float(p.target[((size_t)r * (p.gamma + 1) + rr.A) * p.V + colbase + et]);
    if (kind == kPendResid)
      bcol = __bfloat162float(p.base[((size_t)r * p.gamma + min(rr.A, p.gamma - 1)) * p.V + colbase + et]);
  }
  if (kind == kPendResid) {  // bias of the 64 columns (group-uniform branch)
    const int uc = et & 7, rg = et >> 3;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    if (colbase + uc * 8 < p.V) {
      uint4 w[8];
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int i = rg + 32 * it;
        w[it] = i < p.rank ? __ldg(reinterpret_cast<const uint4*>(p.W2 + (size_t)i * p.V + colbase + uc * 8))
                           : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int i = rg + 32 * it;
        const float w1 = i < p.rank ? sW1f[i] : 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = __fmaf_rn(w1, unpack_bf16(w[it], e), acc[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) red[rg][uc * 8 + e] = acc[e];
  }
  eg_sync();
  if (et < kChunk) {
    float w = 0.f;
    if (colbase + et < p.V) {
      float bias = 0.f;
      if (kind == kPendResid) {
#pragma unroll 8
        for (int g = 0; g < 32; ++g) bias = __fadd_rn(bias, red[g][et]);
      }
      float P;
      w = resid_w(kind, tcol, __fadd_rn(bcol, bias), rr, p.kT, P);
    }
    sW[et] = w;
  }
  eg_sync();
  if (ew == 0) {
    const unsigned long long d0 = fx40(sW[2 * lane]);
    const unsigned long long d1 = d0 + fx40(sW[2 * lane + 1]);
    const unsigned long long x = warp_inscan_u64(d1, lane);
    unsigned long long ex = __shfl_up_sync(0xffffffffu, x, 1);
    if (lane == 0) ex = 0ull;
    const unsigned long long base_run = *sExclU + ex;
    int c = -1;
    if (!fallback) c = (base_run + d0 > target) ? 2 * lane : ((base_run + d1 > target) ? 2 * lane + 1 : -1);
    const unsigned hit = __ballot_sync(0xffffffffu, c >= 0);
    int xc;
    if (hit) {
      xc = __shfl_sync(0xffffffffu, c, __ffs(hit) - 1);
    } else {
      const int lastw = sW[2 * lane + 1] > 0.f ? 2 * lane + 1 : (sW[2 * lane] > 0.f ? 2 * lane : -1);
      xc = max(0, warp_max_i(lastw));
    }
    if (lane == 0) p.out_tokens[(size_t)r * (p.gamma + 1) + rr.A] = min(colbase + xc, p.V - 1);
  }
}

}  // namespace dspark

namespace dspark {

// kResid = false: the gamma drafting steps. kResid = true: one pass of the
// verifier's residual / bonus draw (A rows = W1[prev] of each request's
// first rejected position, per-request target and base rows read directly).
template <bool kResid, bool kLabel = false, bool kGated = false>
__global__ void __launch_bounds__(kPThreads, 1)
    persistent_sweep_kernel(const __grid_constant__ CUtensorMap mapW2, const __grid_constant__ CUtensorMap mapBase,
                            const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapT,
                            const __grid_constant__ PersistParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // drafting: A | 3 W2 stages | base ring; residual pass: A | 2 W2 stages |
  // row staging (the W2 ring gives up a stage to keep more rows in flight)
  constexpr int kBStages = kResid ? 2 : kPBStages;
  unsigned char* sA = smem;
  unsigned char* sB = sA + kPABytes;
  unsigned char* sBase = sB + kBStages * kPBStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sA + kPABytes + kPBStages * kPBStage + 2 * kPBaseStages * kPBaseBox);
  uint64_t* bFull = bars;
  uint64_t* bEmpty = bFull + kPBStages;
  uint64_t* baseFull = bEmpty + kPBStages;          // [half][stage]
  uint64_t* baseEmpty = baseFull + 2 * kPBaseStages;
  uint64_t* accFull = baseEmpty + 2 * kPBaseStages;
  uint64_t* accEmpty = accFull + 2;
  uint64_t* aFull = accEmpty + 2;  // [4]: one per 64-column K box of A
  uint64_t* drain = aFull + 4;
  uint64_t* w1Full = drain + 1;
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(w1Full + 1);
  volatile int* sAbort = reinterpret_cast<volatile int*>(sTmem + 1);
  volatile int* sDecide = reinterpret_cast<volatile int*>(sTmem + 2);  // epilogue-group verdict

  if (!kResid && p.sched_on && blockIdx.x >= (unsigned)p.n_cta) {
    side_cta_work(p, smem);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c_begin = (int)(((long long)blockIdx.x * p.nc) / p.n_cta);
  const int c_end = (int)(((long long)(blockIdx.x + 1) * p.nc) / p.n_cta);
  const int n_tiles = (c_end - c_begin + 3) / 4;
  const int nkc = p.rank / kPKC;
  const int n_steps = kResid ? 1 : p.gamma;

  if (tid == 0) {
    for (int i = 0; i < kPBStages; ++i) { mbar_init(&bFull[i], 1); mbar_init(&bEmpty[i], 1); }
    // base slots are released by the four warps of one epilogue half; the label pass's shared
    // slots by all eight (every warp reads every chunk there)
    const uint32_t empty_count = (kLabel && p.label_tma) ? kPEpiWarps : 4;
    for (int i = 0; i < 2 * kPBaseStages; ++i) { mbar_init(&baseFull[i], 1); mbar_init(&baseEmpty[i], empty_count); }
    for (int i = 0; i < 2; ++i) { mbar_init(&accFull[i], 1); mbar_init(&accEmpty[i], kPEpiWarps); }
    for (int i = 0; i < 4; ++i) mbar_init(&aFull[i], 1);
    mbar_init(drain, 1);
    mbar_init(w1Full, 1);
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
    if (lane == 0) {  // W2 producer: streams across steps, ahead of the tokens
      prefetch_tensormap(&mapW2);
      const uint64_t pol = l2_policy_evict_last();
      int n = 0;
      bool stop = false;
      for (int k = 1; k <= n_steps && !stop; ++k)
        for (int mt = 0; mt < p.n_mt && !stop; ++mt)
          for (int t = 0; t < n_tiles && !stop; ++t) {
            const int c0 = c_begin + 4 * t, nbox = min(4, c_end - c0);
            for (int kc = 0; kc < nkc; ++kc) {
              const int stage = n % kBStages;
              if (!mbar_wait(&bEmpty[stage], ((n / kBStages) & 1) ^ 1, sAbort, p.status)) { stop = true; break; }
              mbar_expect_tx(&bFull[stage], nbox * kPBBox);
              for (int j = 0; j < nbox; ++j)
                tma_load_2d(sB + stage * kPBStage + j * kPBBox, &mapW2, (c0 + j) * 64, kc * kPKC, &bFull[stage], pol);
              ++n;
            }
          }
      for (int i = 1; i <= kBStages && n - i >= 0; ++i)
        mbar_wait_drain(&bFull[(n - i) % kBStages], ((n - i) / kBStages) & 1, p.status);
    }
  } else if (warp == 2) {
    if (!kResid && lane == 0) {  // base-logit producer: chunk j of a tile -> ring of half j & 1
      prefetch_tensormap(&mapBase);
      const uint64_t pol = l2_policy_evict_first();
      const uint32_t bytes = (uint32_t)p.box_rows * 128;
      int nh[2] = {0, 0};
      bool stop = false;
      for (int k = 1; k <= n_steps && !stop; ++k)
        for (int mt = 0; mt < p.n_mt && !stop; ++mt)
          for (int t = 0; t < n_tiles && !stop; ++t) {
            const int c0 = c_begin + 4 * t, nbox = min(4, c_end - c0);
            for (int j = 0; j < nbox; ++j) {
              const int h = j & 1, n = nh[h], slot = h * kPBaseStages + n % kPBaseStages;
              if (!mbar_wait(&baseEmpty[slot], ((n / kPBaseStages) & 1) ^ 1, sAbort, p.status)) { stop = true; break; }
              mbar_expect_tx(&baseFull[slot], bytes);
              tma_load_3d(sBase + slot * kPBaseBox, &mapBase, (c0 + j) * 64, k - 1, mt * kPM, &baseFull[slot], pol);
              nh[h] = n + 1;
            }
          }
      for (int h = 0; h < 2; ++h)
        for (int i = 1; i <= kPBaseStages && nh[h] - i >= 0; ++i) {
          const int n = nh[h] - i;
          mbar_wait_drain(&baseFull[h * kPBaseStages + n % kPBaseStages], (n / kPBaseStages) & 1, p.status);
        }
    } else if (kLabel && p.label_tma && lane == 0) {  // label pass: target and base boxes, chunk order
      prefetch_tensormap(&mapBase);
      prefetch_tensormap(&mapT);
      const uint64_t pol = l2_policy_evict_first();
      const uint32_t bytes = (uint32_t)p.box_rows * 128;
      const int per_req = p.box_rows / p.gamma;  // requests per M tile of pairs
      int n = 0;
      bool stop = false;
      for (int mt = 0; mt < p.n_mt && !stop; ++mt)
        for (int t = 0; t < n_tiles && !stop; ++t) {
          const int c0 = c_begin + 4 * t, nbox = min(4, c_end - c0);
          for (int j = 0; j < nbox; ++j, ++n) {
            const int slot = n % kLSlots;
            if (!mbar_wait(&baseEmpty[slot], ((n / kLSlots) & 1) ^ 1, sAbort, p.status)) { stop = true; break; }
            mbar_expect_tx(&baseFull[slot], 2 * bytes);
            unsigned char* dst = sBase + (size_t)slot * kLSlotBytes;
            tma_load_3d(dst, &mapT, (c0 + j) * 64, 0, mt * per_req, &baseFull[slot], pol);
            tma_load_3d(dst + kPBaseBox, &mapBase, (c0 + j) * 64, mt * kPM, 0, &baseFull[slot], pol);
          }
        }
      for (int i = 1; i <= kLSlots && n - i >= 0; ++i)
        mbar_wait_drain(&baseFull[(n - i) % kLSlots], ((n - i) / kLSlots) & 1, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      int n = 0, T = 0, a_use = 0;
      bool stop = false;
      for (int k = 1; k <= n_steps && !stop; ++k)
        for (int mt = 0; mt < p.n_mt && !stop; ++mt) {
          // the A boxes are awaited one by one, as the first tile reaches them
          const uint32_t apar = (uint32_t)(a_use & 1);
          ++a_use;
          uint32_t a_ready = 0;
          for (int t = 0; t < n_tiles && !stop; ++t, ++T) {
            const int buf = T & 1;
            const uint32_t use = (uint32_t)(T >> 1);
            if (!mbar_wait(&accEmpty[buf], (use & 1) ^ 1, sAbort, p.status)) { stop = true; break; }
            tc_fence_after();
            const int c0 = c_begin + 4 * t, nbox = min(4, c_end - c0);
            const uint32_t idesc = idesc_bf16_f32(kPM, (uint32_t)(64 * nbox), 1);
            const uint32_t d = tmem + (uint32_t)(buf * 256);
            for (int kc = 0; kc < nkc; ++kc, ++n) {
              const int stage = n % kBStages;
              const int ka = (kc * kPKC) >> 6;
              if (!((a_ready >> ka) & 1u)) {
                if (!mbar_wait(&aFull[ka], apar, sAbort, p.status)) { stop = true; break; }
                a_ready |= 1u << ka;
              }
              if (!mbar_wait(&bFull[stage], (n / kBStages) & 1, sAbort, p.status)) { stop = true; break; }
              tc_fence_after();
              // K rows [kc * kPKC, +kPKC): A chunk of 64 K-columns, then 32-byte K16 steps inside it
              const unsigned char* a_k = sA + ((kc * kPKC) >> 6) * kPAChunk + (((kc * kPKC) & 63) >> 4) * 32;
              for (int kk = 0; kk < kPKC / 16; ++kk) {
                const uint64_t a_desc = smem_desc_sw128(smem_u32(a_k + kk * 32), 0, 1024);
                const uint64_t b_desc = smem_desc_sw128(smem_u32(sB + stage * kPBStage + kk * 2048), kPBBox, 1024);
                tc_mma_bf16(d, a_desc, b_desc, idesc, (kc | kk) != 0);
              }
              tc_commit(&bEmpty[stage]);
            }
            if (stop) break;
            tc_commit(&accFull[buf]);
          }
        }
      tc_commit(drain);
      mbar_wait_drain(drain, 0, p.status);
    }
  } else {
    // epilogue warps 3..10: A gather, softmax partials, grid barriers, locate
    const int et = tid - 96, ew = et >> 5;
    const bool ltma = kLabel && p.label_tma;  // label pass fed by TMA boxes (warp 2)
    // Philox draws of the CTA's first request for every step, computed once here instead of on the
    // draw's dependent path (many barriers pass before the first read)
    uint64_t* sOdd = reinterpret_cast<uint64_t*>(reinterpret_cast<unsigned char*>(bars) + kOddOffset);
    const bool odd_pre = !kResid && !p.greedy && p.gamma <= kOddCap && (int)blockIdx.x < p.R;
    if (odd_pre && et < p.gamma) sOdd[et] = philox_odd53(p.seed, (uint64_t)blockIdx.x, (uint64_t)(et + 1), kDraft);
    // residual pass: the one draw of the CTA's first request (its kind and position are inputs)
    const bool odd_res = kResid && !kLabel && !p.greedy && (int)blockIdx.x < p.R;
    if (odd_res && et == 0) {
      const ResidRow r0 = load_resid_row(p, blockIdx.x);
      if (r0.kind == kPendResid || r0.kind == kPendBonus)
        sOdd[0] = philox_odd53(p.seed, (uint64_t)blockIdx.x, (uint64_t)(r0.A + 1),
                               r0.kind == kPendResid ? Purpose::kResid : Purpose::kBonus);
    }
    const int q = warp & 3, h = (warp - 3) >> 2;
    const int row = 32 * q + lane;
    const float kT = p.kT;
    int T = 0, nh = 0;
    unsigned int epoch = 0;
    uint32_t w1_use = 0;
    uint32_t a_phases = 0;  // A-operand phases completed by this group (both gather paths)
    const uint64_t pol_a = l2_policy_evict_last();
    bool stop = false;
    for (int k = 1; k <= n_steps && !stop; ++k) {
      for (int mt = 0; mt < p.n_mt && !stop; ++mt) {
        // A = W1[prev] rows of this M tile (the previous MMAs on sA are done:
        // every tile of the previous tile sequence was received below)
        if (kResid || k > 1) {
          // drafting: the rows staged by the CTAs that drew the tokens of step
          // k - 1 (visible since the grid barrier); residual pass: the rows the
          // verifier's chain staged (previous launch). Four TMA boxes of 64
          // K-columns.
          if (et == 0) {
            const int nka = p.rank / 64;
            fence_proxy_async_global();
            for (int ka = 0; ka < 4; ++ka) {
              if (ka < nka) {
                mbar_expect_tx(&aFull[ka], (uint32_t)(p.box_rows * 128));
                tma_load_3d(sA + ka * kPAChunk, &mapA, ka * 64, mt * kPM, kResid ? 0 : (k - 1) & 1, &aFull[ka],
                            pol_a);
              } else {
                mbar_arrive(&aFull[ka]);  // unused box: keeps the four phases in step
              }
            }
          }
        } else {  // k == 1: the anchors' rows, two threads per row, 16 independent 16-byte loads each
          const int m = et >> 1, j0 = (et & 1) * 16, r = mt * kPM + m;
          int prev = -1;
          if (r < p.R) {
            prev = __ldg(p.anchor + r);
            if (prev < 0 || prev >= p.V) {
              set_status(p.status, DSPARK_ERR_RANGE);
              prev = min(max(prev, 0), p.V - 1);
            }
          }
          const uint4* src = reinterpret_cast<const uint4*>(p.W1 + (size_t)max(prev, 0) * p.rank);
          if (kGated) {  // gated head: s_1 = z[anchor] * W1[anchor] (exact), rounded to bf16
            const uint4* zsrc = reinterpret_cast<const uint4*>(p.gate + (size_t)max(prev, 0) * p.rank);
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
              uint4 wv[8], zv[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int j = j0 + 8 * hh + i;
                const bool ok = prev >= 0 && 8 * j < p.rank;
                wv[i] = ok ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
                zv[i] = ok ? __ldg(zsrc + j) : make_uint4(0, 0, 0, 0);
              }
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int j = j0 + 8 * hh + i, kc = j >> 3, uu = j & 7;
                float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                gated_update8(s8, zv[i], wv[i]);
                *reinterpret_cast<uint4*>(sA + kc * kPAChunk + m * 128 + ((uu ^ (m & 7)) << 4)) = pack_bf16x8(s8);
              }
            }
          } else {
            uint4 val[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              val[i] = (prev >= 0 && 8 * (j0 + i) < p.rank) ? __ldg(src + j0 + i) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j = j0 + i, kc = j >> 3, uu = j & 7;
              *reinterpret_cast<uint4*>(sA + kc * kPAChunk + m * 128 + ((uu ^ (m & 7)) << 4)) = val[i];
            }
          }
          fence_proxy_async_smem();
          eg_sync();
          if (et == 0)
            for (int ka = 0; ka < 4; ++ka) mbar_arrive(&aFull[ka]);
        }
        ++a_phases;

        ResidRow rr{};
        ResidCopyRows cr{};
        // residual pass: this warp's half-chunk sequence s = 0, 1, ...: chunk
        // kth = s >> 1 of this half (c_begin + 4 (kth >> 1) + h + 2 (kth & 1)),
        // columns 32 (s & 1) .. +32; copies run one half-chunk ahead
        const uint32_t rs_base = smem_u32(sBase) + (uint32_t)ew * kRsWarpBytes;
        auto hc_col = [&](int sidx) -> int {
          const int kth = sidx >> 1, c = c_begin + 4 * (kth >> 1) + h + 2 * (kth & 1);
          return c < c_end ? c * 64 + 32 * (sidx & 1) : -1;
        };
        int hs = 0;
        unsigned long long lacc = 0ull;  // label pass: this thread's 2^-40 sum over its chunks
        const int pr = mt * kPM + row;   // the request (residual) or the (request, position) pair (labels)
        if (kResid) {
          __syncwarp();  // the previous M tile's reads of the buffers are done
          rr = kLabel ? load_label_row(p, pr) : load_resid_row(p, pr);
          if (!ltma) {
            cr = resid_copy_rows(p, rr, kLabel ? pr / p.gamma : pr, lane);
            resid_issue(p, cr, hc_col(0), lane, rs_base);
            resid_issue(p, cr, hc_col(1), lane, rs_base + kRsBufBytes);
          }
        }
        for (int t = 0; t < n_tiles; ++t, ++T) {
          const int buf = T & 1;
          const uint32_t use = (uint32_t)(T >> 1);
          const int c0 = c_begin + 4 * t, nbox = min(4, c_end - c0);
          if (!__all_sync(0xffffffffu, mbar_wait(&accFull[buf], use & 1, sAbort, p.status))) { stop = true; break; }
          tc_fence_after();
          // label pass with TMA rows: every warp takes every chunk of the tile (its half h of the 64
          // columns), so each warp waits on the shared slots in chunk order and is never more than
          // one phase ahead of a slot's barrier; otherwise half h takes chunks h, h + 2
          for (int j = ltma ? 0 : h; j < nbox; j += ltma ? 1 : 2) {
            if (kResid) {
              const int r = mt * kPM + row;
              float sw[4] = {0.f, 0.f, 0.f, 0.f}, sp[4] = {0.f, 0.f, 0.f, 0.f};
              if (ltma) {  // this chunk's slot: chunk number n of the CTA's chunk sequence
                const int n = mt * (c_end - c_begin) + 4 * t + j, slot = n % kLSlots;
                if (!__all_sync(0xffffffffu, mbar_wait(&baseFull[slot], (n / kLSlots) & 1, sAbort, p.status))) {
                  stop = true;
                  break;
                }
                const unsigned char* sl = sBase + (size_t)slot * kLSlotBytes;
                label_half_tma(p, rr, (c0 + j) * 64 + 32 * h,
                               tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * 256 + j * 64 + 32 * h), sl, row,
                               h, sw);
                __syncwarp();
                if (lane == 0) mbar_arrive(&baseEmpty[slot]);
              } else {
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh, ++hs) {
                  __syncwarp();  // every lane is done with the buffer the next copies overwrite
                  resid_issue(p, cr, hc_col(hs + 2), lane, rs_base + (uint32_t)((hs + 2) % kRsBufs) * kRsBufBytes);
                  asm volatile("cp.async.wait_group 2;" ::: "memory");
                  __syncwarp();
                  resid_half(p, rr, (c0 + j) * 64 + 32 * hh,
                             tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * 256 + j * 64 + 32 * hh),
                             sBase + (size_t)ew * kRsWarpBytes + (size_t)(hs % kRsBufs) * kRsBufBytes, lane, sw, sp);
                }
              }
              if (kLabel) {
                if (rr.kind != kPendNone) lacc += fx40((sw[0] + sw[1]) + (sw[2] + sw[3]));
              } else if (rr.kind != kPendNone) {
                __stcg(p.rpart + (size_t)r * p.nc + (c0 + j),
                       make_float2((sw[0] + sw[1]) + (sw[2] + sw[3]), (sp[0] + sp[1]) + (sp[2] + sp[3])));
              }
              continue;
            }
            const int s = h * kPBaseStages + nh % kPBaseStages;
            if (!__all_sync(0xffffffffu, mbar_wait(&baseFull[s], (nh / kPBaseStages) & 1, sAbort, p.status))) {
              stop = true;
              break;
            }
            ++nh;
            const unsigned char* brow = sBase + s * kPBaseBox + row * 128;
            const int vbase = (c0 + j) * 64;
            float m, ssum = 0.f;
            int am = 0x7fffffff;
            uint32_t accr[64];
            __syncwarp();
            // the accumulator load lands while the base logits are read from shared memory; both
            // buffers are given back as soon as their values are in registers. For the base slot
            // that is made explicit: each lane first stores a value that needs all eight of its
            // loads, and the release (which orders stores) follows the warp's stores. Releasing
            // right after the loads were issued let some drafts read a slot the next box had
            // already overwritten.
            tmem_ld64_nowait(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * 256 + j * 64), accr);
            uint4 bx[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) bx[u] = *reinterpret_cast<const uint4*>(brow + ((u ^ (row & 7)) << 4));
            tmem_ld_wait64(accr);
            {
              uint32_t dep = 0;
#pragma unroll
              for (int u = 0; u < 8; ++u) dep ^= bx[u].x ^ bx[u].w;
              *reinterpret_cast<volatile uint32_t*>(reinterpret_cast<unsigned char*>(bars) + kDepOffset + 4 * ew) = dep;
              __syncwarp();
              if (lane == 0) mbar_arrive(&baseEmpty[s]);
            }
            if (j + 2 >= nbox) {  // this half's last chunk of the tile: the accumulator is free
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&accEmpty[buf]);
            }
            float l[64];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint32_t w[4] = {bx[u].x, bx[u].y, bx[u].z, bx[u].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                l[8 * u + 2 * e] = __fadd_rn(__uint_as_float(w[e] << 16), __uint_as_float(accr[8 * u + 2 * e]));
                l[8 * u + 2 * e + 1] =
                    __fadd_rn(__uint_as_float(w[e] & 0xffff0000u), __uint_as_float(accr[8 * u + 2 * e + 1]));
              }
            }
            if (vbase + 64 > p.V) {
#pragma unroll
              for (int i = 0; i < 64; ++i)
                if (vbase + i >= p.V) l[i] = -INFINITY;
            }
            if (p.greedy) {
              m = -INFINITY;
#pragma unroll
              for (int i = 0; i < 64; ++i)
                if (l[i] > m) { m = l[i]; am = vbase + i; }
            } else {
              // one pass: the chunk maximum (exact in any order), then the weights
              // relative to it in eight independent chains (a float32 chunk partial)
              float mq[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) mq[i] = l[i];
#pragma unroll
              for (int i = 8; i < 64; ++i) mq[i & 7] = fmaxf(mq[i & 7], l[i]);
              m = fmaxf(fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])), fmaxf(fmaxf(mq[4], mq[5]), fmaxf(mq[6], mq[7])));
              const float mk = __fmul_rn(m, kT);
              // chain c = i & 7 adds the weights of i = c, c + 8, ... in order; the pairs (i, i + 1) of
              // chains (c, c + 1) go through one f32x2 fma each (the argument; the sum as an fma by 1.0):
              // the same operations, in the same order, as eight scalar chains
              const unsigned long long k2 = f32x2_pack(kT, kT), nmk2 = f32x2_pack(-mk, -mk),
                                       one2 = f32x2_pack(1.f, 1.f);
              unsigned long long sq2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
              for (int i = 0; i < 64; i += 2) {
                float a0, a1;
                f32x2_unpack(f32x2_fma(f32x2_pack(l[i], l[i + 1]), k2, nmk2), a0, a1);
                sq2[(i & 7) >> 1] = f32x2_fma(f32x2_pack(px2(a0), px2(a1)), one2, sq2[(i & 7) >> 1]);
              }
              float s0, s1, s2, s3, s4, s5, s6, s7;
              f32x2_unpack(sq2[0], s0, s1);
              f32x2_unpack(sq2[1], s2, s3);
              f32x2_unpack(sq2[2], s4, s5);
              f32x2_unpack(sq2[3], s6, s7);
              ssum = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
            }
            const int r = mt * kPM + row;
            if (r < p.R)
              __stcg(p.part + (size_t)r * p.nc + (c0 + j),
                     p.greedy ? make_float2(m, __int_as_float(am)) : make_float2(m, ssum));
          }
          if (kResid || h >= nbox) {  // residual / label mode, or a half with no chunk in this tile
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&accEmpty[buf]);
          }
          if (stop) break;
        }
        if (kLabel && lacc) atomicAdd(p.lsum + pr, lacc);  // exact, order-free: deterministic
      }
      // The group never leaves the loop on one warp's say-so: every warp
      // reaches each named barrier, and the verdict written by one thread
      // between two barriers is read by all.
      if (stop) *sAbort = 1;
      eg_sync();
      if (et == 0) {  // every CTA has written its partials of step k
        ++epoch;
        *sDecide = (*sAbort || !grid_barrier(p.gbar, epoch * (unsigned)p.n_cta, p.status, sAbort)) ? 1 : 0;
      }
      eg_sync();
      if (*sDecide) break;
      if (kLabel) {  // every CTA's sums are in: c* = 1 - sum max(0, P - Q), and the sums back to zero
        for (int q2 = blockIdx.x * kPEpiThreads + et; q2 < p.n_pairs; q2 += p.n_cta * kPEpiThreads) {
          const unsigned long long v = atomicExch(p.lsum + q2, 0ull);
          p.labels[q2] = (float)(1.0 - (double)v * 0x1p-40);
        }
        continue;
      }
      for (int r = blockIdx.x; r < p.R; r += p.n_cta) {
        if (kResid)
          locate_resid_row(p, r, sA, et, (odd_res && r == (int)blockIdx.x) ? sOdd : nullptr);
        else
          locate_row<kGated>(p, r, k, sA, et, w1Full, w1_use, (odd_pre && r == (int)blockIdx.x) ? sOdd : nullptr);
        eg_sync();
      }
      if (!kResid) {
        eg_sync();
        if (et == 0) {  // every CTA has written its tokens of step k
          ++epoch;
          *sDecide = (*sAbort || !grid_barrier(p.gbar, epoch * (unsigned)p.n_cta, p.status, sAbort)) ? 1 : 0;
        }
        eg_sync();
        if (*sDecide) break;
      }
    }
    // the rows still queued and the chains; the test is the group's verdict of the last barrier, the same
    // for every warp (a warp's own `stop` is not: the work has named barriers)
    if (!kResid && p.vfuse && !*sDecide) after_sweep_work(p, ew, lane, sB, reinterpret_cast<unsigned char*>(bars));
    if (kResid) asm volatile("cp.async.wait_all;" ::: "memory");  // no copy outlives the CTA
    if (et == 0 && a_phases > 0)  // nor an A box the MMA issuer stopped waiting for
      for (int ka = 0; ka < 4; ++ka) mbar_wait_drain(&aFull[ka], (a_phases - 1) & 1, p.status);
    *sAbort = (*sAbort) | (stop ? 1 : 0);  // let the other roles wind down
    (void)ew;
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

namespace dspark {

// Shapes the tensor-core sweep takes: bf16, rank a multiple of 64 up to 256
// (whole 64-column K boxes of A, at most 8 rows per thread in the draw), V a
// multiple of 8 (16-byte TMA row strides) and at least 64 (one column box),
// and 16-byte aligned tensors.
bool draft_tc_eligible(const DraftArgs& a) {
  return a.dtype == DSPARK_BF16 && a.rank % 64 == 0 && a.rank <= 256 && a.V % 8 == 0 && a.V >= 64 &&
         (reinterpret_cast<uintptr_t>(a.base) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.W1) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(a.W2) & 15) == 0;
}

cudaError_t launch_draft_persistent(const DraftArgs& a, cudaStream_t s, int& launches, bool& taken) {
  taken = false;
  if (!draft_tc_eligible(a)) return cudaSuccess;
  int dev = 0, coop = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaSuccess;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (!coop || sms <= 0) return cudaSuccess;
  static std::atomic<unsigned long long> attr{0}, attr_gated{0};
  // the recurrent (gated) head is its own instantiation: the Markov kernel carries none of its code
  const void* fn = a.gate ? (const void*)persistent_sweep_kernel<false, false, true>
                          : (const void*)persistent_sweep_kernel<false>;
  if (set_smem_limit_once(fn, (int)kPSmem, a.gate ? attr_gated : attr) != cudaSuccess)
    return cudaSuccess;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kPThreads, kPSmem) !=
          cudaSuccess ||
      per_sm < 1)
    return cudaSuccess;
  CUtensorMap mapW2, mapBase;
  {
    const uint64_t dims[2] = {(uint64_t)a.V, (uint64_t)a.rank};
    const uint64_t strides[1] = {(uint64_t)a.V * 2};
    const uint32_t box[2] = {64, (uint32_t)kPKC};
    if (!make_tmap_bf16(&mapW2, a.W2, 2, dims, strides, box)) return cudaSuccess;
  }
  const int box_rows = a.R < kPM ? a.R : kPM;
  {
    const uint64_t dims[3] = {(uint64_t)a.V, (uint64_t)a.gamma, (uint64_t)a.R};
    const uint64_t strides[2] = {(uint64_t)a.V * 2, (uint64_t)a.gamma * a.V * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)box_rows};
    if (!make_tmap_bf16(&mapBase, a.base, 3, dims, strides, box)) return cudaSuccess;
  }
  const WsLayout L = ws_layout(a.R, a.gamma, a.V);
  CUtensorMap mapA;  // staged W1 rows [2][R][rank], one box = 64 K-columns of 128 requests
  {
    const uint64_t dims[3] = {(uint64_t)a.rank, (uint64_t)a.R, 2};
    const uint64_t strides[2] = {(uint64_t)a.rank * 2, (uint64_t)a.R * a.rank * 2};
    const uint32_t box[3] = {64, (uint32_t)box_rows, 1};
    if (!make_tmap_bf16(&mapA, ws_at<void>(a.ws, L.astage), 3, dims, strides, box)) return cudaSuccess;
  }
  PersistParams p{};
  p.R = a.R; p.gamma = a.gamma; p.V = a.V; p.rank = a.rank;
  p.nc = ceil_div(a.V, kChunk);
  // with a schedule, one CTA slot is the scheduler's: the sweep takes the others
  const int slots = sms * per_sm;
  const bool sched = a.sched != nullptr && slots >= 2;
  const int sweep_slots = sched ? slots - 1 : slots;
  p.n_cta = p.nc < sweep_slots ? p.nc : sweep_slots;
  // with verification in the launch, the sweep keeps the fewest CTAs that leave its largest shares (chunks
  // and requests per CTA) as they are, and up to kRowCtasMax of the slots left stream row statistics
  const bool vfuse = sched && a.verify != nullptr && (reinterpret_cast<uintptr_t>(a.verify->target) & 15) == 0;
  int n_row_ctas = 0;
  if (vfuse) {
    const int per_c = ceil_div(p.nc, p.n_cta), per_r = ceil_div(a.R, p.n_cta);
    const int need = std::max(ceil_div(p.nc, per_c), ceil_div(a.R, per_r));
    p.n_cta = std::min(p.n_cta, need);
    n_row_ctas = std::min(slots - 1 - p.n_cta, kRowCtasMax);
  }
  p.n_mt = ceil_div(a.R, kPM);
  p.box_rows = box_rows;
  p.greedy = a.temperature == 0.f;
  p.kT = p.greedy ? 0.f : (float)(1.4426950408889634 / (double)a.temperature);
  p.seed = a.seed;
  p.W1 = static_cast<const __nv_bfloat16*>(a.W1);
  p.W2 = static_cast<const __nv_bfloat16*>(a.W2);
  p.base = static_cast<const __nv_bfloat16*>(a.base);
  p.anchor = a.anchor;
  p.tokens = a.tokens;
  p.q_tok = a.q_tok;
  p.q_stats = a.q_stats;
  p.part = ws_at<float2>(a.ws, L.dpart);
  p.status = ws_at<uint32_t>(a.ws, L.status);
  p.gbar = reinterpret_cast<unsigned int*>(p.status + 1);
  p.astage = ws_at<__nv_bfloat16>(a.ws, L.astage);
  p.gate = static_cast<const __nv_bfloat16*>(a.gate);
  p.gcarry = ws_at<float>(a.ws, L.gcarry);
  if (sched) {  // the round's schedule, by the launch's extra CTA
    const ScheduleArgs& sa = *a.sched;
    p.sched_on = 1;
    p.conf = sa.conf;
    p.conf_lag = sa.conf_lagged;
    p.sps = sa.sps;
    p.n_table = sa.n_table;
    p.sched_mode = sa.mode;
    p.sched_len = sa.sched_len;
    p.sched_K = sa.K;
    p.tau_theta = sa.tau_theta;
    p.skey0 = ws_at<uint32_t>(a.ws, L.skey0);
    p.skey1 = ws_at<uint32_t>(a.ws, L.skey1);
    p.sidx0 = ws_at<uint32_t>(a.ws, L.sidx0);
    p.sidx1 = ws_at<uint32_t>(a.ws, L.sidx1);
    p.sched_fx = ws_at<unsigned long long>(a.ws, L.fx);
  }
  if (vfuse) {
    const VerifyArgs& va = *a.verify;
    p.vfuse = 1;
    p.target = static_cast<const __nv_bfloat16*>(va.target);
    p.rowstat = ws_at<float4>(a.ws, L.rowstat);
    p.vpieces = ws_at<float4>(a.ws, L.vsplit);
    p.row_cnt = ws_at<unsigned int>(a.ws, L.vcount);
    p.req_cnt = p.row_cnt + (size_t)a.R * (a.gamma + 1);
    p.vlist = ws_at<uint32_t>(a.ws, L.vlist);
    p.p_tok = va.p_tok;
    p.out_tokens = va.out_tokens;
    p.accepted_len = va.accepted_len;
    p.pend = ws_at<int4>(a.ws, L.pend);
    p.stage_rank = a.gate ? 0 : a.rank;  // the gated head's A rows are staged after the launch
  }
  taken = true;
  // the grid-barrier counter, and with verification in the launch its ready and queue words
  cudaError_t e = cudaMemsetAsync(p.gbar, 0, (vfuse ? kVQueueWord : 1) * sizeof(unsigned int), s);
  if (e != cudaSuccess) return e;
  if (sched && a.sched_done) *a.sched_done = true;
  if (vfuse && a.verify_done) *a.verify_done = true;
  void* args[] = {&mapW2, &mapBase, &mapA, &mapW2, &p};  // no target map in this mode
  e = cudaLaunchCooperativeKernel(fn, dim3(p.n_cta + (sched ? 1 : 0) + n_row_ctas), dim3(kPThreads), args, kPSmem,
                                  s);
  launches += 1;
  return e;
}

}  // namespace dspark

namespace dspark {

// Runs one of the kernels' bounded waits on a condition that nothing ever
// meets, so that it gives up: `which` 0 = the grid barrier (a counter target
// no launch reaches), 1 = an mbarrier phase that no arrival completes, 2 = the
// acquire poll on a counter another CTA advances (a target no one reaches). The
// wait records DSPARK_ERR_TIMEOUT in the status word and the kernel returns;
// nothing traps and the context stays usable.
__global__ void wait_selftest_kernel(int which, uint32_t* status, unsigned int* counter) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  if (which == 0) {
    grid_barrier(counter, 0xFFFFFFFFu, status, &abort_flag);
  } else if (which == 2) {
    wait_count(counter, 0xFFFFFFFFu, status);  // the poll on another CTA's counter (row list, rows done)
  } else {
    mbar_init(&bar, 1);
    mbar_fence_init();
    mbar_wait(&bar, 0, &abort_flag, status);  // phase 0 never completes: no arrival
  }
}

bool gated_supported(const DraftArgs& a) {
  if (!a.gate || !draft_tc_eligible(a) || (reinterpret_cast<uintptr_t>(a.gate) & 15) != 0) return false;
  int dev = 0, coop = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  return coop != 0;
}

// The verifier's residual / bonus draw on the tensor cores: one cooperative
// launch of the sweep kernel in residual mode. Returns taken = false (and
// launches nothing) when the shape or the device does not allow it.
cudaError_t launch_resid_persistent(const VerifyArgs& a, cudaStream_t s, int& launches, bool& taken) {
  taken = false;
  if (a.temperature == 0.f) return cudaSuccess;
  DraftArgs d{a.R, a.gamma, a.V, a.rank, a.dtype, a.base, a.anchor, a.W1, a.W2, a.temperature, a.seed,
              nullptr, nullptr, nullptr, a.ws};
  if (!draft_tc_eligible(d) || (reinterpret_cast<uintptr_t>(a.target) & 15) != 0) return cudaSuccess;
  int dev = 0, coop = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaSuccess;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (!coop || sms <= 0) return cudaSuccess;
  static std::atomic<unsigned long long> attr{0};
  if (set_smem_limit_once((const void*)persistent_sweep_kernel<true>, (int)kPSmem, attr) != cudaSuccess)
    return cudaSuccess;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, persistent_sweep_kernel<true>, kPThreads, kPSmem) !=
          cudaSuccess ||
      per_sm < 1)
    return cudaSuccess;
  CUtensorMap mapW2;
  {
    const uint64_t dims[2] = {(uint64_t)a.V, (uint64_t)a.rank};
    const uint64_t strides[1] = {(uint64_t)a.V * 2};
    const uint32_t box[2] = {64, (uint32_t)kPKC};
    if (!make_tmap_bf16(&mapW2, a.W2, 2, dims, strides, box)) return cudaSuccess;
  }
  const WsLayout L = ws_layout(a.R, a.gamma, a.V);
  CUtensorMap mapA;  // the A rows the verifier staged in astage[0]
  {
    const uint64_t dims[3] = {(uint64_t)a.rank, (uint64_t)a.R, 2};
    const uint64_t strides[2] = {(uint64_t)a.rank * 2, (uint64_t)a.R * a.rank * 2};
    const uint32_t box[3] = {64, (uint32_t)(a.R < kPM ? a.R : kPM), 1};
    if (!make_tmap_bf16(&mapA, ws_at<void>(a.ws, L.astage), 3, dims, strides, box)) return cudaSuccess;
  }
  PersistParams p{};
  p.R = a.R; p.gamma = a.gamma; p.V = a.V; p.rank = a.rank;
  p.nc = ceil_div(a.V, kChunk);
  p.n_cta = p.nc < sms ? p.nc : sms;
  p.n_mt = ceil_div(a.R, kPM);
  p.box_rows = a.R < kPM ? a.R : kPM;
  p.greedy = 0;
  p.kT = (float)(1.4426950408889634 / (double)a.temperature);
  p.seed = a.seed;
  p.W1 = static_cast<const __nv_bfloat16*>(a.W1);
  p.W2 = static_cast<const __nv_bfloat16*>(a.W2);
  p.base = static_cast<const __nv_bfloat16*>(a.base);
  p.anchor = a.anchor;
  p.q_stats = const_cast<float*>(a.q_stats);
  p.status = ws_at<uint32_t>(a.ws, L.status);
  p.gbar = reinterpret_cast<unsigned int*>(p.status + 1);
  p.target = static_cast<const __nv_bfloat16*>(a.target);
  p.pend = ws_at<int4>(a.ws, L.pend);
  p.rowstat = ws_at<float4>(a.ws, L.rowstat);
  p.out_tokens = a.out_tokens;
  p.rpart = ws_at<float2>(a.ws, L.rpart);
  p.astage = ws_at<__nv_bfloat16>(a.ws, L.astage);
  taken = true;
  cudaError_t e = cudaMemsetAsync(p.gbar, 0, sizeof(unsigned int), s);
  if (e != cudaSuccess) return e;
  void* args[] = {&mapW2, &mapW2, &mapA, &mapW2, &p};  // no base or target map in residual mode
  e = cudaLaunchCooperativeKernel((const void*)persistent_sweep_kernel<true>, dim3(p.n_cta), dim3(kPThreads), args,
                                  kPSmem, s);
  launches += 1;
  return e;
}

}  // namespace dspark

namespace dspark {

// The acceptance-label pass: one cooperative launch of the sweep in label
// mode over ceil(R * gamma / 128) M tiles of (request, position) pairs. The
// row stats of target rows 0..gamma-1 and the staged W1 rows of every pair
// must already be in the workspace. taken = false when the shape or the device
// does not allow it (nothing is launched).
cudaError_t launch_label_persistent(const LabelArgs& a, cudaStream_t s, int& launches, bool& taken) {
  taken = false;
  DraftArgs d{a.R, a.gamma, a.V, a.rank, a.dtype, a.base, a.anchor, a.W1, a.W2, a.temperature, 0,
              nullptr, nullptr, nullptr, a.ws};
  if (a.temperature == 0.f || !draft_tc_eligible(d) || (reinterpret_cast<uintptr_t>(a.target) & 15) != 0)
    return cudaSuccess;
  int dev = 0, coop = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaSuccess;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (!coop || sms <= 0) return cudaSuccess;
  static std::atomic<unsigned long long> attr{0};
  if (set_smem_limit_once((const void*)persistent_sweep_kernel<true, true>, (int)kPSmem, attr) != cudaSuccess)
    return cudaSuccess;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, persistent_sweep_kernel<true, true>, kPThreads,
                                                    kPSmem) != cudaSuccess ||
      per_sm < 1)
    return cudaSuccess;
  const int n_pairs = a.R * a.gamma;
  CUtensorMap mapW2, mapA;
  {
    const uint64_t dims[2] = {(uint64_t)a.V, (uint64_t)a.rank};
    const uint64_t strides[1] = {(uint64_t)a.V * 2};
    const uint32_t box[2] = {64, (uint32_t)kPKC};
    if (!make_tmap_bf16(&mapW2, a.W2, 2, dims, strides, box)) return cudaSuccess;
  }
  const WsLayout L = ws_layout(a.R, a.gamma, a.V);
  {  // staged W1 rows [R * gamma][rank] as a 3D map with a unit z extent
    const uint64_t dims[3] = {(uint64_t)a.rank, (uint64_t)n_pairs, 1};
    const uint64_t strides[2] = {(uint64_t)a.rank * 2, (uint64_t)n_pairs * a.rank * 2};
    const uint32_t box[3] = {64, (uint32_t)(n_pairs < kPM ? n_pairs : kPM), 1};
    if (!make_tmap_bf16(&mapA, ws_at<void>(a.ws, L.lstage), 3, dims, strides, box)) return cudaSuccess;
  }
  PersistParams p{};
  p.R = a.R; p.gamma = a.gamma; p.V = a.V; p.rank = a.rank;
  p.nc = ceil_div(a.V, kChunk);
  p.n_cta = p.nc < sms ? p.nc : sms;
  p.n_mt = ceil_div(n_pairs, kPM);
  p.box_rows = n_pairs < kPM ? n_pairs : kPM;
  p.greedy = 0;
  p.kT = (float)(1.4426950408889634 / (double)a.temperature);
  p.W1 = static_cast<const __nv_bfloat16*>(a.W1);
  p.W2 = static_cast<const __nv_bfloat16*>(a.W2);
  p.base = static_cast<const __nv_bfloat16*>(a.base);
  p.anchor = a.anchor;
  p.q_stats = const_cast<float*>(a.q_stats);
  p.status = ws_at<uint32_t>(a.ws, L.status);
  p.gbar = reinterpret_cast<unsigned int*>(p.status + 1);
  p.target = static_cast<const __nv_bfloat16*>(a.target);
  p.rowstat = ws_at<float4>(a.ws, L.rowstat);
  p.n_pairs = n_pairs;
  p.lsum = ws_at<unsigned long long>(a.ws, L.lsum);
  p.labels = a.labels;
  // rows by TMA when a tile's pairs are whole requests' position ranges (gamma divides the tile's rows)
  CUtensorMap mapBL = mapW2, mapT = mapW2;
  bool ltma = p.box_rows % a.gamma == 0 && (reinterpret_cast<uintptr_t>(a.base) & 15) == 0;
  if (ltma) {  // base logits as [R * gamma][V] in pair order; a box = 64 columns of box_rows pairs
    const uint64_t dims[3] = {(uint64_t)a.V, (uint64_t)n_pairs, 1};
    const uint64_t strides[2] = {(uint64_t)a.V * 2, (uint64_t)n_pairs * a.V * 2};
    const uint32_t box[3] = {64, (uint32_t)p.box_rows, 1};
    ltma = make_tmap_bf16(&mapBL, a.base, 3, dims, strides, box);
  }
  if (ltma) {  // target rows 0..gamma-1 of each request; a box = 64 columns x gamma rows x box_rows/gamma requests
    const uint64_t dims[3] = {(uint64_t)a.V, (uint64_t)a.gamma, (uint64_t)a.R};
    const uint64_t strides[2] = {(uint64_t)a.V * 2, (uint64_t)(a.gamma + 1) * a.V * 2};
    const uint32_t box[3] = {64, (uint32_t)a.gamma, (uint32_t)(p.box_rows / a.gamma)};
    ltma = make_tmap_bf16(&mapT, a.target, 3, dims, strides, box);
  }
  p.label_tma = ltma ? 1 : 0;
  taken = true;
  cudaError_t e = cudaMemsetAsync(p.gbar, 0, sizeof(unsigned int), s);
  if (e != cudaSuccess) return e;
  void* args[] = {&mapW2, &mapBL, &mapA, &mapT, &p};
  e = cudaLaunchCooperativeKernel((const void*)persistent_sweep_kernel<true, true>, dim3(p.n_cta), dim3(kPThreads),
                                  args, kPSmem, s);
  launches += 1;
  return e;
}

}  // namespace dspark

extern "C" dspark_status dspark_wait_selftest(int32_t which, void* workspace, size_t workspace_bytes,
                                              dspark_stream_t stream) {
  if (which < 0 || which > 2) return DSPARK_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0 || workspace_bytes < 256)
    return DSPARK_ERR_WORKSPACE;
  uint32_t* status = static_cast<uint32_t*>(workspace);
  // a counter of its own (word 16 of the status block), zeroed first: the target is never reached
  unsigned int* counter = reinterpret_cast<unsigned int*>(status + 16);
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(counter, 0, sizeof(unsigned int), s) != cudaSuccess) return DSPARK_ERR_CUDA;
  dspark::wait_selftest_kernel<<<1, 32, 0, s>>>(which, status, counter);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}
