// tcgen05 GEMM for the dense contractions around the attention: the folded output
// projection (huny.dev "DeepSeek MLA 해부" §3-2), the cache-append projection h W_DKV_KR
// (§2-1, §2-3), the per-head query absorption q_nope W_UK^T (§3-1), the query-side
// compression (§2-2) and the one-time W^UV W^O fold (§3-2).
//
// All of them have a short "rows" side (the batch's tokens) or a per-head weight, so the
// kernel computes the transposed product D^T = W^T X^T ("swap AB"): the weight dimension
// is the MMA's M = 128 (one TMEM lane per weight column), the tokens are N. Per 64-deep
// K block a CTA TMA-loads the weight tile (MN-major, 128-byte swizzle, two 64-column
// boxes) and the token tile (K-major, 128-byte swizzle) into a multi-stage ring; one
// thread issues 4 MMAs (K = 16 each) per block into a TMEM accumulator; the four warps
// then read the accumulator (tcgen05.ld).
//
// Two kernels share that K loop:
//   * tc_gemm_kernel: one CTA per output tile, the accumulator handed element by element
//     to an epilogue functor (query absorption, lift, fold);
//   * tc_gemm_cluster_kernel: long K ranges split across the CTAs of a thread-block
//     cluster (up to 16); each CTA parks its fp32 partial tile in its own shared memory,
//     and after a cluster barrier CTA r sums column slice r of the tile over every CTA of
//     the cluster (distributed shared memory, in rank order, so the sum is deterministic)
//     and hands the sums to a finishing functor (bf16 store; or RoPE, cache encoding and
//     the page scatter of an append). No zeroed accumulator, no atomics, one launch.
#include <cudaTypedefs.h>

#include "internal.h"
#include "prologue.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace gemm {

constexpr int kBM = 128, kBK = 64;
constexpr int kThreads = 128;
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct Params {
  int M, N, K;           // D^T is M x N; K is the contraction length
  int batch;             // z dimension (heads for the query absorption)
  int m_tiles, n_tiles, k_blocks, k_splits;
  int m_tiles_a;         // cluster kernel: M tiles [0, m_tiles_a) read the first A map, the rest
                         // the second (two weights of one token operand in one launch)
  int32_t* status;
  int reset_status;      // 1: block 0 clears *status first (the first kernel of a decode call)
  int pdl;               // 1: launched with programmatic serialization after the kernel it
                         // overlaps; the grid waits for that kernel at its end
  int wait_first;        // 1: launched with programmatic serialization as the first kernel of a
                         // call; every block waits for the kernel before it ahead of reading
                         // any input (only the launch and set-up overlap that kernel)
  int plan_block;        // 1: one extra block runs the decode's split planner
  PlanParams plan;
  int rope_blocks;       // extra blocks that rotate q_pe (after the planner block)
  RopeJob rope;
};

template <int BN, int NS>
struct Cfg {
  static constexpr int kABytes = kBM * kBK * 2;          // 16 KB: two 64x64 MN-major boxes
  static constexpr int kBBytes = BN * kBK * 2;            // BN rows of 128 bytes
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = NS;
  // the cluster kernel parks its fp32 partial tile [BN][128] over the idle ring
  static constexpr int kPartBytes = BN * kBM * 4;
  static constexpr int kBarOff =
      kStages * kStageBytes > kPartBytes ? kStages * kStageBytes : kPartBytes;
  // after the barriers: 4 KB in which a finishing functor may keep per-column values that
  // it looks up while the K loop runs (up to 256 columns of 16 bytes)
  static constexpr int kScratchOff = kBarOff + 256;
  static constexpr int kSmem = kScratchOff + 4096 + 1024;
  static constexpr uint32_t kTmemCols = (BN <= 32) ? 32 : (BN <= 64 ? 64 : (BN <= 128 ? 128 : 256));
  static constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, BN, true, false);
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort,
                                         int32_t* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (ptx::globaltimer() - t0 > kTimeoutNs) {
      *abort = 1;
      flag_status(status, MLA_ERR_TIMEOUT);
      return false;
    }
  }
}

// The K loop: warp 0 lane 0 streams the A (weight) and B (token) tiles of K blocks
// [kb0, kb1) through the ring; warp 1 lane 0 issues the MMAs and, after the last, commits
// `done` (at once if the range is empty). A wait that runs out sets *abort and the status.
template <int BN, int NS>
__device__ __forceinline__ void k_loop(const CUtensorMap* tmA, const CUtensorMap* tmB, uint32_t base,
                                       uint32_t tmem, int m0, int n0, int z, int kb0, int kb1,
                                       volatile int* abort, int32_t* status) {
  using C = Cfg<BN, NS>;
  auto full = [&](int s) { return base + C::kBarOff + 8 * s; };
  auto empty = [&](int s) { return base + C::kBarOff + 8 * (C::kStages + s); };
  const uint32_t done = base + C::kBarOff + 8 * (2 * C::kStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0 && lane == 0) {
    // every A operand here is a weight read once per decode step: its lines go first out of L2
    const uint64_t pol = ptx::l2_policy_evict_first();
    int stage = 0;
    uint32_t wrap = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!wait_bar(empty(stage), (wrap & 1) ^ 1, abort, status)) break;
      const uint32_t st = base + stage * C::kStageBytes;
      ptx::mbar_arrive_expect_tx(full(stage), C::kStageBytes);
      ptx::tma_load_3d_hint(st, tmA, m0, kb * kBK, z, full(stage), pol);
      ptx::tma_load_3d_hint(st + 8192, tmA, m0 + 64, kb * kBK, z, full(stage), pol);
      ptx::tma_load_3d(st + C::kABytes, tmB, kb * kBK, n0, z, full(stage));
      if (++stage == C::kStages) { stage = 0; ++wrap; }
    }
  } else if (warp == 1 && lane == 0) {
    int stage = 0;
    uint32_t wrap = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!wait_bar(full(stage), wrap & 1, abort, status)) break;
      ptx::tc_fence_after();
      const uint32_t st = base + stage * C::kStageBytes;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t a = ptx::smem_desc(st + 2048 * k, 8192, 1024, ptx::kSwizzle128);
        const uint64_t b = ptx::smem_desc(st + C::kABytes + 32 * k, 16, 1024, ptx::kSwizzle128);
        ptx::mma_bf16_ss(tmem, a, b, C::kIdesc, (kb > kb0 || k > 0) ? 1u : 0u);
      }
      ptx::mma_commit(empty(stage));
      if (++stage == C::kStages) { stage = 0; ++wrap; }
    }
    ptx::mma_commit(done);
  }
  __syncwarp();
}

// L2 prefetch of the weight (A) tiles of the first `ahead` K blocks, issued before the wait
// for the kernel before this one: the weights are not what that kernel writes in a step, and
// a prefetch only warms L2 (the loads after the wait read whatever is current), so the
// weight stream starts while that kernel ends.
__device__ __forceinline__ void prefetch_a(const CUtensorMap* tmA, int m0, int z, int kb0, int kb1,
                                           int ahead) {
  const uint64_t pol = ptx::l2_policy_evict_first();
  for (int kb = kb0; kb < kb1 && kb < kb0 + ahead; ++kb) {
    ptx::tma_prefetch_3d_hint(tmA, m0, kb * kBK, z, pol);
    ptx::tma_prefetch_3d_hint(tmA, m0 + 64, kb * kBK, z, pol);
  }
}

// D^T[z][m][n] = sum_k A[z][k][m] * B[z][n][k]; A is the MN-major weight, B the K-major
// token matrix. Work unit = (z, m tile, n tile, k split), one per CTA.
template <int BN, int NS, class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const Params gp, const Epi epi) {
  using C = Cfg<BN, NS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* basep = smem_raw + (base - raw);
  volatile int* abort = reinterpret_cast<volatile int*>(basep + C::kBarOff + 200);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(basep + C::kBarOff + 208);
  auto full = [&](int s) { return base + C::kBarOff + 8 * s; };
  auto empty = [&](int s) { return base + C::kBarOff + 8 * (C::kStages + s); };
  const uint32_t done = base + C::kBarOff + 8 * (2 * C::kStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a kernel launched after this one with programmatic serialization may start now (it
  // waits for this grid's completion before it reads what this grid writes)
  ptx::griddep_launch_dependents();
  // the decode prologue's small jobs in extra blocks: the planner (which clears the status
  // word first) as block 0, so that it starts first, and the q_pe rotation after the GEMM's
  // blocks, so that it does not displace them
  const int side_blocks = gp.plan_block;
  const int main_end = (int)gridDim.x - gp.rope_blocks;
  if ((int)blockIdx.x < side_blocks || (int)blockIdx.x >= main_end) {
    if (gp.wait_first) ptx::griddep_wait();
    if ((int)blockIdx.x < side_blocks) {
      plan_body(gp.plan, reinterpret_cast<int*>(basep), true);
    } else {
      const int r = (int)blockIdx.x - main_end;
      const RopeJob& q = gp.rope;
      if (q.d_r % 16 == 0)
        rope_body_bf16x8(q.q_pe, q.seq_lens, q.q_len, q.H, q.d_c, q.d_r, q.rt, q.qs, q.planar, q.q_lat,
                         r / q.hblocks, r % q.hblocks, 32, q.f16);
      else
        rope_body<bf16>(q.q_pe, q.seq_lens, q.q_len, q.H, q.d_c, q.d_r, q.rt, q.qs, q.planar, q.q_lat,
                        r / q.hblocks, r % q.hblocks, 32, q.f16);
    }
    ptx::griddep_wait();
    return;
  }
  if (gp.reset_status && (int)blockIdx.x == side_blocks && threadIdx.x == 0) {
    atomicExch(gp.status, 0);
    __threadfence();
  }

  int unit = (int)blockIdx.x - side_blocks;
  const int ks = unit % gp.k_splits;  unit /= gp.k_splits;
  const int nt = unit % gp.n_tiles;   unit /= gp.n_tiles;
  const int mt = unit % gp.m_tiles;   unit /= gp.m_tiles;
  const int z = unit;
  const int kb0 = (int)((long long)ks * gp.k_blocks / gp.k_splits);
  const int kb1 = (int)((long long)(ks + 1) * gp.k_blocks / gp.k_splits);
  const int m0 = mt * kBM, n0 = nt * BN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(full(s), 1);
      ptx::mbar_init(empty(s), 1);
    }
    ptx::mbar_init(done, 1);
    *abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tmA);
    ptx::prefetch_tensormap(&tmB);
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (gp.wait_first && warp == 0 && lane == 0) prefetch_a(&tmA, m0, z, kb0, kb1, C::kStages);
  if (gp.wait_first) ptx::griddep_wait();   // the inputs (the token operand) are the previous kernels'
  bool ok = true;

  k_loop<BN, NS>(&tmA, &tmB, base, tmem, m0, n0, z, kb0, kb1, abort, gp.status);
  // epilogue: every thread owns one TMEM lane = one row m of D^T
  ok = wait_bar(done, 0, abort, gp.status);
  ptx::tc_fence_after();
  if (ok && !*abort) {
    const int m = m0 + 32 * warp + lane;
    const uint32_t t_row = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t v[32];
      ptx::tmem_ld32(t_row + c, v);
      ptx::tmem_wait_ld();
      if (m < gp.M) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int n = n0 + c + j;
          if (n < gp.N) epi(z, m, n, __uint_as_float(v[j]));
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
  // under programmatic serialization: this grid completes only after the kernel before it,
  // so a kernel that waits for this one sees that kernel's results too (no-op otherwise)
  ptx::griddep_wait();
}

// D^T[m][n] = sum_k A[k][m] * B[n][k] with the K blocks split across the CTAs of a
// cluster (gp.k_splits of them, cluster rank = split). Cluster = one (m tile, n tile).
// After the K loop each CTA stores its partial tile as part[n][m] (fp32) over its idle
// ring; after a cluster barrier, CTA r sums columns [r c, (r + 1) c) of the tile over the
// cluster's CTAs in rank order (c = ceil(BN / k_splits)) and calls, for each such column,
// fin(m0, t, n, i, v, good, scratch) with every thread t of the CTA (m = m0 + t; i = the
// column's index in the slice; all threads take part, so fin may synchronise the CTA);
// good is false if a wait of this CTA ran out. fin.prepare(m0, n_begin, n_end, j, nj,
// scratch), run by warps 2-3 (thread j of nj) during the K loop, may fill the scratch for
// the slice's columns. A second cluster barrier keeps every CTA's partial alive until its
// peers have read it.
template <int BN, int NS, class Fin>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_cluster_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmA2,
                           const __grid_constant__ CUtensorMap tmB, const Params gp, const Fin fin) {
  using C = Cfg<BN, NS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* basep = smem_raw + (base - raw);
  volatile int* abort = reinterpret_cast<volatile int*>(basep + C::kBarOff + 200);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(basep + C::kBarOff + 208);
  const uint32_t done = base + C::kBarOff + 8 * (2 * C::kStages);
  const int warp = threadIdx.x >> 5, t = threadIdx.x;
  ptx::griddep_launch_dependents();

  const int KS = gp.k_splits;
  const int rank = (int)ptx::cluster_ctarank();
  const int tile = (int)blockIdx.x / KS;
  const int nt = tile % gp.n_tiles, mt = tile / gp.n_tiles;
  const int kb0 = (int)((long long)rank * gp.k_blocks / KS);
  const int kb1 = (int)((long long)(rank + 1) * gp.k_blocks / KS);
  // m0: the tile's first row of D^T in the concatenation of the two weights (each padded to
  // whole tiles), as the functor sees it; ma: the same row within its own weight
  const bool second = mt >= gp.m_tiles_a;
  const int m0 = mt * kBM, ma = (second ? mt - gp.m_tiles_a : mt) * kBM, n0 = nt * BN;
  const CUtensorMap* A = second ? &tmA2 : &tmA;

  if (t == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(base + C::kBarOff + 8 * s, 1);
      ptx::mbar_init(base + C::kBarOff + 8 * (C::kStages + s), 1);
    }
    ptx::mbar_init(done, 1);
    *abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(A);
    ptx::prefetch_tensormap(&tmB);
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // launched with programmatic serialization: the token operand may be the previous
  // kernel's output (and the weight a still earlier one's)
  if (t == 0) prefetch_a(A, ma, 0, kb0, kb1, C::kStages);
  ptx::griddep_wait();
  const int per = (BN + KS - 1) / KS;
  const int c0 = rank * per, c1 = min(BN, c0 + per);
  // warps 2 and 3 have nothing to do in the K loop: the functor's per-column look-ups of
  // this CTA's columns go there (visible to every thread after the first cluster barrier)
  void* scratch = basep + C::kScratchOff;
  if (warp >= 2) fin.prepare(m0, n0 + c0, n0 + c1, t - 64, kThreads - 64, scratch);
  k_loop<BN, NS>(A, &tmB, base, tmem, ma, n0, 0, kb0, kb1, abort, gp.status);
  const bool ok = wait_bar(done, 0, abort, gp.status);
  const bool good = __syncthreads_and(ok && !*abort) != 0;
  ptx::tc_fence_after();

  // this CTA's partial tile, part[n][m], over the ring (every MMA that read it has completed)
  float* part = reinterpret_cast<float*>(basep);
  const uint32_t t_row = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
  for (int c = 0; c < BN; c += 32) {
    uint32_t v[32];
    if (good && kb1 > kb0) {
      ptx::tmem_ld32(t_row + c, v);
      ptx::tmem_wait_ld();
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0u;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) part[(c + j) * kBM + t] = __uint_as_float(v[j]);
  }
  ptx::cluster_sync();

  const uint32_t mine = ptx::smem_u32(part) + 4u * (uint32_t)t;
  for (int c = c0; c < c1; ++c) {
    float v = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r)
      if (r < KS) v += ptx::ld_dsmem_f32(ptx::map_to_rank(mine + 4u * (uint32_t)(c * kBM), (uint32_t)r));
    fin(m0, t, n0 + c, c - c0, v, good, scratch);
  }
  ptx::cluster_sync();

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------------------ epilogues
struct EpiQLat {              // bf16(qs * v) (f16 if f16) at (group n, head z, latent dim m),
  bf16* q;                    // row-major or planar
  int H, D;
  float qs;
  int planar, f16;
  __device__ __forceinline__ void operator()(int z, int m, int n, float v) const {
    const long long i = planar ? (long long)n * H * D + ((long long)(m >> 3) * H + z) * 8 + (m & 7)
                               : ((long long)n * H + z) * D + m;
    q[i] = f16 ? __ushort_as_bfloat16(__half_as_ushort(__float2half_rn(qs * v)))
               : __float2bfloat16_rn(qs * v);
  }
};

struct EpiU {                 // bf16 u[n][z * dv + m]: head z's latent output of row n, lifted
  bf16* u;
  long long ld;
  int dv;
  __device__ __forceinline__ void operator()(int z, int m, int n, float v) const {
    u[(long long)n * ld + (long long)z * dv + m] = __float2bfloat16_rn(v);
  }
};


struct EpiStore {             // bf16 out[z][n][m] (leading dims ld_n, ld_z): the W^UV W^O fold
  bf16* out;
  long long ld_n, ld_z;
  int M;
  __device__ __forceinline__ void operator()(int z, int m, int n, float v) const {
    if (m < M) out[(long long)z * ld_z + (long long)n * ld_n + m] = __float2bfloat16_rn(v);
  }
};

// ------------------------------------------------------------------- cluster finishing
struct FinStore {             // bf16 out[n][m] = v
  bf16* out;
  long long ld;
  int M, N;
  __device__ __forceinline__ void prepare(int, int, int, int, int, void*) const {}
  __device__ __forceinline__ void operator()(int m0, int t, int n, int, float v, bool good,
                                             const void*) const {
    const int m = m0 + t;
    if (good && m < M && n < N) out[(long long)n * ld + m] = __float2bfloat16_rn(v);
  }
};

struct FinStore2 {            // rows m < Ma: out_a[n][m]; rows m >= Ma: out_b[n][m - Ma]
  bf16* out_a;
  bf16* out_b;
  int M_a, Ma, M_b, N;     // M_a: A's columns, Ma: A's M tiles x 128, M_b: A2's columns
  __device__ __forceinline__ void prepare(int, int, int, int, int, void*) const {}
  __device__ __forceinline__ void operator()(int m0, int t, int n, int, float v, bool good,
                                             const void*) const {
    const int m = m0 + t;
    if (!good || n >= N) return;
    if (m < Ma) {
      if (m < M_a) out_a[(long long)n * M_a + m] = __float2bfloat16_rn(v);
    } else if (m - Ma < M_b) {
      out_b[(long long)n * M_b + (m - Ma)] = __float2bfloat16_rn(v);
    }
  }
};

// Append from hidden states: v is column m of [c | k_raw] = h_n W_DKV_KR for token row n;
// rotates the k_pe pairs (2i, 2i + 1), encodes and writes the row's element m into its page
// slot. kMode 0: bf16 cache; 1: e4m3 with a per-tensor scale; 2: e4m3 latent with one fp32
// scale per 128 elements (amax / 448, the block being this CTA's 128 columns) and bf16 k_pe,
// row [d_c codes][d_c / 128 scales][d_r bf16].
template <int kMode>
struct FinAppend {
  const int32_t* req_ids;
  const int32_t* positions;
  const int32_t* block_table;
  int T, batch, max_pages, num_pages, P, d_c, d_r;
  void* cache;
  RopeTable rt;
  float cache_scale;
  int32_t* status;
  // page slot and position of each token row of the slice (slot -1: row skipped)
  __device__ __forceinline__ void prepare(int m0, int n_begin, int n_end, int j, int nj,
                                          void* scratch) const {
    long long* sp = reinterpret_cast<long long*>(scratch);
    for (int i = j; i < n_end - n_begin; i += nj) {
      const int n = n_begin + i;
      int pos = 0;
      long long slot = -1;
      if (n < T)     // the CTAs of the first column tile report a bad row
        slot = append_slot(req_ids, positions, block_table, batch, max_pages, num_pages, P, n,
                           m0 == 0 ? status : nullptr, &pos);
      sp[2 * i] = slot;
      sp[2 * i + 1] = pos;
    }
  }
  __device__ __forceinline__ void operator()(int m0, int t, int n, int i, float v, bool good,
                                             const void* scratch) const {
    __shared__ float red[kThreads / 32];
    const int m = m0 + t, D = d_c + d_r;
    const long long slot = reinterpret_cast<const long long*>(scratch)[2 * i];
    const int pos = (int)reinterpret_cast<const long long*>(scratch)[2 * i + 1];
    // the partner of a rotation pair sits in the neighbouring lane
    const float other = __shfl_xor_sync(0xffffffffu, v, 1);
    float y = v;
    if (m >= d_c && m < D) {
      const int kc = m - d_c;
      float sn, cs;
      rope_sincos(rt, kc >> 1, pos, &sn, &cs);
      y = (kc & 1) ? other * sn + v * cs : v * cs - other * sn;
    }
    const bool live = good && slot >= 0 && m < D;
    if (kMode == 0) {
      if (live) reinterpret_cast<bf16*>(cache)[slot * D + m] = __float2bfloat16_rn(y);
    } else if (kMode == 1) {
      if (live) reinterpret_cast<uint8_t*>(cache)[slot * D + m] = CacheCodec<uint8_t>::encode(y, cache_scale);
    } else {
      uint8_t* dst = reinterpret_cast<uint8_t*>(cache) + slot * (long long)(d_c + d_c / 32 + 2 * d_r);
      if (m0 < d_c) {           // a whole latent block: CTA-wide amax (uniform branch)
        const float w = warp_max(fabsf(y));
        __syncthreads();
        if ((t & 31) == 0) red[t >> 5] = w;
        __syncthreads();
        float amax = red[0];
#pragma unroll
        for (int i = 1; i < kThreads / 32; ++i) amax = fmaxf(amax, red[i]);
        const float scale = amax / 448.f;
        if (live) {
          dst[m] = scale > 0.f ? f32_to_fp8(y / scale) : (uint8_t)0;
          if (t == 0) reinterpret_cast<float*>(dst + d_c)[m0 >> 7] = scale;
        }
      } else if (live) {
        reinterpret_cast<bf16*>(dst + d_c + d_c / 32)[m - d_c] = __float2bfloat16_rn(y);
      }
    }
  }
};

// ------------------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 3-D bf16 map: dims {d0 (contiguous), d1, d2}, byte strides of d1 and d2, box {b0, b1, 1}.
static bool map3d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

template <int BN, int NS, class Epi>
static cudaError_t run(const CUtensorMap& A, const CUtensorMap& B, Params gp, const Epi& epi,
                       cudaStream_t s) {
  using C = Cfg<BN, NS>;
  auto kern = tc_gemm_kernel<BN, NS, Epi>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const long long units = (long long)gp.batch * gp.m_tiles * gp.n_tiles * gp.k_splits;
  if (units <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  if (gp.plan_block && plan_smem_bytes(gp.plan.batch * gp.plan.q_len, gp.plan.workers) > (size_t)C::kBarOff)
    return cudaErrorInvalidValue;
  cfg.gridDim = dim3((unsigned)(units + gp.plan_block + gp.rope_blocks), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = gp.pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, A, B, gp, epi);
  note_launch();
  return e;
}

// Chooses the N tile for the one-CTA-per-tile kernel (no K split).
template <class Epi>
static cudaError_t dispatch(const CUtensorMap& A, const CUtensorMap& Bmap32, const CUtensorMap& Bmap64,
                            const CUtensorMap& Bmap128, const CUtensorMap& Bmap256, Params gp,
                            const Epi& epi, cudaStream_t s) {
  int bn = gp.N <= 32 ? 32 : (gp.N <= 64 ? 64 : (gp.N <= 128 ? 128 : 256));
  gp.n_tiles = (gp.N + bn - 1) / bn;
  gp.k_blocks = (gp.K + kBK - 1) / kBK;
  gp.k_splits = 1;
  const bool shallow = gp.k_blocks <= 2;   // a ring of 2 is enough
  switch (bn) {
    case 32: return shallow ? run<32, 2>(A, Bmap32, gp, epi, s) : run<32, 4>(A, Bmap32, gp, epi, s);
    case 64: return shallow ? run<64, 2>(A, Bmap64, gp, epi, s) : run<64, 4>(A, Bmap64, gp, epi, s);
    case 128: return shallow ? run<128, 2>(A, Bmap128, gp, epi, s) : run<128, 5>(A, Bmap128, gp, epi, s);
    default: return shallow ? run<256, 2>(A, Bmap256, gp, epi, s) : run<256, 4>(A, Bmap256, gp, epi, s);
  }
}

// Whether clusters of 16 CTAs of this kernel fit on the device (`need` of them at once);
// clusters above 8 CTAs are a non-portable size that the kernel must opt in to.
template <int BN, int NS, class Fin>
static bool cluster16_fits(int need) {
  // per instantiation and device: number of co-resident clusters of 16 (-1: not asked yet)
  static int fits[64] = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1,
                         -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1,
                         -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1,
                         -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (fits[dev] < 0) {
    using C = Cfg<BN, NS>;
    auto kern = tc_gemm_cluster_kernel<BN, NS, Fin>;
    int n = 0;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16, 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = C::kSmem;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = 16;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    }
    if (e != cudaSuccess) {
      n = 0;
      cudaGetLastError();      // the refusal of our own query: leave no error behind
    }
    fits[dev] = n;
  }
  return fits[dev] >= need;
}

template <int BN, int NS, class Fin>
static cudaError_t run_cluster(const CUtensorMap& A, const CUtensorMap& A2, const CUtensorMap& B,
                               Params gp, const Fin& fin, cudaStream_t s) {
  using C = Cfg<BN, NS>;
  auto kern = tc_gemm_cluster_kernel<BN, NS, Fin>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e == cudaSuccess && gp.k_splits > 8)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  const long long ctas = (long long)gp.m_tiles * gp.n_tiles * gp.k_splits;
  if (ctas <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = (unsigned)gp.k_splits;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, A, A2, B, gp, fin);
  note_launch();
  return e;
}

// Tile and split choice of the cluster GEMM. Grids that fit once on the SMs with one CTA
// per SM take a deep ring (8 stages) and the widest cluster that fits (16 where the device
// allows, else 8, at least 2 K blocks per CTA); larger grids take a 4-stage ring (two CTAs
// fit on an SM for N tiles up to 64) and about 1.6 CTAs per SM (at most 8 splits, at least
// 4 K blocks per CTA). Measured at the 40-tile output projection of DeepSeek-V2 shapes
// (W_comb, 671 MB): splits of 3, 4, 5, 6 and 7 take 117.6, 104, 100, 96.6 and 134 us;
// clusters of 7 at two CTAs per SM do not all fit on the SMs at once.
template <int BN, class Fin>
static cudaError_t cluster_bn(const CUtensorMap& A, const CUtensorMap& A2, const CUtensorMap& B,
                              Params gp, const Fin& fin, cudaStream_t s) {
  const int sms = sm_count();
  const int tiles = gp.m_tiles * gp.n_tiles;
  const int kmax2 = gp.k_blocks / 2 > 0 ? gp.k_blocks / 2 : 1;
  if constexpr (BN <= 64) {
    if (tiles * 8 <= sms) {
      int ks = sms / tiles;
      if (ks > 16) ks = 16;
      if (ks > 8 && !cluster16_fits<BN, 8, Fin>(tiles)) ks = 8;
      if (ks > kmax2) ks = kmax2;
      gp.k_splits = ks < 1 ? 1 : ks;
      return run_cluster<BN, 8>(A, A2, B, gp, fin, s);
    }
  }
  int ks = (16 * sms + 5 * tiles) / (10 * tiles);     // round(1.6 sms / tiles)
  const int kmax4 = gp.k_blocks / 4 > 0 ? gp.k_blocks / 4 : 1;
  if (ks * tiles > 2 * sms) ks = 2 * sms / tiles;     // every CTA resident at once
  if (ks > 8) ks = 8;
  if (ks > kmax4) ks = kmax4;
  gp.k_splits = ks < 1 ? 1 : ks;
  return run_cluster<BN, 4>(A, A2, B, gp, fin, s);
}

// gp.m_tiles = the M tiles of A, plus those of A2 if A2 is given (m_tiles_a = A's).
template <class Fin>
static cudaError_t dispatch_cluster(const CUtensorMap (&Bm)[4], const CUtensorMap& A,
                                    const CUtensorMap* A2, Params gp, const Fin& fin, cudaStream_t s) {
  const int bn = gp.N <= 32 ? 32 : (gp.N <= 64 ? 64 : (gp.N <= 128 ? 128 : 256));
  gp.n_tiles = (gp.N + bn - 1) / bn;
  gp.k_blocks = (gp.K + kBK - 1) / kBK;
  gp.batch = 1;
  if (!A2) gp.m_tiles_a = gp.m_tiles;
  const CUtensorMap& a2 = A2 ? *A2 : A;
  switch (bn) {
    case 32: return cluster_bn<32>(A, a2, Bm[0], gp, fin, s);
    case 64: return cluster_bn<64>(A, a2, Bm[1], gp, fin, s);
    case 128: return cluster_bn<128>(A, a2, Bm[2], gp, fin, s);
    default: return cluster_bn<256>(A, a2, Bm[3], gp, fin, s);
  }
}

// B maps for every N tile size (the box height is part of the map).
static bool b_maps(CUtensorMap (&maps)[4], const void* ptr, uint64_t K, uint64_t N, uint64_t Z,
                   uint64_t sN, uint64_t sZ) {
  const uint32_t bns[4] = {32, 64, 128, 256};
  for (int i = 0; i < 4; ++i)
    if (!map3d(&maps[i], ptr, K, N, Z, sN, sZ, 64, bns[i])) return false;
  return true;
}

}  // namespace gemm

// out[rows][N] = x[rows][K] . W[K][N] (bf16 in and out, fp32 accumulation): the folded
// output projection, the unfolded path's W_O product and the query-side GEMMs.
cudaError_t launch_output_proj_tc(const void* x, const void* W, int rows, int K, int N, void* out,
                                  int32_t* status, cudaStream_t s) {
  using namespace gemm;
  if (rows <= 0) return cudaSuccess;
  CUtensorMap A, Bm[4];
  // A = W as D^T's M x K: dims {N (m, contiguous), K}
  if (!map3d(&A, W, (uint64_t)N, (uint64_t)K, 1, (uint64_t)N * 2, (uint64_t)N * K * 2, 64, 64) ||
      !b_maps(Bm, x, (uint64_t)K, (uint64_t)rows, 1, (uint64_t)K * 2, (uint64_t)K * rows * 2))
    return cudaErrorInvalidValue;
  Params gp{};
  gp.M = N;
  gp.N = rows;
  gp.K = K;
  gp.m_tiles = (N + kBM - 1) / kBM;
  gp.status = status;
  return dispatch_cluster(Bm, A, nullptr, gp, FinStore{reinterpret_cast<bf16*>(out), (long long)N, N, rows}, s);
}

// out_a[rows][N_a] = x . W_a and out_b[rows][N_b] = x . W_b in one launch (x [rows][K],
// W_a [K][N_a], W_b [K][N_b]; bf16 in and out, fp32 sums): two weights applied to the same
// tokens, e.g. the query-side W_DQ and W_QR applied to h.
cudaError_t launch_two_proj_tc(const void* x, const void* W_a, const void* W_b, int rows, int K,
                               int N_a, int N_b, void* out_a, void* out_b, int32_t* status,
                               cudaStream_t s) {
  using namespace gemm;
  if (rows <= 0) return cudaSuccess;
  CUtensorMap A, A2, Bm[4];
  if (!map3d(&A, W_a, (uint64_t)N_a, (uint64_t)K, 1, (uint64_t)N_a * 2, (uint64_t)N_a * K * 2, 64, 64) ||
      !map3d(&A2, W_b, (uint64_t)N_b, (uint64_t)K, 1, (uint64_t)N_b * 2, (uint64_t)N_b * K * 2, 64, 64) ||
      !b_maps(Bm, x, (uint64_t)K, (uint64_t)rows, 1, (uint64_t)K * 2, (uint64_t)K * rows * 2))
    return cudaErrorInvalidValue;
  Params gp{};
  gp.M = N_a + N_b;
  gp.N = rows;
  gp.K = K;
  gp.m_tiles_a = (N_a + kBM - 1) / kBM;
  gp.m_tiles = gp.m_tiles_a + (N_b + kBM - 1) / kBM;
  gp.status = status;
  return dispatch_cluster(Bm, A, &A2, gp,
                          FinStore2{reinterpret_cast<bf16*>(out_a), reinterpret_cast<bf16*>(out_b), N_a,
                                    gp.m_tiles_a * kBM, N_b, rows}, s);
}

// u[r][h][0:d_v] = o_lat[r][h][:] . W_UV[:, h d_v : (h + 1) d_v]  (per head, bf16 out).
cudaError_t launch_lift_tc(const void* o_lat, const void* W_UV, int rows, int H, int d_c, int d_v,
                           void* u, int32_t* status, cudaStream_t s) {
  using namespace gemm;
  if (rows <= 0) return cudaSuccess;
  CUtensorMap A, Bm[4];
  // A = W_UV as head z's M x K: dims {d_v (m), d_c (k), H (z)}; a row of W_UV holds every head
  if (!map3d(&A, W_UV, (uint64_t)d_v, (uint64_t)d_c, (uint64_t)H, (uint64_t)H * d_v * 2,
             (uint64_t)d_v * 2, 64, 64) ||
      // B = o_lat : dims {d_c (k), rows (n), H (z)}
      !b_maps(Bm, o_lat, (uint64_t)d_c, (uint64_t)rows, (uint64_t)H, (uint64_t)H * d_c * 2,
              (uint64_t)d_c * 2))
    return cudaErrorInvalidValue;
  Params gp{};
  gp.M = d_v;
  gp.N = rows;
  gp.K = d_c;
  gp.batch = H;
  gp.m_tiles = (d_v + kBM - 1) / kBM;
  gp.status = status;
  // launched with programmatic serialization; every block waits for the kernel before it
  // (typically the decode's combine, which writes o_lat) ahead of reading any input
  gp.pdl = 1;
  gp.wait_first = 1;
  return dispatch(A, Bm[0], Bm[1], Bm[2], Bm[3], gp,
                  EpiU{reinterpret_cast<bf16*>(u), (long long)H * d_v, d_v}, s);
}

// W_comb[h][r][0:d] = W_UV[r][h d_v : (h + 1) d_v] . W_O[h d_v : (h + 1) d_v][0:d] for every
// head h (bf16 in and out, fp32 accumulation): the one-time fold, per head a 512 x d_v by
// d_v x d product. D^T's M is W_O's output column, N the latent row r, K the value dim.
cudaError_t launch_fold_tc(const void* W_UV, const void* W_O, int H, int d_c, int d_v, int d,
                           void* W_comb, int32_t* status, cudaStream_t s) {
  using namespace gemm;
  CUtensorMap A, Bm[4];
  // A = W_O as head z's M x K: dims {d (m), d_v (k), H (z)}
  if (!map3d(&A, W_O, (uint64_t)d, (uint64_t)d_v, (uint64_t)H, (uint64_t)d * 2,
             (uint64_t)d_v * d * 2, 64, 64) ||
      // B = W_UV as head z's N x K: dims {d_v (k), d_c (n), H (z)}
      !b_maps(Bm, W_UV, (uint64_t)d_v, (uint64_t)d_c, (uint64_t)H, (uint64_t)H * d_v * 2,
              (uint64_t)d_v * 2))
    return cudaErrorInvalidValue;
  Params gp{};
  gp.M = d;
  gp.N = d_c;
  gp.K = d_v;
  gp.batch = H;
  gp.m_tiles = (d + kBM - 1) / kBM;
  gp.status = status;
  return dispatch(A, Bm[0], Bm[1], Bm[2], Bm[3], gp,
                  EpiStore{reinterpret_cast<bf16*>(W_comb), (long long)d, (long long)d_c * d, d}, s);
}

// q_lat[g][h][0:d_c] = q_nope[g][h][:] . W_UK_abs[h]  (per head, bf16 out).
cudaError_t launch_query_absorb_tc(const void* q_nope, const void* W_UK_abs, int groups, int H,
                                   int d_n, int d_c, int D, float q_scale, int planar, int f16,
                                   void* q_lat, int32_t* status, const PlanParams* plan,
                                   const RopeJob* rope, cudaStream_t s) {
  using namespace gemm;
  CUtensorMap A, Bm[4];
  // A = W_UK_abs[h] : dims {d_c (m), d_n (k), H (z)}
  if (!map3d(&A, W_UK_abs, (uint64_t)d_c, (uint64_t)d_n, (uint64_t)H, (uint64_t)d_c * 2,
             (uint64_t)d_n * d_c * 2, 64, 64) ||
      // B = q_nope : dims {d_n (k), groups (n), H (z)}, strides: group H*d_n, head d_n
      !b_maps(Bm, q_nope, (uint64_t)d_n, (uint64_t)groups, (uint64_t)H, (uint64_t)H * d_n * 2,
              (uint64_t)d_n * 2))
    return cudaErrorInvalidValue;
  Params gp{};
  gp.M = d_c;
  gp.N = groups;
  gp.K = d_n;
  gp.batch = H;
  gp.m_tiles = (d_c + kBM - 1) / kBM;
  gp.status = status;
  // with the planner as an extra block this is the decode's first kernel and the planner
  // clears the status word; otherwise the prep kernel before it did
  gp.reset_status = 0;
  // with the planner it is also launched with programmatic serialization, waiting for the
  // kernel before it (whatever the caller ran) ahead of every read of an input
  gp.pdl = 1;
  gp.wait_first = plan ? 1 : 0;
  gp.plan_block = plan ? 1 : 0;
  if (plan) gp.plan = *plan;
  gp.rope_blocks = rope ? rope->groups * rope->hblocks : 0;
  if (rope) gp.rope = *rope;
  return dispatch(A, Bm[0], Bm[1], Bm[2], Bm[3], gp,
                  EpiQLat{reinterpret_cast<bf16*>(q_lat), H, D, q_scale, planar, f16}, s);
}

// The append from hidden states in one launch: [c | k_raw] = h W_DKV_KR (h [T][d],
// W [d][d_c + d_r]), then per token row RoPE of k_raw at its position, the cache encoding
// and the scatter into its page slot (the cluster GEMM's finishing step).
cudaError_t launch_append_tc(mla_dtype cache_dtype, const void* h, const void* W, int T, int d,
                             int d_c, int d_r, const int32_t* req_ids, const int32_t* positions,
                             const int32_t* block_table, int batch, int max_pages, void* cache,
                             int num_pages, int P, const RopeTable& rt, float cache_scale,
                             int32_t* status, cudaStream_t s) {
  using namespace gemm;
  if (T <= 0) return cudaSuccess;
  const int Dc = d_c + d_r;
  CUtensorMap A, Bm[4];
  if (!map3d(&A, W, (uint64_t)Dc, (uint64_t)d, 1, (uint64_t)Dc * 2, (uint64_t)Dc * d * 2, 64, 64) ||
      !b_maps(Bm, h, (uint64_t)d, (uint64_t)T, 1, (uint64_t)d * 2, (uint64_t)d * T * 2))
    return cudaErrorInvalidValue;
  Params gp{};
  gp.M = Dc;
  gp.N = T;
  gp.K = d;
  gp.m_tiles = (Dc + kBM - 1) / kBM;
  gp.status = status;
  auto fill = [&](auto f) {
    f.req_ids = req_ids;
    f.positions = positions;
    f.block_table = block_table;
    f.T = T;
    f.batch = batch;
    f.max_pages = max_pages;
    f.num_pages = num_pages;
    f.P = P;
    f.d_c = d_c;
    f.d_r = d_r;
    f.cache = cache;
    f.rt = rt;
    f.cache_scale = cache_scale;
    f.status = status;
    return f;
  };
  if (cache_dtype == MLA_BF16) return dispatch_cluster(Bm, A, nullptr, gp, fill(FinAppend<0>{}), s);
  if (cache_dtype == MLA_FP8_E4M3)
    return dispatch_cluster(Bm, A, nullptr, gp, fill(FinAppend<1>{}), s);
  return dispatch_cluster(Bm, A, nullptr, gp, fill(FinAppend<2>{}), s);
}

}  // namespace mla
