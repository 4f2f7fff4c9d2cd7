// tcgen05 GEMM for the dense contractions around the attention: the folded output
// projection (huny.dev "DeepSeek MLA 해부" §3-2), the cache-append projection h W_DKV_KR
// (§2-1, §2-3) and the per-head query absorption q_nope W_UK^T (§3-1).
//
// All three have a short "rows" side (the batch's tokens) and a long weight side, so the
// kernel computes the transposed product D^T = W^T X^T ("swap AB"): the weight dimension
// is the MMA's M = 128 (one TMEM lane per weight column), the tokens are N. Per 64-deep
// K block a CTA TMA-loads the weight tile (MN-major, 128-byte swizzle, two 64-column
// boxes) and the token tile (K-major, 128-byte swizzle) into a multi-stage ring; one
// thread issues 4 MMAs (K = 16 each) per block into a TMEM accumulator; the four warps
// then read the accumulator (tcgen05.ld) and hand each fp32 value to an epilogue functor.
// Long K ranges are split across CTAs; split partial sums are added with fp32 atomics
// into a workspace accumulator and finished by a small conversion kernel.
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
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kSmem = kBarOff + 256 + 1024;
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
                         r / q.hblocks, r % q.hblocks, 32);
      else
        rope_body<bf16>(q.q_pe, q.seq_lens, q.q_len, q.H, q.d_c, q.d_r, q.rt, q.qs, q.planar, q.q_lat,
                        r / q.hblocks, r % q.hblocks, 32);
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
  if (gp.wait_first) ptx::griddep_wait();   // the inputs (the token operand) are the previous kernels'
  bool ok = true;

  if (warp == 0 && lane == 0) {
    // every A operand here is a weight read once per decode step: its lines go first out of L2
    const uint64_t pol = ptx::l2_policy_evict_first();
    int stage = 0;
    uint32_t wrap = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!wait_bar(empty(stage), (wrap & 1) ^ 1, abort, gp.status)) break;
      const uint32_t st = base + stage * C::kStageBytes;
      ptx::mbar_arrive_expect_tx(full(stage), C::kStageBytes);
      ptx::tma_load_3d_hint(st, &tmA, m0, kb * kBK, z, full(stage), pol);
      ptx::tma_load_3d_hint(st + 8192, &tmA, m0 + 64, kb * kBK, z, full(stage), pol);
      ptx::tma_load_3d(st + C::kABytes, &tmB, kb * kBK, n0, z, full(stage));
      if (++stage == C::kStages) { stage = 0; ++wrap; }
    }
  } else if (warp == 1 && lane == 0) {
    int stage = 0;
    uint32_t wrap = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!wait_bar(full(stage), wrap & 1, abort, gp.status)) break;
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

// ------------------------------------------------------------------------------ epilogues
struct EpiAtomic {            // acc[n][m] += v  (split-K partial sums, fp32 workspace)
  float* acc;
  long long ld;
  __device__ __forceinline__ void operator()(int, int m, int n, float v) const {
    atomicAdd(acc + (long long)n * ld + m, v);
  }
};
struct EpiQLat {              // bf16(qs * v) at (group n, head z, latent dim m), row-major or planar
  bf16* q;
  int H, D;
  float qs;
  int planar;
  __device__ __forceinline__ void operator()(int z, int m, int n, float v) const {
    const long long i = planar ? (long long)n * H * D + ((long long)(m >> 3) * H + z) * 8 + (m & 7)
                               : ((long long)n * H + z) * D + m;
    q[i] = __float2bfloat16_rn(qs * v);
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

// Chooses the N tile and the K split: enough CTAs to cover the SMs about once.
template <class Epi>
static cudaError_t dispatch(const CUtensorMap& A, const CUtensorMap& Bmap32, const CUtensorMap& Bmap64,
                            const CUtensorMap& Bmap128, const CUtensorMap& Bmap256, Params gp,
                            const Epi& epi, bool allow_split, cudaStream_t s) {
  int bn = gp.N <= 32 ? 32 : (gp.N <= 64 ? 64 : (gp.N <= 128 ? 128 : 256));
  gp.n_tiles = (gp.N + bn - 1) / bn;
  gp.k_blocks = (gp.K + kBK - 1) / kBK;
  gp.k_splits = 1;
  if (allow_split) {
    // about two CTAs per SM, each with at least 4 K blocks
    const long long base_units = (long long)gp.batch * gp.m_tiles * gp.n_tiles;
    const int per_sm = bn <= 64 ? 2 : 1;
    int want = (int)(((long long)per_sm * sm_count()) / (base_units > 0 ? base_units : 1));
    const int max_splits = gp.k_blocks / 4 > 0 ? gp.k_blocks / 4 : 1;
    if (want > max_splits) want = max_splits;
    gp.k_splits = want < 1 ? 1 : want;
  }
  const bool shallow = (gp.k_blocks + gp.k_splits - 1) / gp.k_splits <= 2;   // ring of 2 is enough
  switch (bn) {
    case 32: return shallow ? run<32, 2>(A, Bmap32, gp, epi, s) : run<32, 4>(A, Bmap32, gp, epi, s);
    case 64: return shallow ? run<64, 2>(A, Bmap64, gp, epi, s) : run<64, 4>(A, Bmap64, gp, epi, s);
    case 128: return shallow ? run<128, 2>(A, Bmap128, gp, epi, s) : run<128, 5>(A, Bmap128, gp, epi, s);
    default: return shallow ? run<256, 2>(A, Bmap256, gp, epi, s) : run<256, 4>(A, Bmap256, gp, epi, s);
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

__global__ void finish_oproj_kernel(float* __restrict__ acc, bf16* __restrict__ out, long long n) {
  // launched with programmatic serialization after the split-K GEMM that fills `acc`
  ptx::griddep_wait();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    out[i] = __float2bfloat16_rn(acc[i]);
  }
}

}  // namespace gemm

// out[rows][N] = o_lat[rows][K] . W_comb[K][N] (bf16), fp32 accumulator `acc` [rows][N].
cudaError_t launch_output_proj_tc(const void* o_lat, const void* W_comb, int rows, int K, int N,
                                  void* out, float* acc, int32_t* status, cudaStream_t s) {
  using namespace gemm;
  if (rows <= 0) return cudaSuccess;
  CUtensorMap A, Bm[4];
  // A = W_comb as D^T's M x K: dims {N (m, contiguous), K}
  if (!map3d(&A, W_comb, (uint64_t)N, (uint64_t)K, 1, (uint64_t)N * 2, (uint64_t)N * K * 2, 64, 64) ||
      !b_maps(Bm, o_lat, (uint64_t)K, (uint64_t)rows, 1, (uint64_t)K * 2, (uint64_t)K * rows * 2))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(acc, 0, (size_t)rows * N * sizeof(float), s);
  if (e != cudaSuccess) return e;
  Params gp{};
  gp.M = N;
  gp.N = rows;
  gp.K = K;
  gp.batch = 1;
  gp.m_tiles = (N + kBM - 1) / kBM;
  gp.status = status;
  e = dispatch(A, Bm[0], Bm[1], Bm[2], Bm[3], gp, EpiAtomic{acc, (long long)N}, true, s);
  if (e != cudaSuccess) return e;
  const long long n = (long long)rows * N;
  // programmatic serialization: the conversion's blocks start while the GEMM (which signals
  // launch_dependents at its start) ends, and wait for it before reading `acc`
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((n + 255) / 256 < 2048 ? (n + 255) / 256 : 2048), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, finish_oproj_kernel, acc, reinterpret_cast<bf16*>(out), n);
  note_launch();
  return e;
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
  return dispatch(A, Bm[0], Bm[1], Bm[2], Bm[3], gp,
                  EpiU{reinterpret_cast<bf16*>(u), (long long)H * d_v, d_v}, false, s);
}

// q_lat[g][h][0:d_c] = q_nope[g][h][:] . W_UK_abs[h]  (per head, bf16 out).
cudaError_t launch_query_absorb_tc(const void* q_nope, const void* W_UK_abs, int groups, int H,
                                   int d_n, int d_c, int D, float q_scale, int planar, void* q_lat,
                                   int32_t* status, const PlanParams* plan, const RopeJob* rope,
                                   cudaStream_t s) {
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
                  EpiQLat{reinterpret_cast<bf16*>(q_lat), H, D, q_scale, planar}, false, s);
}

// acc[T][Dc] += h[T][d] . W[d][Dc]  (split-K partial sums into a zeroed fp32 buffer).
cudaError_t launch_append_proj_tc(const void* h, const void* W, int T, int d, int Dc, float* acc,
                                  int32_t* status, cudaStream_t s) {
  using namespace gemm;
  CUtensorMap A, Bm[4];
  if (!map3d(&A, W, (uint64_t)Dc, (uint64_t)d, 1, (uint64_t)Dc * 2, (uint64_t)Dc * d * 2, 64, 64) ||
      !b_maps(Bm, h, (uint64_t)d, (uint64_t)T, 1, (uint64_t)d * 2, (uint64_t)d * T * 2))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(acc, 0, (size_t)T * Dc * sizeof(float), s);
  if (e != cudaSuccess) return e;
  Params gp{};
  gp.M = Dc;
  gp.N = T;
  gp.K = d;
  gp.batch = 1;
  gp.m_tiles = (Dc + kBM - 1) / kBM;
  gp.status = status;
  return dispatch(A, Bm[0], Bm[1], Bm[2], Bm[3], gp, EpiAtomic{acc, (long long)Dc}, true, s);
}

}  // namespace mla
