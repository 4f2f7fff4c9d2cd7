// Tensor-core MLA decode for sm_103a: tcgen05 MMAs with TMEM accumulators, TMA-staged
// cache pages, a CTA pair per worker.
//
// Math (huny.dev "DeepSeek MLA 해부" §3-1/§3-2; secrett2633.cloud "MLA의 MQA 디코딩 경로"):
// every head of one query token attends, MQA-style, over the request's shared 576-wide
// latent rows [c_kv | k_pe]; score = q_lat . row * scale; output = softmax . c_kv.
//
// Work split. 128 heads x 512 latent dims of fp32 output fill all 512 TMEM columns of
// one SM, leaving no room for the scores, so each worker is a 2-CTA cluster that splits
// the latent dimensions: CTA r owns c_kv dims [256r, 256r+256) and k_pe dims
// [512+32r, 512+32r+32). Per 64-token page each CTA
//   1. TMA-loads only its 288-column slice of the page (36 KB; the pair reads each byte of
//      the page once) into a 4-stage ring,
//   2. computes its partial score S_r = Q_r K_r^T (M = 128 heads, N = 64 tokens, K = 288)
//      into TMEM (A = the latent part of Q_r held in TMEM, and the k_pe part from shared
//      memory),
//   3. send warps read S_r, round it to fp16 (columns past the last token as 0, values
//      beyond the fp16 range saturated), stage it in shared memory and, once the four warps
//      have staged their rows, move it with one 16 KB bulk copy into one of the peer's two
//      receive buffers (counted on the peer's mbarrier),
//   4. softmax warps combine the peer's fp16 partial with their own staged fp16 partial
//      (identical combined scores f16(S_0) + f16(S_1) in both CTAs; the fp16 rounding,
//      relative 2^-11, is below the bf16 rounding of P), run the online softmax (one thread
//      per head row, exp2, O rescaled lazily, only when the running maximum grows by more
//      than 2^8) and write P (bf16; f16 with the per-tensor fp8 cache, whose MMAs all
//      take f16 operands) into one of two TMEM buffers,
//   5. O_r += P C_r (M = 128, N = 256, K = 64; A = P from TMEM, B = the staged page).
// The query arrives pre-multiplied by softmax_scale * log2(e), so scores are already in
// log2 units: the softmax forms each exponent as (f32) own half + (f32) peer half - m with
// two mixed fp16/fp32 adds, and takes the running maximum on packed fp16 sums.
// The send warps run ahead of the softmax warps, so the cluster transfer, the score MMAs
// and the softmax of consecutive pages overlap.
// Roles: warp 0 issues TMA; warp 1 issues the score MMAs and owns the TMEM allocation;
// warps 2-5 send partial scores and load Q_r into TMEM at each work item's start (a thread
// owns one head row = one TMEM lane); warps 6-13 combine the partials, run the softmax and
// write the outputs, two threads per head row: warps 6-9 columns 0-31 and warps 10-13
// columns 32-63 of each page (and the matching halves of O), sharing the row maximum
// through shared memory with a 64-thread named barrier per lane quarter; warp 14 issues the
// P.C MMAs.
// TMEM: O_r 256 columns, raw S 64, P 2 x 32, Q_r latent part 128.
// Split partials are written bf16 [item][d_c / 8][128 heads][8], so the 32 threads of a
// warp (32 consecutive heads) store one contiguous 512-byte run per instruction.
// Every mbarrier wait is bounded (2 s unless the caller sets a limit): on timeout the kernel records MLA_ERR_TIMEOUT,
// every role leaves its loop, TMEM is freed and the pair meets at a final cluster
// barrier before exit.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "decode_tc.h"
#include "sm100_ptx.cuh"

namespace mla {
namespace tc {

constexpr int kH = 128, kDC = 512, kDR = 64, kD = 576, kP = 64;
constexpr int kNS = 4;                                   // cache-page pipeline stages
constexpr int kXB = 2;                                   // score-exchange buffers (page n uses n % kXB)
constexpr int kL2Ahead = 1;                              // L2 prefetch distance, in pages
constexpr int kQAhead = 4;                               // next item's query into L2, pages before the end
constexpr int kKTileC = 64 * 64 * 2;                     // one 64-dim SW128 chunk of a page
constexpr int kKTilePE = 64 * 32 * 2;                    // the 32-dim SW64 k_pe half
constexpr int kStageBytes = 4 * kKTileC + kKTilePE;      // 36864
constexpr int kXBytes = 128 * 64 * 2;                    // one fp16 partial-score buffer
// Block-scaled fp8 cache rows: [512 e4m3 codes][4 fp32 scales][64 bf16 k_pe] = 656 bytes.
// A stage receives this CTA's 256 codes (16 KB, unswizzled, over the back half of the
// latent tiles), the row's 4 scales (1 KB, just below them) and its 32 k_pe values straight
// into the SW64 rope tile.
constexpr int kB128RowBytes = kDC + kDC / 32 + 2 * kDR;    // 656
constexpr int kB128Codes = 16384;                          // stage offset of the codes
constexpr int kB128Scales = kB128Codes - 64 * 16;          // stage offset of the scales
constexpr int kQPeBytes = 128 * 32 * 2;                  // Q_r k_pe part, SW64 [128][32]
constexpr int kOffStage = 0;
constexpr int kOffX = kOffStage + kNS * kStageBytes;     // receive buffers (the peer's partial)
constexpr int kOffStg = kOffX + kXB * kXBytes;           // staging buffers (own partial)
constexpr int kOffQPe = kOffStg + kXB * kXBytes;
constexpr int kOffRed = kOffQPe + kQPeBytes;             // row max [2 pages][2 halves][128 rows] fp32
constexpr int kOffLsum = kOffRed + 2 * 2 * 128 * 4;      // row sum [2 halves][128 rows] fp32
constexpr int kOffBar = kOffLsum + 2 * 128 * 4;
constexpr int kBarArea = 512;                            // mbarriers, then the abort flag and TMEM slot
constexpr int kSmemBytes = kOffBar + kBarArea + 1024;    // + slack to align the base to 1 KB
static_assert(kSmemBytes <= 232448, "dynamic shared memory per CTA");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;                            // O_r: 256 fp32 columns
constexpr uint32_t kColS = 256;                          // raw partial S: 64 fp32 columns
constexpr uint32_t kColP = 320;                          // P: two buffers of 64 bf16 = 32
constexpr uint32_t kColQ = 384;                          // Q_r latent part: 256 bf16 = 128
constexpr int kThreads = 480;                            // 15 warps (bf16 cache)
constexpr int kWarpConv0 = 15;                           // fp8 cache: 4 converter warps after them
constexpr int kThreadsFp8 = kThreads + 4 * 32;
constexpr int kSoftmaxWarps = 8;                         // two per head row (column halves)
// kF16: the operands of every MMA in f16 instead of bf16 (the per-tensor e4m3 cache, whose
// codes convert to f16 exactly in one instruction per pair); query, cache and P then all
// share that type.
template <bool kF16>
constexpr uint32_t idesc_qk() {
  return kF16 ? ptx::idesc_f16_f32(128, 64, false, false) : ptx::idesc_bf16_f32(128, 64, false, false);
}
template <bool kF16>
constexpr uint32_t idesc_pv() {
  return kF16 ? ptx::idesc_f16_f32(128, 256, false, true) : ptx::idesc_bf16_f32(128, 256, false, true);
}

// mbarrier slots (8 bytes each) at kOffBar
enum {
  B_FULL0 = 0, B_EMPTY0 = kNS, B_QFULL = 2 * kNS, B_QPEFULL, B_QPEEMPTY, B_SFULL, B_SFREE,
  B_PFULL0, B_PFULL1, B_PVDONE0, B_PVDONE1, B_XFULL0, B_XFULL1, B_XEMPTY0, B_XEMPTY1, B_OFREE, B_TEARDOWN,
  B_STGREADY0, B_STGREADY1, B_STGFREE0, B_STGFREE1,
  B_RED0,                    // [quarter][page parity]: both halves' row maxima written (2 warps)
  B_LRED0 = B_RED0 + 8,      // [quarter]: both halves' row sums written (2 warps)
  B_CONV0 = B_LRED0 + 4,     // [stage] fp8 cache: the stage converted to bf16 (4 converter warps)
  B_CVREAD = B_CONV0 + kNS,  // fp8 cache: every converter has read the page's e4m3 bytes (4 warps)
  B_COUNT = B_CVREAD + 1
};
static_assert(B_COUNT * 8 <= kBarArea - 16, "barrier area");

struct Shared {
  uint8_t* base;       // 1 KB aligned
  uint32_t base_u32;
  volatile int* abort;
  uint32_t* tmem_slot;
  __device__ uint32_t bar(int i) const { return base_u32 + kOffBar + 8 * i; }
  __device__ uint32_t stage(int s) const { return base_u32 + kOffStage + s * kStageBytes; }
  __device__ uint32_t xbuf(int j) const { return base_u32 + kOffX + j * kXBytes; }
  __device__ uint32_t stg(int j) const { return base_u32 + kOffStg + j * kXBytes; }
  __device__ uint32_t qpe() const { return base_u32 + kOffQPe; }
};

// The limit and the status word are read from the kernel's parameters on the slow path only:
// a limit held in a register cost the fp8 kernel (96 registers a thread) about 4% of its time.
__device__ __forceinline__ bool wait_bar(const Shared& sh, uint32_t bar, uint32_t parity,
                                         const DecodeParams& p, bool cluster_scope = false) {
  // polled without a suspend hint: waking a suspended warp costs more than the issue
  // slots the polling takes from the other warps
  auto probe = [&]() {
    return cluster_scope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
  };
  if (probe()) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (probe()) return true;
    if (*sh.abort) return false;
    if (ptx::globaltimer() - t0 > p.wait_limit_ns) {
      *sh.abort = 1;
      flag_status(p.status, MLA_ERR_TIMEOUT);
      return false;
    }
  }
}

// This worker's pages in processing order.
struct PageCursor {
  const WorkItem* items;
  int it, it1, pg;
  WorkItem item;
  __device__ void init(const DecodeParams& pp, int it0, int it_end) {
    items = pp.items;
    it = it0;
    it1 = it_end;
    if (it < it1) {
      item = items[it];
      pg = item.page_begin;
    }
  }
  __device__ bool valid() const { return it < it1; }
  __device__ bool first() const { return pg == item.page_begin; }
  __device__ bool last() const { return pg == item.page_end - 1; }
  __device__ void next() {
    if (++pg >= item.page_end) {
      if (++it < it1) {
        item = items[it];
        pg = item.page_begin;
      }
    }
  }
};

// ------------------------------------------------------------------------------- roles
// TMA: the k_pe part of Q_r once per work item, then the item's pages. A block-table
// entry outside the cache is flagged and replaced by page 0 (the request's result is then
// undefined, but nothing is read out of bounds). Rank 0 also asks L2 for the whole page
// (both CTAs' halves, 72 KB contiguous) kL2Ahead pages before its TMA load, so that the
// load, issued when a stage frees up, reads L2 rather than HBM.
// An fp8 cache lands as e4m3 bytes (18 KB, unswizzled) in the back half of the stage, for
// the converter warps to expand into the bf16 layout the MMAs read.
// kHook: the testing hook (mla_decode_opts.withhold_page) is compiled into a loop of its own,
// taken by worker 0 only when the hook is set: inside the common loop its test cost the fp8
// kernel about 4% of its time.
template <bool kFp8, bool kB128, bool kHook>
__device__ void producer_loop(const Shared& sh, const DecodeParams& p, const CUtensorMap* tm_kc,
                              const CUtensorMap* tm_kpe, const CUtensorMap* tm_qpe,
                              const CUtensorMap* tm_sc, int worker, int rank) {
  constexpr int kRowBytes = kB128 ? kB128RowBytes : kD * (kFp8 ? 1 : 2);   // cache bytes per row
  const int it0 = p.worker_off[worker], it1 = p.worker_off[worker + 1];
  const uint8_t* cache = reinterpret_cast<const uint8_t*>(p.cache);
  // the cache is read once: its lines go first out of L2, so that what this decode reads
  // again (queries, and the split partials the combine kernel merges) stays there
  const uint64_t pol = ptx::l2_policy_evict_first();
  PageCursor ahead;
  ahead.init(p, it0, it1);
  auto prefetch_next = [&]() {
    if (rank != 0 || !ahead.valid()) return;
    const int page = p.block_table[(long long)(ahead.item.group / p.q_len) * p.max_pages + ahead.pg];
    if (page >= 0 && page < p.num_pages)
      ptx::bulk_prefetch_l2_hint(cache + (long long)page * (kP * kRowBytes), kP * kRowBytes, pol);
    ahead.next();
  };
  for (int i = 0; i < kL2Ahead; ++i) ahead.next();      // pages 0..kL2Ahead-1 load directly
  int stage = 0;
  uint32_t wrap = 0, q_iter = 0, np_seq = 0;
  for (int it = it0; it < it1; ++it) {
    const WorkItem item = p.items[it];
    const int g = item.group, b = g / p.q_len;
    if (!wait_bar(sh, sh.bar(B_QPEEMPTY), (q_iter & 1) ^ 1, p)) return;
    ptx::mbar_arrive_expect_tx(sh.bar(B_QPEFULL), kQPeBytes);
    ptx::tma_load_3d(sh.qpe(), tm_qpe, 32 * rank, 0, g, sh.bar(B_QPEFULL));
    ++q_iter;
    // the next item's latent query half (read by the send warps at its first page) and its
    // rotated part into L2, kQAhead pages before this item ends (earlier, it would be
    // evicted by the cache stream before use)
    const int q_at = max(item.page_begin, item.page_end - kQAhead);
    for (int pg = item.page_begin; pg < item.page_end; ++pg) {
      if (pg == q_at && it + 1 < it1) {
        const bf16* qn = reinterpret_cast<const bf16*>(p.q_lat) + (long long)p.items[it + 1].group * kH * kD;
        ptx::bulk_prefetch_l2(qn + 32 * rank * kH * 8, 32 * kH * 8 * 2);
        ptx::bulk_prefetch_l2(qn + kDC * kH, kH * kDR * 2);
      }
      int page = p.block_table[(long long)b * p.max_pages + pg];
      if (page < 0 || page >= p.num_pages) {
        if (rank == 0) flag_status(p.status, MLA_ERR_DEVICE_GUARD);
        page = 0;
      }
      if (!wait_bar(sh, sh.bar(B_EMPTY0 + stage), (wrap & 1) ^ 1, p)) return;
      const uint32_t full = sh.bar(B_FULL0 + stage);
      if constexpr (kHook) {
        // testing hook: this page of worker 0 is never loaded, so the wait for it runs out
        if (np_seq == (uint32_t)(p.withhold_page - 1)) {
          prefetch_next();
          ++np_seq;
          if (++stage == kNS) {
            stage = 0;
            ++wrap;
          }
          continue;
        }
        ++np_seq;
      }
      if constexpr (kB128) {
        const uint32_t st = sh.stage(stage);
        ptx::mbar_arrive_expect_tx(full, 16384 + 64 * 16 + kKTilePE);
        ptx::tma_load_2d_hint(st + kB128Codes, tm_kc, 256 * rank, page * kP, full, pol);
        ptx::tma_load_2d_hint(st + kB128Codes + 8192, tm_kc, 256 * rank + 128, page * kP, full, pol);
        ptx::tma_load_2d_hint(st + kB128Scales, tm_sc, kDC, page * kP, full, pol);
        ptx::tma_load_2d_hint(st + 4 * kKTileC, tm_kpe, kDC + kDC / 32 + 64 * rank, page * kP, full,
                              pol);
      } else if constexpr (kFp8) {
        const uint32_t land = sh.stage(stage) + kStageBytes / 2;
        ptx::mbar_arrive_expect_tx(full, kStageBytes / 2);
        ptx::tma_load_2d_hint(land, tm_kc, 256 * rank, page * kP, full, pol);
        ptx::tma_load_2d_hint(land + 8192, tm_kc, 256 * rank + 128, page * kP, full, pol);
        ptx::tma_load_2d_hint(land + 16384, tm_kpe, kDC + 32 * rank, page * kP, full, pol);
      } else {
        ptx::mbar_arrive_expect_tx(full, kStageBytes);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          ptx::tma_load_2d_hint(sh.stage(stage) + c * kKTileC, tm_kc, 256 * rank + 64 * c, page * kP,
                                full, pol);
        ptx::tma_load_2d_hint(sh.stage(stage) + 4 * kKTileC, tm_kpe, kDC + 32 * rank, page * kP, full,
                              pol);
      }
      prefetch_next();
      if (++stage == kNS) {
        stage = 0;
        ++wrap;
      }
    }
  }
}

template <bool kFp8, bool kB128>
__device__ void producer(const Shared& sh, const DecodeParams& p, const CUtensorMap* tm_kc,
                         const CUtensorMap* tm_kpe, const CUtensorMap* tm_qpe,
                         const CUtensorMap* tm_sc, int worker, int rank) {
  if (worker == 0 && p.withhold_page > 0)
    producer_loop<kFp8, kB128, true>(sh, p, tm_kc, tm_kpe, tm_qpe, tm_sc, worker, rank);
  else
    producer_loop<kFp8, kB128, false>(sh, p, tm_kc, tm_kpe, tm_qpe, tm_sc, worker, rank);
}

// Score MMAs: S = Q_r K_r^T for every page, as soon as the page has landed (with an fp8
// cache: has been converted) and the exchange warps have read the previous raw scores.
template <bool kFp8, bool kF16>
__device__ void qk_issuer(const Shared& sh, const DecodeParams& p, uint32_t tmem, int worker) {
  constexpr uint32_t kIdescQK = idesc_qk<kF16>();
  const int it0 = p.worker_off[worker], it1 = p.worker_off[worker + 1];
  int stage = 0;
  uint32_t wrap = 0, n = 0, item_idx = 0;
  for (int it = it0; it < it1; ++it) {
    const WorkItem item = p.items[it];
    for (int pg = item.page_begin; pg < item.page_end; ++pg) {
      if (pg == item.page_begin) {
        if (!wait_bar(sh, sh.bar(B_QFULL), item_idx & 1, p)) return;
        if (!wait_bar(sh, sh.bar(B_QPEFULL), item_idx & 1, p)) return;
      }
      if (!wait_bar(sh, sh.bar((kFp8 ? B_CONV0 : B_FULL0) + stage), wrap & 1, p)) return;
      if (!wait_bar(sh, sh.bar(B_SFREE), (n & 1) ^ 1, p)) return;
      ptx::tc_fence_after();
      const uint32_t st = sh.stage(stage);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint64_t bd = ptx::smem_desc(st + (j >> 2) * kKTileC + 32 * (j & 3), 16, 1024,
                                           ptx::kSwizzle128);
        ptx::mma_bf16_ts(tmem + kColS, tmem + kColQ + 8 * j, bd, kIdescQK, j ? 1u : 0u);
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint64_t a = ptx::smem_desc(sh.qpe() + 32 * k, 16, 512, ptx::kSwizzle64);
        const uint64_t bd = ptx::smem_desc(st + 4 * kKTileC + 32 * k, 16, 512, ptx::kSwizzle64);
        ptx::mma_bf16_ss(tmem + kColS, a, bd, kIdescQK, 1u);
      }
      ptx::mma_commit(sh.bar(B_SFULL));
      if (pg == item.page_end - 1) ptx::mma_commit(sh.bar(B_QPEEMPTY));
      ++n;
      if (++stage == kNS) {
        stage = 0;
        ++wrap;
      }
    }
    ++item_idx;
  }
}

// Output MMAs: O_r += P C_r once P is in TMEM. The page's score MMA finished before its P
// existed, so the stage is free once this product is done.
template <bool kF16>
__device__ void pv_issuer(const Shared& sh, const DecodeParams& p, uint32_t tmem, int worker) {
  constexpr uint32_t kIdescPV = idesc_pv<kF16>();
  const int it0 = p.worker_off[worker], it1 = p.worker_off[worker + 1];
  int stage = 0;
  uint32_t n = 0, item_idx = 0;
  for (int it = it0; it < it1; ++it) {
    const WorkItem item = p.items[it];
    for (int pg = item.page_begin; pg < item.page_end; ++pg) {
      const bool first = (pg == item.page_begin);
      if (!wait_bar(sh, sh.bar(B_PFULL0 + (n & 1)), (n >> 1) & 1, p)) return;
      if (first && !wait_bar(sh, sh.bar(B_OFREE), (item_idx & 1) ^ 1, p)) return;
      ptx::tc_fence_after();
      const uint32_t sb = sh.stage(stage);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t bd = ptx::smem_desc(sb + 2048 * k, kKTileC, 1024, ptx::kSwizzle128);
        ptx::mma_bf16_ts(tmem + kColO, tmem + kColP + 32 * (n & 1) + 8 * k, bd, kIdescPV,
                         (!first || k) ? 1u : 0u);
      }
      ptx::mma_commit(sh.bar(B_EMPTY0 + stage));
      ptx::mma_commit(sh.bar(B_PVDONE0 + (n & 1)));
      ++n;
      if (++stage == kNS) stage = 0;
    }
    ++item_idx;
  }
}

// Q_r latent part of one head row (group g) into TMEM: 256 bf16, two per column. The query
// is planar ([d_c / 8][128 heads][8] per group), so each 16-byte load of a warp (32
// consecutive head rows) reads one contiguous 512-byte run. Four batches of 64 dims, the
// loads of batch k + 1 issued before batch k is stored.
__device__ __forceinline__ void store_q(const DecodeParams& p, uint32_t t_row, int g, int row,
                                        int rank) {
  const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(p.q_lat) +
                                                    (long long)g * kH * kD) + (32 * rank) * kH + row;
  uint4 cur[8], nxt[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) cur[i] = src[i * kH];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k < 3) {
#pragma unroll
      for (int i = 0; i < 8; ++i) nxt[i] = src[(8 * (k + 1) + i) * kH];
    }
    uint32_t v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[4 * i] = cur[i].x; v[4 * i + 1] = cur[i].y; v[4 * i + 2] = cur[i].z; v[4 * i + 3] = cur[i].w;
    }
    ptx::tmem_st32(t_row + kColQ + 32 * k, v);
    if (k < 3) {
#pragma unroll
      for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
    }
  }
  ptx::tmem_wait_st();
}

// Send warps: raw partial of every page -> fp16 -> staging buffer n & 1 -> (bulk copy)
// the peer's receive buffer n & 1; Q_r's latent part into TMEM at each item's start.
__device__ void send_warps(const Shared& sh, const DecodeParams& p, uint32_t tmem, int worker, int rank,
                           int warp, int lane) {
  const int quarter = warp & 3;
  const int row = 32 * quarter + lane;
  const uint32_t t_row = tmem + ((uint32_t)(32 * quarter) << 16);
  const uint32_t peer = (uint32_t)(rank ^ 1);
  const uint32_t peer_x = ptx::map_to_rank(sh.xbuf(0), peer);
  const uint32_t peer_xfull0 = ptx::map_to_rank(sh.bar(B_XFULL0), peer);
  const int sw = row & 7;                                // 16-byte chunk swizzle of 128-byte rows
  PageCursor cur;
  cur.init(p, p.worker_off[worker], p.worker_off[worker + 1]);
  uint32_t n = 0;
  while (cur.valid()) {
    // a page that opens a work item needs that item's Q_r: every score MMA of the previous
    // item is done, since the previous page's raw scores were read
    if (cur.first()) {
      store_q(p, t_row, cur.item.group, row, rank);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sh.bar(B_QFULL));
    }
    if (!wait_bar(sh, sh.bar(B_SFULL), n & 1, p)) return;
    ptx::tc_fence_after();
    uint32_t r[64];
    ptx::tmem_ld32(t_row + kColS, *reinterpret_cast<uint32_t(*)[32]>(r));
    ptx::tmem_ld32(t_row + kColS + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
    ptx::tmem_wait_ld();
    ptx::tc_fence_before();
    __syncwarp();
    const uint32_t j = n % kXB, xpar = (n / kXB) & 1;
    int ok = 1;
    if (lane == 0) {
      ptx::mbar_arrive(sh.bar(B_SFREE));
      // staging buffer j: our softmax has read page n - kXB from it, and the peer has read
      // its receive buffer j (so the copy of page n - kXB out of staging j has landed)
      ok = wait_bar(sh, sh.bar(B_STGFREE0 + j), xpar ^ 1, p) &&
                   wait_bar(sh, sh.bar(B_XEMPTY0 + j), xpar ^ 1, p, true)
               ? 1 : 0;
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    // columns past the last token (rows that may hold anything) go out as 0, and finite
    // values beyond the fp16 range saturate instead of becoming infinite
    const int ntok = min(kP, cur.item.kv - cur.pg * kP);
    if (ntok < kP) {
#pragma unroll
      for (int i = 0; i < 64; ++i)
        if (i >= ntok) r[i] = 0u;
    }
    uint8_t* srow = sh.base + kOffStg + j * kXBytes + row * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        w[k] = ptx::f2h2_satfinite(__uint_as_float(r[8 * c + 2 * k]), __uint_as_float(r[8 * c + 2 * k + 1]));
      *reinterpret_cast<uint4*>(srow + ((c ^ sw) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      ptx::mbar_arrive(sh.bar(B_STGREADY0 + j));
      // one 16 KB copy per page once all four quarters are staged: a bulk copy between
      // CTAs costs about the same fixed time whatever its size up to 16 KB
      if (quarter == 0) {
        ok = wait_bar(sh, sh.bar(B_STGREADY0 + j), xpar, p) ? 1 : 0;
        if (ok) {
          ptx::bulk_s2s(peer_x + j * kXBytes, sh.stg(j), kXBytes, peer_xfull0 + 8 * j);
          ptx::bulk_commit();
        }
      }
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    ++n;
    cur.next();
  }
}

// Softmax warps: the pair's fp16 partial scores -> combined scores -> online softmax -> P
// into TMEM buffer n & 1; the item's output at its last page. Thread (row, half) handles
// columns [32 half, 32 half + 32) of each page and O columns [128 half, 128 half + 128).
template <bool kF16>
__device__ void softmax_epilogue(const Shared& sh, const DecodeParams& p, uint32_t tmem, int worker,
                                 int rank, int warp, int lane) {
  const int quarter = warp & 3;
  const int half = (warp - 6) >> 2;
  const int row = 32 * quarter + lane;
  const int tid = 32 * (warp - 6) + lane;                // 0..255 over the softmax warps
  const uint32_t t_row = tmem + ((uint32_t)(32 * quarter) << 16);
  const uint32_t peer_xempty0 = ptx::map_to_rank(sh.bar(B_XEMPTY0), (uint32_t)(rank ^ 1));
  const int sw = row & 7;
  float* red = reinterpret_cast<float*>(sh.base + kOffRed);    // [page parity][half][row]
  float* lsum = reinterpret_cast<float*>(sh.base + kOffLsum);  // [half][row]
  uint32_t n_items = 0;
  PageCursor cur;
  cur.init(p, p.worker_off[worker], p.worker_off[worker + 1]);
  uint32_t n = 0;
  float m_used = -INFINITY, l = 0.f;
  while (cur.valid()) {
    const WorkItem& item = cur.item;
    const int pg = cur.pg;
    if (cur.first()) {
      m_used = -INFINITY;
      l = 0.f;
    }
    const int ntok = min(kP, item.kv - pg * kP);

    // page n's fp16 partials for our 32 columns: the peer's (receive buffer n % kXB) and
    // our own (staging n % kXB); P goes to TMEM buffer n & 1
    const uint32_t xj = n % kXB, xpar = (n / kXB) & 1;
    const uint32_t j = n & 1;
    if (!wait_bar(sh, sh.bar(B_XFULL0 + xj), xpar, p, true)) return;
    if (warp == 6 && lane == 0) ptx::mbar_arrive_expect_tx(sh.bar(B_XFULL0 + xj), kXBytes);
    if (!wait_bar(sh, sh.bar(B_STGREADY0 + xj), xpar, p)) return;
    uint32_t xa[16], xb[16];                              // packed fp16 pairs, columns 32 half + 2i, +1
    {
      const uint8_t* xrow = sh.base + kOffX + xj * kXBytes + row * 128;
      const uint8_t* srow = sh.base + kOffStg + xj * kXBytes + row * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int cc = 4 * half + c;
        const uint4 a = *reinterpret_cast<const uint4*>(xrow + ((cc ^ sw) * 16));
        const uint4 b = *reinterpret_cast<const uint4*>(srow + ((cc ^ sw) * 16));
        xa[4 * c] = a.x; xa[4 * c + 1] = a.y; xa[4 * c + 2] = a.z; xa[4 * c + 3] = a.w;
        xb[4 * c] = b.x; xb[4 * c + 1] = b.y; xb[4 * c + 2] = b.z; xb[4 * c + 3] = b.w;
      }
      // every lane's buffer reads have returned before the buffers are released
      uint32_t dep = 0;
#pragma unroll
      for (int i = 0; i < 16; i += 4) dep ^= xa[i] ^ xb[i];
      const uint32_t all = __ballot_sync(0xffffffffu, dep != 0x7fc00001u);
      if (lane == 0) {
        ptx::mbar_arrive_remote_relaxed(peer_xempty0 + 8 * xj, all);
        ptx::mbar_arrive(sh.bar(B_STGFREE0 + xj));
      }
    }
    // Columns past the last token: both partials arrive as 0; make the peer's -inf so the
    // column gets P = 0. Their c_kv rows may hold anything, NaN included, and 0 * NaN would
    // poison O: zero them in the staged tiles before the P . C product reads them (the
    // score MMA that read them is done).
    bool zeroed = false;
    if (ntok < kP) {
      uint8_t* stg = sh.base + kOffStage + (int)(n % kNS) * kStageBytes;
      const int nrows = kP - ntok;
      const int per_tile = nrows * 8;
      for (int i = tid; i < 4 * per_tile; i += 32 * kSoftmaxWarps) {
        const int tile = i / per_tile, rem = i % per_tile;
        *reinterpret_cast<uint4*>(stg + tile * kKTileC + (ntok + rem / 8) * 128 + (rem % 8) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int col = 32 * half + 2 * i;
        if (col >= ntok) xa[i] = 0xFC00FC00u;
        else if (col + 1 >= ntok) xa[i] = (xa[i] & 0xFFFFu) | 0xFC000000u;
      }
      zeroed = true;
    }
    // row maximum (a reference point only: P may exceed 1 by the fp16 rounding of the sum,
    // far inside the 2^8 rescale margin): our 32 columns on packed fp16 sums, then the other
    // half's through shared memory
    volatile float* slot = red + (j * 2) * 128;
    float mine;
    {
      __half2 t[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const __half2 s0 = __hadd2(*reinterpret_cast<const __half2*>(&xa[2 * i]),
                                   *reinterpret_cast<const __half2*>(&xb[2 * i]));
        const __half2 s1 = __hadd2(*reinterpret_cast<const __half2*>(&xa[2 * i + 1]),
                                   *reinterpret_cast<const __half2*>(&xb[2 * i + 1]));
        t[i] = __hmax2(s0, s1);
      }
#pragma unroll
      for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) t[i] = __hmax2(t[i], t[i + w]);
      const float2 f = __half22float2(t[0]);
      mine = fmaxf(f.x, f.y);
      slot[half * 128 + row] = mine;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sh.bar(B_RED0 + 2 * quarter + j));
    }
    // P and its row sum against reference value m_ref
    uint32_t packed[16];
    float psum = 0.f;
    auto exps = [&](float m_ref) {
      const float neg_m = -m_ref;
      float e[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        e[2 * i] = ptx::add_f16lo_f32(xa[i], ptx::add_f16lo_f32(xb[i], neg_m));
        e[2 * i + 1] = ptx::add_f16hi_f32(xa[i], ptx::add_f16hi_f32(xb[i], neg_m));
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) e[i] = ptx::ex2(e[i]);
      float ps[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) ps[i] = (e[8 * i] + e[8 * i + 1]) + (e[8 * i + 2] + e[8 * i + 3]) +
                                      ((e[8 * i + 4] + e[8 * i + 5]) + (e[8 * i + 6] + e[8 * i + 7]));
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if constexpr (kF16) {
          const __half2 h2 = __floats2half2_rn(e[2 * i], e[2 * i + 1]);
          packed[i] = *reinterpret_cast<const uint32_t*>(&h2);
        } else {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(e[2 * i], e[2 * i + 1]);
          packed[i] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      }
      psum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
    };
    // Usually the running reference value stays (our half does not exceed it by more than
    // 2^8, and the other half rarely does): form P from it while the other half's maximum is
    // on its way, and recompute only if the full row maximum moves the reference (an item's
    // first page, or a rescale).
    const bool early = (m_used != -INFINITY) && !(mine > m_used + 8.f);
    if (early) exps(m_used);
    if (!wait_bar(sh, sh.bar(B_RED0 + 2 * quarter + j), (n >> 1) & 1, p)) return;
    const float mx = fmaxf(mine, slot[(half ^ 1) * 128 + row]);
    bool rescale = false;
    float alpha = 1.f;
    if (mx > -INFINITY) {
      if (m_used == -INFINITY) {
        m_used = mx;
      } else if (mx > m_used + 8.f) {
        alpha = ptx::ex2(m_used - mx);
        m_used = mx;
        l *= alpha;
        rescale = true;
      }
    }
    if (!early || rescale) {
      if (m_used == -INFINITY) {
#pragma unroll
        for (int i = 0; i < 16; ++i) packed[i] = 0u;
        psum = 0.f;
      } else {
        exps(m_used);
      }
    }
    l += psum;
    // P buffer n & 1 was last read by the product of page n-2; a rescale of O needs the
    // product of page n-1 done too
    if (n >= 2 && !wait_bar(sh, sh.bar(B_PVDONE0 + j), ((n >> 1) & 1) ^ 1, p)) return;
    // tcgen05 loads and stores are warp-collective: the warp rescales its 32 rows together
    // when any of them needs it (alpha is 1 for the others)
    const bool warp_rescale = __any_sync(0xffffffffu, rescale);
    if (warp_rescale && n >= 1 &&
        !wait_bar(sh, sh.bar(B_PVDONE0 + ((n - 1) & 1)), ((n - 1) >> 1) & 1, p))
      return;
    ptx::tc_fence_after();
    if (warp_rescale) {
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        const uint32_t col = kColO + 128 * half + 32 * c;
        ptx::tmem_ld32(t_row + col, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
        ptx::tmem_st32(t_row + col, v);
      }
    }
    ptx::tmem_st16(t_row + kColP + 32 * j + 16 * half, packed);
    ptx::tmem_wait_st();
    if (zeroed) ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(sh.bar(B_PFULL0 + j));

    // after the item's last page: normalise O_r and write it (output or split partial)
    if (cur.last()) {
      const int it = cur.it, g = item.group;
      // the row sum over both halves
      volatile float* lslot = lsum;
      lslot[half * 128 + row] = l;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sh.bar(B_LRED0 + quarter));
      if (!wait_bar(sh, sh.bar(B_LRED0 + quarter), n_items & 1, p)) return;
      ++n_items;
      const float l_row = l + lslot[(half ^ 1) * 128 + row];
      if (!wait_bar(sh, sh.bar(B_PVDONE0 + j), (n >> 1) & 1, p)) return;
      ptx::tc_fence_after();
      const float inv = (l_row > 0.f) ? p.out_scale / l_row : 0.f;
      const float lse_v = (l_row > 0.f) ? (m_used + log2f(l_row)) * kLn2 : -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        ptx::tmem_ld32(t_row + kColO + 128 * half + 32 * c, v);
        ptx::tmem_wait_ld();
        if (item.single) {
          const int col = 256 * rank + 128 * half + 32 * c;
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(p.out_latent) +
                                                ((long long)g * kH + row) * kDC + col);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[8 * q + 2 * jj]) * inv,
                                                              __uint_as_float(v[8 * q + 2 * jj + 1]) * inv);
              w[jj] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          // octet-planar bf16 partial: dims 8o..8o+7 of head row at part_o[it][o][row][0:8]
          const int o0 = 32 * rank + 16 * half + 4 * c;
          uint4* dst = reinterpret_cast<uint4*>(p.part_o) + ((long long)it * (kDC / 8) + o0) * kH + row;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[8 * q + 2 * jj]) * inv,
                                                              __uint_as_float(v[8 * q + 2 * jj + 1]) * inv);
              w[jj] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            dst[(long long)q * kH] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sh.bar(B_OFREE));
      if (rank == 0 && half == 0) {
        if (item.single) p.lse[(long long)g * kH + row] = lse_v;
        else p.part_lse[(long long)it * kH + row] = lse_v;
      }
    }
    ++n;
    cur.next();
  }
}

// Four e4m3 values (low byte first) -> four f16 as two f16x2 words (low pair first), exactly:
// every e4m3 value (at most 4 significant bits, exponents 2^-9 .. 2^8) is an f16 value. The
// word's two 16-bit halves go to the two conversions without shifts or masks.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi) : "r"(w));
}

// Four e4m3 codes (low byte first) times a block scale -> four bf16 as two bf16x2 words, each
// rounded to nearest even once: the codes convert exactly to f16 and then f32, the products
// are IEEE f32 multiplies (two at a time), and only their bf16 rounding is inexact.
__device__ __forceinline__ void e4m3x4_to_bf16x4_scaled(uint32_t w, uint64_t s2, uint32_t& lo,
                                                        uint32_t& hi) {
  uint32_t h0, h1;
  e4m3x4_to_f16x4(w, h0, h1);
  asm("{\n\t.reg .b16 a, b, c, d;\n\t.reg .f32 fa, fb, fc, fd;\n\t.reg .b64 p, q;\n\t"
      "mov.b32 {a, b}, %2;\n\tmov.b32 {c, d}, %3;\n\t"
      "cvt.f32.f16 fa, a;\n\tcvt.f32.f16 fb, b;\n\tcvt.f32.f16 fc, c;\n\tcvt.f32.f16 fd, d;\n\t"
      "mov.b64 p, {fa, fb};\n\tmov.b64 q, {fc, fd};\n\t"
      "mul.rn.f32x2 p, p, %4;\n\tmul.rn.f32x2 q, q, %4;\n\t"
      "mov.b64 {fa, fb}, p;\n\tmov.b64 {fc, fd}, q;\n\t"
      "cvt.rn.bf16x2.f32 %0, fb, fa;\n\tcvt.rn.bf16x2.f32 %1, fd, fc;\n\t}"
      : "=r"(lo), "=r"(hi) : "r"(h0), "r"(h1), "l"(s2));
}

__device__ __forceinline__ void e4m3x16_to_bf16_scaled(const uint4& in, float s, uint4& lo, uint4& hi) {
  const uint64_t s2 = ((uint64_t)__float_as_uint(s) << 32) | __float_as_uint(s);
  e4m3x4_to_bf16x4_scaled(in.x, s2, lo.x, lo.y);
  e4m3x4_to_bf16x4_scaled(in.y, s2, lo.z, lo.w);
  e4m3x4_to_bf16x4_scaled(in.z, s2, hi.x, hi.y);
  e4m3x4_to_bf16x4_scaled(in.w, s2, hi.z, hi.w);
}

// 16 e4m3 bytes -> 16 f16 as two 16-byte vectors (elements in order).
__device__ __forceinline__ void e4m3x16_to_f16(const uint4& in, uint4& lo, uint4& hi) {
  e4m3x4_to_f16x4(in.x, lo.x, lo.y);
  e4m3x4_to_f16x4(in.y, lo.z, lo.w);
  e4m3x4_to_f16x4(in.z, hi.x, hi.y);
  e4m3x4_to_f16x4(in.w, hi.z, hi.w);
}

// Converter warps (fp8 cache): each page's e4m3 slice (two 128-dim boxes and the 32-dim
// rope box, unswizzled, in the back half of the stage) -> the 16-bit slice in the layout the
// MMAs read (four 64-dim SW128 chunks and the SW64 rope tile, the whole stage). Per-tensor
// codes become f16 exactly, one instruction per pair (the kernel's MMAs then run on f16
// operands); the cache's scale is folded into the query and the output.
// The 16-bit writes overlap the e4m3 bytes, so every converter reads its share first and the
// four warps meet at a barrier before any writes. Thread t reads eight 16-byte units of the
// c boxes (a warp covers 4 rows x 128 bytes, conflict-free) and one of the rope box.
// Block-scaled cache (kB128): the 256 codes of each row are read with the row's two scales
// of this CTA's dims (blocks 2 rank, 2 rank + 1), converted as code * scale rounded to bf16,
// and written like the per-tensor codes; k_pe arrived in bf16 and is not touched.
template <bool kB128>
__device__ void convert_warps(const Shared& sh, const DecodeParams& p, int worker, int rank, int warp,
                              int lane) {
  const int t = 32 * (warp - kWarpConv0) + lane;         // 0..127
  PageCursor cur;
  cur.init(p, p.worker_off[worker], p.worker_off[worker + 1]);
  int stage = 0;
  uint32_t wrap = 0, n = 0;
  while (cur.valid()) {
    if (!wait_bar(sh, sh.bar(B_FULL0 + stage), wrap & 1, p)) return;
    uint8_t* st = sh.base + kOffStage + stage * kStageBytes;
    const uint8_t* land = st + (kB128 ? kB128Codes : kStageBytes / 2);
    uint4 in[9];
    float scl[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = t + 128 * k, j = i >> 9, r = (i >> 3) & 63, u = i & 7;
      in[k] = *reinterpret_cast<const uint4*>(land + 8192 * j + 128 * r + 16 * u);
      if constexpr (kB128)
        scl[k] = reinterpret_cast<const float*>(st + kB128Scales)[4 * r + 2 * rank + j];
    }
    if constexpr (kB128) in[8] = in[0];
    else in[8] = *reinterpret_cast<const uint4*>(land + 16384 + 32 * (t >> 1) + 16 * (t & 1));
    // every lane's reads have returned (their values are used) before the warp reports
    uint32_t dep = 0;
#pragma unroll
    for (int k = 0; k < 9; ++k) dep ^= in[k].x;
    if constexpr (kB128) {
#pragma unroll
      for (int k = 0; k < 8; ++k) dep ^= __float_as_uint(scl[k]);
    }
    const uint32_t all = __ballot_sync(0xffffffffu, dep != 0x7fc00001u);
    if (lane == 0 && all != 0x12345678u) ptx::mbar_arrive(sh.bar(B_CVREAD));
    if (!wait_bar(sh, sh.bar(B_CVREAD), n & 1, p)) return;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = t + 128 * k, j = i >> 9, r = (i >> 3) & 63, u = i & 7;
      // dims 128 j + 16 u .. +15 = 64-dim chunk 2 j + u / 4, 16-byte units 2 (u % 4), +1
      uint8_t* row = st + (2 * j + (u >> 2)) * kKTileC + 128 * r;
      const int cb = 2 * (u & 3);
      uint4 lo, hi;
      if constexpr (kB128) e4m3x16_to_bf16_scaled(in[k], scl[k], lo, hi);
      else e4m3x16_to_f16(in[k], lo, hi);
      *reinterpret_cast<uint4*>(row + ((cb ^ (r & 7)) * 16)) = lo;
      *reinterpret_cast<uint4*>(row + (((cb + 1) ^ (r & 7)) * 16)) = hi;
    }
    if constexpr (!kB128) {
      // rope dims 16 u .. +15 of row r -> 16-byte units 2 u, +1 of the 64-byte SW64 row
      // (64-byte swizzle: unit ^= (row >> 1) & 3)
      const int r = t >> 1, cb = 2 * (t & 1);
      uint8_t* row = st + 4 * kKTileC + 64 * r;
      uint4 lo, hi;
      e4m3x16_to_f16(in[8], lo, hi);
      *reinterpret_cast<uint4*>(row + ((cb ^ ((r >> 1) & 3)) * 16)) = lo;
      *reinterpret_cast<uint4*>(row + (((cb + 1) ^ ((r >> 1) & 3)) * 16)) = hi;
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(sh.bar(B_CONV0 + stage));
    ++n;
    if (++stage == kNS) {
      stage = 0;
      ++wrap;
    }
    cur.next();
  }
}

template <bool kFp8, bool kB128>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFp8 ? kThreadsFp8 : kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_kc,
                     const __grid_constant__ CUtensorMap tm_kpe,
                     const __grid_constant__ CUtensorMap tm_qpe,
                     const __grid_constant__ CUtensorMap tm_sc, const DecodeParams p) {
  // per-tensor e4m3 cache: f16 operands (the query arrives in f16 from the prologue)
  constexpr bool kF16 = kFp8 && !kB128;
  extern __shared__ uint8_t smem_raw[];
  Shared sh;
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t aligned = (raw + 1023u) & ~1023u;
  sh.base = smem_raw + (aligned - raw);
  sh.base_u32 = aligned;
  sh.abort = reinterpret_cast<volatile int*>(sh.base + kOffBar + kBarArea - 16);
  sh.tmem_slot = reinterpret_cast<uint32_t*>(sh.base + kOffBar + kBarArea - 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)ptx::cluster_ctarank();
  const int worker = blockIdx.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      ptx::mbar_init(sh.bar(B_FULL0 + s), 1);
      ptx::mbar_init(sh.bar(B_EMPTY0 + s), 1);
    }
    ptx::mbar_init(sh.bar(B_QFULL), 4);
    ptx::mbar_init(sh.bar(B_QPEFULL), 1);
    ptx::mbar_init(sh.bar(B_QPEEMPTY), 1);
    ptx::mbar_init(sh.bar(B_SFULL), 1);
    ptx::mbar_init(sh.bar(B_SFREE), 4);
    ptx::mbar_init(sh.bar(B_PFULL0), kSoftmaxWarps);
    ptx::mbar_init(sh.bar(B_PFULL1), kSoftmaxWarps);
    ptx::mbar_init(sh.bar(B_PVDONE0), 1);
    ptx::mbar_init(sh.bar(B_PVDONE1), 1);
    ptx::mbar_init(sh.bar(B_XFULL0), 1);
    ptx::mbar_init(sh.bar(B_XFULL1), 1);
    ptx::mbar_init(sh.bar(B_XEMPTY0), kSoftmaxWarps);
    ptx::mbar_init(sh.bar(B_XEMPTY1), kSoftmaxWarps);
    ptx::mbar_init(sh.bar(B_OFREE), kSoftmaxWarps);
    ptx::mbar_init(sh.bar(B_TEARDOWN), 2);
    if (kFp8) {
      for (int s = 0; s < kNS; ++s) ptx::mbar_init(sh.bar(B_CONV0 + s), 4);
      ptx::mbar_init(sh.bar(B_CVREAD), 4);
    }
    ptx::mbar_init(sh.bar(B_STGREADY0), 4);
    ptx::mbar_init(sh.bar(B_STGREADY1), 4);
    ptx::mbar_init(sh.bar(B_STGFREE0), kSoftmaxWarps);
    ptx::mbar_init(sh.bar(B_STGFREE1), kSoftmaxWarps);
    for (int i = 0; i < 12; ++i) ptx::mbar_init(sh.bar(B_RED0 + i), 2);
    *sh.abort = 0;
    ptx::fence_mbar_init();
    // first phase of each receive buffer (the peer's partials of pages 0 .. kXB - 1)
    for (int x = 0; x < kXB; ++x) ptx::mbar_arrive_expect_tx(sh.bar(B_XFULL0 + x), kXBytes);
    ptx::prefetch_tensormap(&tm_kc);
    ptx::prefetch_tensormap(&tm_kpe);
    ptx::prefetch_tensormap(&tm_qpe);
    if (kB128) ptx::prefetch_tensormap(&tm_sc);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(sh.tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::cluster_sync();
  const uint32_t tmem = *sh.tmem_slot;
  // launched with programmatic serialization: the set-up above overlapped the prologue
  // kernels; the work list and the query are theirs, so wait for them here
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();

  if (warp == 0) {
    if (lane == 0) producer<kFp8, kB128>(sh, p, &tm_kc, &tm_kpe, &tm_qpe, &tm_sc, worker, rank);
  } else if (warp == 1) {
    if (lane == 0) qk_issuer<kFp8, kF16>(sh, p, tmem, worker);
  } else if (kFp8 && warp >= kWarpConv0) {
    convert_warps<kB128>(sh, p, worker, rank, warp, lane);
  } else if (warp <= 5) {
    send_warps(sh, p, tmem, worker, rank, warp, lane);
  } else if (warp <= 13) {
    softmax_epilogue<kF16>(sh, p, tmem, worker, rank, warp, lane);
  } else {
    if (lane == 0) pv_issuer<kF16>(sh, p, tmem, worker);
  }

  // teardown: every role gets here, normally or after a bounded wait gave up
  // both MMA issuers commit: every issued MMA must have finished before TMEM is released
  if ((warp == 1 || warp == 14) && lane == 0) ptx::mma_commit(sh.bar(B_TEARDOWN));
  if (warp >= 2 && warp <= 5 && lane == 0) ptx::bulk_wait_read_all();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {
      const uint64_t t0 = ptx::globaltimer();
      while (!ptx::mbar_try_wait(sh.bar(B_TEARDOWN), 0) && ptx::globaltimer() - t0 < p.wait_limit_ns) {
      }
    }
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  if (*sh.abort) {
    // let copies already in flight into this CTA's shared memory land before it exits
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < 2000000ull) {
    }
  }
  ptx::cluster_sync();
}

// ------------------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// 2-D bf16 tensor map over a row-major [rows][576] array; box = box_cols x box_rows.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_cols, uint32_t box_rows,
              CUtensorMapSwizzle swz) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over an e4m3 cache viewed as bytes [rows][576], unswizzled; box = box_cols x box_rows.
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_cols, uint32_t box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over a block-scaled fp8 cache viewed as bytes [rows][656]; box = box_cols x
// box_rows bytes, with the given swizzle.
bool make_map_b128(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_cols, uint32_t box_rows,
                   CUtensorMapSwizzle swz) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kB128RowBytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kB128RowBytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over the rotated query parts of the planar query ([groups][128][64] bf16 at
// element offset 512 * 128 of each 128 x 576 group block); box = 32 columns x 128 heads.
bool make_qpe_map(CUtensorMap* m, const void* q_lat, uint64_t groups) {
  auto enc = encoder();
  if (!enc) return false;
  const void* base = reinterpret_cast<const bf16*>(q_lat) + (long long)kDC * kH;
  cuuint64_t dims[3] = {(cuuint64_t)kDR, (cuuint64_t)kH, (cuuint64_t)groups};
  cuuint64_t strides[2] = {(cuuint64_t)kDR * 2, (cuuint64_t)kH * kD * 2};
  cuuint32_t box[3] = {32, (cuuint32_t)kH, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

bool tc_decode_supported(const mla_config* c) {
  return c && c->act_dtype == MLA_BF16 &&
         (c->cache_dtype == MLA_BF16 || c->cache_dtype == MLA_FP8_E4M3 ||
          c->cache_dtype == MLA_FP8_E4M3_B128) && c->num_heads == tc::kH &&
         c->d_latent == tc::kDC && c->d_rope == tc::kDR && c->page_size == tc::kP;
}

bool tc_decode_default_enabled() { return true; }

int tc_decode_max_workers() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    if (cudaFuncSetAttribute(tc::decode_tc_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             tc::kSmemBytes) != cudaSuccess)
      return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(tc::kThreads, 1, 1);
    cfg.dynamicSmemBytes = tc::kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc::decode_tc_kernel<false, false>, &cfg) != cudaSuccess || n <= 0)
      return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

cudaError_t launch_decode_tc(mla_dtype cache, const DecodeParams& p, cudaStream_t s) {
  if (cache != MLA_BF16 && cache != MLA_FP8_E4M3 && cache != MLA_FP8_E4M3_B128)
    return cudaErrorNotSupported;
  const bool b128 = (cache == MLA_FP8_E4M3_B128);
  const bool fp8 = (cache == MLA_FP8_E4M3) || b128;
  CUtensorMap kc, kpe, qpe, sc;
  const uint64_t cache_rows = (uint64_t)p.num_pages * tc::kP;
  const uint64_t groups = (uint64_t)p.batch * p.q_len;
  bool maps;
  if (b128)
    maps = tc::make_map_b128(&kc, p.cache, cache_rows, 128, 64, CU_TENSOR_MAP_SWIZZLE_NONE) &&
           tc::make_map_b128(&sc, p.cache, cache_rows, 16, 64, CU_TENSOR_MAP_SWIZZLE_NONE) &&
           tc::make_map_b128(&kpe, p.cache, cache_rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_64B);
  else if (fp8)
    maps = tc::make_map_u8(&kc, p.cache, cache_rows, 128, 64) &&
           tc::make_map_u8(&kpe, p.cache, cache_rows, 32, 64);
  else
    maps = tc::make_map(&kc, p.cache, cache_rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
           tc::make_map(&kpe, p.cache, cache_rows, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B);
  if (!maps || !tc::make_qpe_map(&qpe, p.q_lat, groups)) return cudaErrorInvalidValue;
  if (!b128) sc = kc;                                       // unused by the other layouts
  auto kern = b128 ? tc::decode_tc_kernel<true, true>
                   : (fp8 ? tc::decode_tc_kernel<true, false> : tc::decode_tc_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.workers, 1, 1);
  cfg.blockDim = dim3(fp8 ? tc::kThreadsFp8 : tc::kThreads, 1, 1);
  cfg.dynamicSmemBytes = tc::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, kc, kpe, qpe, sc, p);
  note_launch();
  return e;
}

}  // namespace mla
