// SIMT kernels of libmla: cache append (from latents or from hidden states), the tiled
// fp32-accumulating GEMM used by the weight fold, the query prologue and the output
// projection, the split planner, the SIMT decode kernel and the LSE combine.
//
// Page notation: huny.dev "DeepSeek MLA 해부" §2-1 (c_t = h_t W^DKV), §2-3 (k^R =
// RoPE(h_t W^KR), scores = content + rotary), §3-1 (absorbed query), §3-2 (W^UV W^O
// fold); secrett2633.cloud "[vLLM] Multi-head Latent Attention" (64-token pages, MQA
// decode over one combined kv_c_and_k_pe_cache, LSE return, split count num_splits).
#include <math.h>
#include <stdio.h>

#include "internal.h"
#include "prologue.cuh"
#include "sm100_ptx.cuh"

namespace mla {

// ======================================================================== tiled SIMT GEMM
// C[z] (M x N) = A[z] (M x K, row-major, lda) * B[z] (K x N, row-major, ldb), fp32
// accumulation; the epilogue receives 4 consecutive columns of one row.
constexpr int GT_M = 64, GT_N = 64, GT_K = 16;

template <typename TA, typename TB, class Epi>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const TA* __restrict__ A, long long lda,
                                                        long long sA, const TB* __restrict__ B,
                                                        long long ldb, long long sB, int M, int N,
                                                        int K, int k_chunk, Epi epi) {
  __shared__ float As[GT_K][GT_M + 4];
  __shared__ float Bs[GT_K][GT_N + 4];
  const int z = blockIdx.z;
  const int zb = z / ((K + k_chunk - 1) / k_chunk);       // batch index
  const int zk = z % ((K + k_chunk - 1) / k_chunk);       // K split index
  A += (long long)zb * sA;
  B += (long long)zb * sB;
  const int m0 = blockIdx.y * GT_M, n0 = blockIdx.x * GT_N;
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  const int kb = zk * k_chunk, ke = min(K, kb + k_chunk);
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = kb; k0 < ke; k0 += GT_K) {
    for (int i = tid; i < GT_M * GT_K; i += 256) {
      const int r = i / GT_K, kk = i % GT_K, gm = m0 + r, gk = k0 + kk;
      As[kk][r] = (gm < M && gk < ke) ? to_f32(A[(long long)gm * lda + gk]) : 0.f;
    }
    for (int i = tid; i < GT_K * GT_N; i += 256) {
      const int kk = i / GT_N, c = i % GT_N, gk = k0 + kk, gn = n0 + c;
      Bs[kk][c] = (gk < ke && gn < N) ? to_f32(B[(long long)gk * ldb + gn]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < GT_K; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = m0 + ty * 4 + i;
    if (row < M) epi(zb, row, n0 + tx * 4, acc[i], N);
  }
}

template <typename TA, typename TB, class Epi>
static cudaError_t simt_gemm(const TA* A, long long lda, long long sA, const TB* B, long long ldb,
                             long long sB, int M, int N, int K, int batch, int k_splits, Epi epi,
                             cudaStream_t s) {
  if (M <= 0 || N <= 0 || K <= 0 || batch <= 0) return cudaSuccess;
  int k_chunk = (K + k_splits - 1) / k_splits;
  k_chunk = (k_chunk + GT_K - 1) / GT_K * GT_K;
  const int splits = (K + k_chunk - 1) / k_chunk;
  dim3 grid((N + GT_N - 1) / GT_N, (M + GT_M - 1) / GT_M, batch * splits);
  simt_gemm_kernel<TA, TB, Epi><<<grid, 256, 0, s>>>(A, lda, sA, B, ldb, sB, M, N, K, k_chunk, epi);
  note_launch();
  return cudaGetLastError();
}

// Plain store into C[z * sC + row * ldc + col].
template <typename TC>
struct StoreEpi {
  TC* C;
  long long ldc, sC;
  __device__ void operator()(int z, int row, int col0, const float* v, int N) const {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (col0 + j < N) C[(long long)z * sC + (long long)row * ldc + col0 + j] = from_f32<TC>(v[j]);
  }
};

// fp32 atomic accumulation (split-K partial sums).
struct AtomicAddEpi {
  float* C;
  long long ldc;
  __device__ void operator()(int, int row, int col0, const float* v, int N) const {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (col0 + j < N) atomicAdd(&C[(long long)row * ldc + col0 + j], v[j]);
  }
};

// ======================================================================== cache append
// One block per token row: [c_kv | RoPE(k_pe)] encoded into its page slot.
template <typename AT, typename CT>
__global__ void __launch_bounds__(128) append_latent_kernel(
    const AT* __restrict__ c_kv, const AT* __restrict__ k_pe, long long ld_c, long long ld_k,
    const int32_t* req_ids, const int32_t* positions, const int32_t* block_table, int batch,
    int max_pages, CT* __restrict__ cache, int num_pages, int P, int d_c, int d_r, int rotate,
    RopeTable rt, float cache_scale, int32_t* status) {
  const int r = blockIdx.x;
  int pos = 0;
  const long long slot = append_slot(req_ids, positions, block_table, batch, max_pages, num_pages,
                                     P, r, (threadIdx.x == 0) ? status : nullptr, &pos);
  // a kernel launched after this one with programmatic serialization may start its set-up
  ptx::griddep_launch_dependents();
  if (slot < 0) return;
  // launched with programmatic serialization after the projection that writes c_kv / k_pe
  // (the finish of an append from h): its page slot is found while that GEMM ends (no-op
  // otherwise)
  ptx::griddep_wait();
  const int D = d_c + d_r;
  CT* dst = cache + slot * D;
  for (int e = threadIdx.x; e < D / 2; e += blockDim.x) {
    const int col = 2 * e;
    float x0, x1;
    if (col < d_c) {
      x0 = to_f32(c_kv[(long long)r * ld_c + col]);
      x1 = to_f32(c_kv[(long long)r * ld_c + col + 1]);
    } else {
      const int kc = col - d_c;
      x0 = to_f32(k_pe[(long long)r * ld_k + kc]);
      x1 = to_f32(k_pe[(long long)r * ld_k + kc + 1]);
      if (rotate) {
        float sn, cs;
        rope_sincos(rt, kc / 2, pos, &sn, &cs);
        const float y0 = x0 * cs - x1 * sn;
        const float y1 = x0 * sn + x1 * cs;
        x0 = y0;
        x1 = y1;
      }
    }
    dst[col] = CacheCodec<CT>::encode(x0, cache_scale);
    dst[col + 1] = CacheCodec<CT>::encode(x1, cache_scale);
  }
}

// One block (128 threads) per token row, block-scaled fp8 cache: the latent in e4m3 with
// one fp32 scale per 128 elements (amax / 448, then code = e4m3(x / scale), both IEEE
// divisions; a block of zeros keeps scale 0 and codes 0), then the rotated k_pe in bf16.
// Row bytes: [d_c codes][d_c / 128 fp32 scales][d_r bf16]. Warp w encodes latent blocks
// w, w + 4, ...: four consecutive elements per lane, the block maximum by warp shuffles.
template <typename AT>
__global__ void __launch_bounds__(128) append_latent_b128_kernel(
    const AT* __restrict__ c_kv, const AT* __restrict__ k_pe, long long ld_c, long long ld_k,
    const int32_t* req_ids, const int32_t* positions, const int32_t* block_table, int batch,
    int max_pages, uint8_t* __restrict__ cache, int num_pages, int P, int d_c, int d_r, int rotate,
    RopeTable rt, int32_t* status) {
  const int r = blockIdx.x;
  int pos = 0;
  const long long slot = append_slot(req_ids, positions, block_table, batch, max_pages, num_pages,
                                     P, r, (threadIdx.x == 0) ? status : nullptr, &pos);
  ptx::griddep_launch_dependents();
  if (slot < 0) return;
  ptx::griddep_wait();
  const long long row_bytes = (long long)d_c + d_c / 32 + 2LL * d_r;
  uint8_t* dst = cache + slot * row_bytes;
  float* scales = reinterpret_cast<float*>(dst + d_c);
  __nv_bfloat162* kdst = reinterpret_cast<__nv_bfloat162*>(dst + d_c + d_c / 32);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int blk = warp; blk < d_c / 128; blk += 4) {
    const int c0 = 128 * blk + 4 * lane;
    float x[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = to_f32(c_kv[(long long)r * ld_c + c0 + i]);
    const float amax = warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
    const float scale = amax / 448.f;
    uint32_t packed = 0u;
    if (scale > 0.f) {
#pragma unroll
      for (int i = 0; i < 4; ++i) packed |= (uint32_t)f32_to_fp8(x[i] / scale) << (8 * i);
    }
    *reinterpret_cast<uint32_t*>(dst + c0) = packed;
    if (lane == 0) scales[blk] = scale;
  }
  for (int e = threadIdx.x; e < d_r / 2; e += blockDim.x) {
    float x0 = to_f32(k_pe[(long long)r * ld_k + 2 * e]);
    float x1 = to_f32(k_pe[(long long)r * ld_k + 2 * e + 1]);
    if (rotate) {
      float sn, cs;
      rope_sincos(rt, e, pos, &sn, &cs);
      const float y0 = x0 * cs - x1 * sn;
      const float y1 = x0 * sn + x1 * cs;
      x0 = y0;
      x1 = y1;
    }
    kdst[e] = __floats2bfloat162_rn(x0, x1);
  }
}

// GEMM epilogue of the append from hidden states: row r of [c | k_raw] = h_r W.
template <typename CT>
struct AppendEpi {
  const int32_t* req_ids;
  const int32_t* positions;
  const int32_t* block_table;
  int batch, max_pages, num_pages, P, d_c, d_r;
  CT* cache;
  RopeTable rt;
  float cache_scale;
  int32_t* status;
  __device__ void operator()(int, int row, int col0, const float* v, int N) const {
    int pos = 0;
    const long long slot = append_slot(req_ids, positions, block_table, batch, max_pages,
                                       num_pages, P, row, (col0 == 0) ? status : nullptr, &pos);
    if (slot < 0) return;
    CT* dst = cache + slot * (d_c + d_r);
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      const int col = col0 + j;
      if (col >= N) break;
      float x0 = v[j], x1 = v[j + 1];
      if (col >= d_c) {
        float sn, cs;
        rope_sincos(rt, (col - d_c) / 2, pos, &sn, &cs);
        const float y0 = x0 * cs - x1 * sn;
        const float y1 = x0 * sn + x1 * cs;
        x0 = y0;
        x1 = y1;
      }
      dst[col] = CacheCodec<CT>::encode(x0, cache_scale);
      dst[col + 1] = CacheCodec<CT>::encode(x1, cache_scale);
    }
  }
};

// ======================================================================== weight fold
template <typename T>
__global__ void transpose_heads_kernel(const T* __restrict__ W_UK, T* __restrict__ W_UK_abs, int H,
                                       int d_c, int d_n) {
  const long long n_total = (long long)H * d_n * d_c;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(i % d_c);
    const long long hn = i / d_c;
    const int n = (int)(hn % d_n), h = (int)(hn / d_n);
    W_UK_abs[i] = W_UK[(long long)c * H * d_n + (long long)h * d_n + n];
  }
}

// ======================================================================== query prologue
// (rope_body in prologue.cuh)
template <typename T>
__global__ void __launch_bounds__(256) q_rope_kernel(const T* __restrict__ q_pe,
                                                     const int32_t* seq_lens, int batch, int q_len,
                                                     int H, int d_c, int d_r, RopeTable rt,
                                                     float qs, int planar, T* __restrict__ q_lat) {
  rope_body<T>(q_pe, seq_lens, q_len, H, d_c, d_r, rt, qs, planar, q_lat, blockIdx.x, blockIdx.y);
}

// ======================================================================== split planner
// (plan_body in plan.cuh)
__global__ void __launch_bounds__(256) plan_kernel(PlanParams p) {
  extern __shared__ int sm[];
  plan_body(p, sm, true);
}

// The bf16 decode prologue's small jobs in one launch. With a plan (pp.workers > 0) it is
// the first kernel of a decode call: block 0 clears the status word and plans the split
// work, and the query absorption GEMM follows with programmatic serialization. Without one
// (the GEMM's extra block plans) it follows the GEMM with programmatic serialization. The
// other blocks rotate q_pe (16 heads each); the kernel ends by waiting for the kernel before
// it, so that its completion implies the whole prologue's.
template <typename T>
__global__ void __launch_bounds__(256) prep_kernel(PlanParams pp, const T* __restrict__ q_pe,
                                                   const int32_t* seq_lens, int q_len, int H, int d_c,
                                                   int d_r, RopeTable rt, float qs, int planar,
                                                   T* __restrict__ q_lat, int hblocks, int f16) {
  extern __shared__ int sm[];
  const int plan = pp.workers > 0 ? 1 : 0;
  if (plan && blockIdx.x == 0) {
    if (threadIdx.x == 0) *pp.status = 0;
    __syncthreads();
  }
  ptx::griddep_launch_dependents();
  if (plan && blockIdx.x == 0) {
    plan_body(pp, sm, false);
  } else {
    const int b = blockIdx.x - plan;
    rope_body<T>(q_pe, seq_lens, q_len, H, d_c, d_r, rt, qs, planar, q_lat, b / hblocks, b % hblocks, 16,
                 f16);
  }
  ptx::griddep_wait();
}

// ======================================================================== SIMT decode
// One CTA = one worker x 8 heads (one warp per head). Per page: the page rows are
// copied into shared memory with an odd word stride (conflict-free row-parallel reads);
// lanes own tokens for the scores and latent dims for the output accumulation.
template <typename CT> struct PageElem;
template <> struct PageElem<float> {
  __device__ __forceinline__ static float get(const uint32_t* row, int k, int) {
    return __uint_as_float(row[k]);
  }
  __device__ __forceinline__ static float dot(const uint32_t* row, const float* q, int D, int) {
    float acc = 0.f;
    for (int w = 0; w < D; ++w) acc = fmaf(q[w], __uint_as_float(row[w]), acc);
    return acc;
  }
};
template <> struct PageElem<bf16> {
  __device__ __forceinline__ static float get(const uint32_t* row, int k, int) {
    const uint32_t w = row[k >> 1];
    return __uint_as_float((k & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
  __device__ __forceinline__ static float dot(const uint32_t* row, const float* q, int D, int) {
    float acc = 0.f;
    for (int w = 0; w < D / 2; ++w) {
      const uint32_t v = row[w];
      acc = fmaf(q[2 * w], __uint_as_float(v << 16), acc);
      acc = fmaf(q[2 * w + 1], __uint_as_float(v & 0xFFFF0000u), acc);
    }
    return acc;
  }
};
template <> struct PageElem<uint8_t> {
  __device__ __forceinline__ static float get(const uint32_t* row, int k, int) {
    return fp8_to_f32((uint8_t)(row[k >> 2] >> (8 * (k & 3))));
  }
  __device__ __forceinline__ static float dot(const uint32_t* row, const float* q, int D, int) {
    float acc = 0.f;
    for (int w = 0; w < D / 4; ++w) {
      const uint32_t v = row[w];
#pragma unroll
      for (int b = 0; b < 4; ++b) acc = fmaf(q[4 * w + b], fp8_to_f32((uint8_t)(v >> (8 * b))), acc);
    }
    return acc;
  }
};
// Block-scaled fp8 rows: d_c e4m3 codes, d_c / 128 fp32 scales, d_r bf16 (k_pe).
struct E4m3B128 {};
template <> struct PageElem<E4m3B128> {
  __device__ __forceinline__ static float get(const uint32_t* row, int k, int d_c) {
    return fp8_to_f32((uint8_t)(row[k >> 2] >> (8 * (k & 3)))) * __uint_as_float(row[(d_c >> 2) + (k >> 7)]);
  }
  __device__ __forceinline__ static float dot(const uint32_t* row, const float* q, int D, int d_c) {
    float acc = 0.f;
    for (int blk = 0; blk < d_c / 128; ++blk) {
      float part = 0.f;
      for (int w = 32 * blk; w < 32 * blk + 32; ++w) {
        const uint32_t v = row[w];
#pragma unroll
        for (int b = 0; b < 4; ++b) part = fmaf(q[4 * w + b], fp8_to_f32((uint8_t)(v >> (8 * b))), part);
      }
      acc = fmaf(part, __uint_as_float(row[(d_c >> 2) + blk]), acc);
    }
    const uint32_t* kr = row + (d_c >> 2) + (d_c >> 7);
    for (int w = 0; w < (D - d_c) / 2; ++w) {
      const uint32_t v = kr[w];
      acc = fmaf(q[d_c + 2 * w], __uint_as_float(v << 16), acc);
      acc = fmaf(q[d_c + 2 * w + 1], __uint_as_float(v & 0xFFFF0000u), acc);
    }
    return acc;
  }
};

constexpr int SIMT_HEADS = 8;

template <typename QT, typename CT, int VPL>
__global__ void __launch_bounds__(256) decode_simt_kernel(DecodeParams p) {
  extern __shared__ __align__(16) uint32_t smem_simt[];
  const int D = p.D, P = p.P;
  const int row_words = (int)((p.row_bytes + 3) / 4);
  const int stride = row_words | 1;
  uint32_t* page_s = smem_simt;                                   // [P][stride]
  float* q_s = reinterpret_cast<float*>(smem_simt + P * stride);   // [SIMT_HEADS][D]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * SIMT_HEADS + warp;
  const bool head_ok = h < p.H;
  const uint8_t* cache = reinterpret_cast<const uint8_t*>(p.cache);
  const QT* q_lat = reinterpret_cast<const QT*>(p.q_lat);
  const int it0 = p.worker_off[blockIdx.x], it1 = p.worker_off[blockIdx.x + 1];
  for (int it = it0; it < it1; ++it) {
    const WorkItem item = p.items[it];
    const int g = item.group, b = g / p.q_len;
    const int kv = p.group_kv[g];
    __syncthreads();
    for (int i = threadIdx.x; i < SIMT_HEADS * D; i += blockDim.x) {
      const int hh = blockIdx.y * SIMT_HEADS + i / D;
      q_s[i] = hh < p.H ? to_f32(q_lat[((long long)g * p.H + hh) * D + i % D]) : 0.f;
    }
    float m = -INFINITY, l = 0.f;
    float o[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) o[i] = 0.f;
    for (int pg = item.page_begin; pg < item.page_end; ++pg) {
      const int page_id = p.block_table[(long long)b * p.max_pages + pg];
      const bool page_ok = page_id >= 0 && page_id < p.num_pages;
      const int ntok = min(P, kv - pg * P);
      __syncthreads();
      if (page_ok) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(cache + (long long)page_id * P * p.row_bytes);
        for (int i = threadIdx.x; i < ntok * row_words; i += blockDim.x)
          page_s[(i / row_words) * stride + i % row_words] = src[i];
      } else if (threadIdx.x == 0) {
        flag_status(p.status, MLA_ERR_DEVICE_GUARD);
      }
      __syncthreads();
      if (!page_ok || !head_ok) continue;
      const float* qh = q_s + warp * D;
      float s0 = -INFINITY, s1 = -INFINITY;
      if (lane < ntok) s0 = PageElem<CT>::dot(page_s + lane * stride, qh, D, p.d_c) * p.scale_log2;
      if (lane + 32 < ntok) s1 = PageElem<CT>::dot(page_s + (lane + 32) * stride, qh, D, p.d_c) * p.scale_log2;
      const float m_new = fmaxf(m, warp_max(fmaxf(s0, s1)));
      const float alpha = exp2f(m - m_new);
      const float p0 = exp2f(s0 - m_new), p1 = exp2f(s1 - m_new);
      l = l * alpha + warp_sum(p0 + p1);
#pragma unroll
      for (int i = 0; i < VPL; ++i) o[i] *= alpha;
      for (int j = 0; j < ntok; ++j) {
        const float pj = __shfl_sync(0xffffffffu, (j < 32) ? p0 : p1, j & 31);
        const uint32_t* row = page_s + j * stride;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int k = lane + 32 * i;
          if (k < p.d_c) o[i] = fmaf(pj, PageElem<CT>::get(row, k, p.d_c), o[i]);
        }
      }
      m = m_new;
    }
    if (head_ok) {
      const float inv_l = (l > 0.f) ? p.out_scale / l : 0.f;
      const float lse_v = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
      if (item.single) {
        QT* out = reinterpret_cast<QT*>(p.out_latent) + ((long long)g * p.H + h) * p.d_c;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int k = lane + 32 * i;
          if (k < p.d_c) out[k] = from_f32<QT>(o[i] * inv_l);
        }
        if (lane == 0) p.lse[(long long)g * p.H + h] = lse_v;
      } else {
        float* out = p.part_o + ((long long)it * p.H + h) * p.d_c;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int k = lane + 32 * i;
          if (k < p.d_c) out[k] = o[i] * inv_l;
        }
        if (lane == 0) p.part_lse[(long long)it * p.H + h] = lse_v;
      }
    }
  }
}

// ======================================================================== LSE combine
// out = sum_s exp(lse_s - L) o_s with L = log sum_s exp(lse_s) over a group's items;
// groups with no item (empty requests) get out = 0, lse = -inf.
// One warp per (group, head): the warp merges the group's split partials over the d_c
// latent dims with 16-byte loads.
template <typename QT>
__global__ void __launch_bounds__(256) combine_kernel(DecodeParams p, int groups) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gh = (long long)blockIdx.x * 8 + warp;
  if (gh >= (long long)groups * p.H) return;
  const int g = (int)(gh / p.H), h = (int)(gh % p.H);
  const int first = p.group_first[g], last = p.group_last[g];
  const int n = (first >= 0 && last >= first) ? last - first + 1 : 0;
  QT* out = reinterpret_cast<QT*>(p.out_latent) + gh * p.d_c;
  if (n == 1) return;                          // written directly by the attention kernel
  float m = -INFINITY;
  for (int s = 0; s < n; ++s) m = fmaxf(m, p.part_lse[(long long)(first + s) * p.H + h]);
  if (n == 0 || m == -INFINITY) {
    for (int k = lane; k < p.d_c; k += 32) out[k] = from_f32<QT>(0.f);
    if (lane == 0) p.lse[gh] = -INFINITY;
    return;
  }
  float sum = 0.f;
  for (int s = 0; s < n; ++s) sum += expf(p.part_lse[(long long)(first + s) * p.H + h] - m);
  const float L = m + logf(sum);
  // weights of the first 8 splits kept in registers; any further split is streamed
  constexpr int kW = 8;
  float w[kW];
#pragma unroll
  for (int s = 0; s < kW; ++s)
    w[s] = (s < n) ? expf(p.part_lse[(long long)(first + s) * p.H + h] - L) : 0.f;
  const float* base = p.part_o + ((long long)first * p.H + h) * p.d_c;
  const long long stride = (long long)p.H * p.d_c;     // from one split slot to the next
  for (int k = 4 * lane; k < p.d_c; k += 128) {
    float4 v[kW];
#pragma unroll
    for (int s = 0; s < kW; ++s)
      v[s] = (s < n) ? *reinterpret_cast<const float4*>(base + s * stride + k) : make_float4(0, 0, 0, 0);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < kW; ++s) {
      acc.x = fmaf(w[s], v[s].x, acc.x);
      acc.y = fmaf(w[s], v[s].y, acc.y);
      acc.z = fmaf(w[s], v[s].z, acc.z);
      acc.w = fmaf(w[s], v[s].w, acc.w);
    }
    for (int s = kW; s < n; ++s) {
      const float ws = expf(p.part_lse[(long long)(first + s) * p.H + h] - L);
      const float4 x = *reinterpret_cast<const float4*>(base + s * stride + k);
      acc.x = fmaf(ws, x.x, acc.x);
      acc.y = fmaf(ws, x.y, acc.y);
      acc.z = fmaf(ws, x.z, acc.z);
      acc.w = fmaf(ws, x.w, acc.w);
    }
    out[k] = from_f32<QT>(acc.x);
    out[k + 1] = from_f32<QT>(acc.y);
    out[k + 2] = from_f32<QT>(acc.z);
    out[k + 3] = from_f32<QT>(acc.w);
  }
  if (lane == 0) p.lse[gh] = L;
}

// The same merge over octet-planar bf16 partials ([item][d_c / 8][H][8]): block (group,
// 16-dim slice), one thread per head; each split's slice is two coalesced 16-byte loads per
// thread and the merged slice one 32-byte store.
__global__ void __launch_bounds__(128) combine_planar_kernel(DecodeParams p) {
  ptx::griddep_wait();                         // the attention kernel's partials
  const int g = blockIdx.x, o0 = 2 * blockIdx.y, h = threadIdx.x;
  const int first = p.group_first[g], last = p.group_last[g];
  const int n = (first >= 0 && last >= first) ? last - first + 1 : 0;
  if (n == 1 || h >= p.H) return;              // single items are written by the attention kernel
  const long long gh = (long long)g * p.H + h;
  uint4* out = reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(p.out_latent) + gh * p.d_c + 8 * o0);
  if (n == 0) {
    out[0] = make_uint4(0u, 0u, 0u, 0u);
    out[1] = make_uint4(0u, 0u, 0u, 0u);
    if (blockIdx.y == 0) p.lse[gh] = -INFINITY;
    return;
  }
  const long long ostride = p.H, sstride = (long long)(p.d_c / 8) * p.H;
  const uint4* base = reinterpret_cast<const uint4*>(p.part_o) + (long long)first * sstride + (long long)o0 * ostride + h;
  const float* lse_p = p.part_lse + (long long)first * p.H + h;
  // up to kW splits with every load issued before any is used; further splits streamed
  constexpr int kW = 8;
  float ls[kW];
  uint4 va[kW], vb[kW];
#pragma unroll
  for (int s = 0; s < kW; ++s) {
    if (s < n) {
      ls[s] = lse_p[(long long)s * p.H];
      va[s] = base[s * sstride];
      vb[s] = base[s * sstride + ostride];
    }
  }
  float m = -INFINITY;
#pragma unroll
  for (int s = 0; s < kW; ++s)
    if (s < n) m = fmaxf(m, ls[s]);
  for (int s = kW; s < n; ++s) m = fmaxf(m, lse_p[(long long)s * p.H]);
  if (m == -INFINITY) {
    out[0] = make_uint4(0u, 0u, 0u, 0u);
    out[1] = make_uint4(0u, 0u, 0u, 0u);
    if (blockIdx.y == 0) p.lse[gh] = -INFINITY;
    return;
  }
  float wts[kW], sum = 0.f;
#pragma unroll
  for (int s = 0; s < kW; ++s) {
    wts[s] = (s < n) ? expf(ls[s] - m) : 0.f;
    sum += wts[s];
  }
  for (int s = kW; s < n; ++s) sum += expf(lse_p[(long long)s * p.H] - m);
  const float inv = 1.f / sum;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  auto accumulate = [&](float w, const uint4& v0, const uint4& v1) {
    const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[i]));
      acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
      acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
    }
  };
#pragma unroll
  for (int s = 0; s < kW; ++s)
    if (s < n) accumulate(wts[s] * inv, va[s], vb[s]);
  for (int s = kW; s < n; ++s)
    accumulate(expf(lse_p[(long long)s * p.H] - m) * inv, base[s * sstride], base[s * sstride + ostride]);
  uint32_t pk[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  out[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  out[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  if (blockIdx.y == 0) p.lse[gh] = m + logf(sum);
}

template <typename T>
__global__ void f32_to_act_kernel(const float* __restrict__ src, T* __restrict__ dst, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = from_f32<T>(src[i]);
}

// ======================================================================== launchers
cudaError_t launch_plan(const PlanParams& p, cudaStream_t s) {
  const size_t smem = (size_t)(4 * (p.batch * p.q_len + 1) + 3 * (p.workers + 1) + 32) * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  plan_kernel<<<1, 256, smem, s>>>(p);
  note_launch();
  return cudaGetLastError();
}

template <typename T>
static cudaError_t query_prologue_t(const void* q_nope, const void* q_pe, const void* W_UK_abs,
                                    const int32_t* seq_lens, int batch, int q_len, int H, int d_n,
                                    int d_c, int d_r, const RopeTable& rt, void* q_lat,
                                    cudaStream_t s) {
  const int groups = batch * q_len, D = d_c + d_r;
  StoreEpi<T> epi{reinterpret_cast<T*>(q_lat), (long long)H * D, (long long)D};
  // per head h: q_lat[g][h][0:d_c] = q_nope[g][h][:] . W_UK_abs[h]
  cudaError_t e = simt_gemm(reinterpret_cast<const T*>(q_nope), (long long)H * d_n, (long long)d_n,
                            reinterpret_cast<const T*>(W_UK_abs), (long long)d_c,
                            (long long)d_n * d_c, groups, d_c, d_n, H, 1, epi, s);
  if (e != cudaSuccess) return e;
  if (groups > 0) {
    q_rope_kernel<T><<<dim3(groups, (H + 15) / 16), 256, 0, s>>>(reinterpret_cast<const T*>(q_pe), seq_lens, batch, q_len,
                                           H, d_c, d_r, rt, 1.f, 0, reinterpret_cast<T*>(q_lat));
    note_launch();
  }
  return cudaGetLastError();
}

cudaError_t launch_prep(const PlanParams& pp, const void* q_pe, const int32_t* seq_lens, int q_len,
                        int H, int d_c, int d_r, const RopeTable& rt, float q_scale, int planar,
                        int f16, void* q_lat, cudaStream_t s) {
  const int groups = pp.batch * q_len;
  const int hblocks = (H + 15) / 16;
  const bool plan = pp.workers > 0;
  const size_t smem = plan ? plan_smem_bytes(groups, pp.workers) : 0;
  auto kern = prep_kernel<bf16>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((plan ? 1 : 0) + groups * hblocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = plan ? 0 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, pp, reinterpret_cast<const bf16*>(q_pe), seq_lens, q_len,
                                     H, d_c, d_r, rt, q_scale, planar, reinterpret_cast<bf16*>(q_lat),
                                     hblocks, f16);
  note_launch();
  return e;
}

cudaError_t launch_q_rope(mla_dtype act, const void* q_pe, const int32_t* seq_lens, int batch,
                          int q_len, int H, int d_c, int d_r, const RopeTable& rt, float q_scale,
                          int planar, void* q_lat, cudaStream_t s) {
  const int groups = batch * q_len;
  if (groups <= 0) return cudaSuccess;
  const dim3 blocks(groups, (H + 15) / 16);
  if (act == MLA_F32)
    q_rope_kernel<float><<<blocks, 256, 0, s>>>(reinterpret_cast<const float*>(q_pe), seq_lens, batch,
                                               q_len, H, d_c, d_r, rt, q_scale, planar, reinterpret_cast<float*>(q_lat));
  else
    q_rope_kernel<bf16><<<blocks, 256, 0, s>>>(reinterpret_cast<const bf16*>(q_pe), seq_lens, batch,
                                              q_len, H, d_c, d_r, rt, q_scale, planar, reinterpret_cast<bf16*>(q_lat));
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_query_prologue(mla_dtype act, const void* q_nope, const void* q_pe,
                                  const void* W_UK_abs, const int32_t* seq_lens, int batch,
                                  int q_len, int H, int d_n, int d_c, int d_r,
                                  const RopeTable& rt, void* q_lat, cudaStream_t s) {
  if (act == MLA_F32)
    return query_prologue_t<float>(q_nope, q_pe, W_UK_abs, seq_lens, batch, q_len, H, d_n, d_c,
                                   d_r, rt, q_lat, s);
  return query_prologue_t<bf16>(q_nope, q_pe, W_UK_abs, seq_lens, batch, q_len, H, d_n, d_c, d_r,
                                rt, q_lat, s);
}

template <typename QT, typename CT, int VPL>
static cudaError_t decode_simt_t(const DecodeParams& p, cudaStream_t s) {
  const int row_words = (int)((p.row_bytes + 3) / 4);
  const int stride = row_words | 1;
  const size_t smem = (size_t)p.P * stride * 4 + (size_t)SIMT_HEADS * p.D * 4;
  auto kern = decode_simt_kernel<QT, CT, VPL>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(p.workers, (p.H + SIMT_HEADS - 1) / SIMT_HEADS);
  kern<<<grid, 256, smem, s>>>(p);
  note_launch();
  return cudaGetLastError();
}

template <typename QT, typename CT>
static cudaError_t decode_simt_vpl(const DecodeParams& p, cudaStream_t s) {
  const int vpl = (p.d_c + 31) / 32;
  if (vpl <= 2) return decode_simt_t<QT, CT, 2>(p, s);
  if (vpl <= 4) return decode_simt_t<QT, CT, 4>(p, s);
  if (vpl <= 8) return decode_simt_t<QT, CT, 8>(p, s);
  return decode_simt_t<QT, CT, 16>(p, s);
}

cudaError_t launch_decode_simt(mla_dtype act, mla_dtype cache, const DecodeParams& p,
                               cudaStream_t s) {
  if (act == MLA_F32) return decode_simt_vpl<float, float>(p, s);
  if (cache == MLA_BF16) return decode_simt_vpl<bf16, bf16>(p, s);
  if (cache == MLA_FP8_E4M3_B128) return decode_simt_vpl<bf16, E4m3B128>(p, s);
  return decode_simt_vpl<bf16, uint8_t>(p, s);
}

cudaError_t launch_combine(mla_dtype act, const DecodeParams& p, int groups, cudaStream_t s) {
  if (groups <= 0) return cudaSuccess;
  if (p.part_planar) {
    if (act != MLA_BF16 || p.H > 128 || p.d_c % 16) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(groups, p.d_c / 16, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, combine_planar_kernel, p);
    note_launch();
    return e;
  }
  const int blocks = (int)(((long long)groups * p.H + 7) / 8);
  if (act == MLA_F32) combine_kernel<float><<<blocks, 256, 0, s>>>(p, groups);
  else combine_kernel<bf16><<<blocks, 256, 0, s>>>(p, groups);
  note_launch();
  return cudaGetLastError();
}

template <typename AT, typename CT>
static cudaError_t append_latent_t(const void* c_kv, const void* k_pe, int T,
                                   const int32_t* req_ids, const int32_t* positions,
                                   const int32_t* block_table, int batch, int max_pages,
                                   void* cache_ptr, int num_pages, int P, int d_c, int d_r,
                                   int rotate, const RopeTable& rt, float cache_scale,
                                   int32_t* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  append_latent_kernel<AT, CT><<<T, 128, 0, s>>>(
      reinterpret_cast<const AT*>(c_kv), reinterpret_cast<const AT*>(k_pe), (long long)d_c,
      (long long)d_r, req_ids, positions,
      block_table, batch, max_pages, reinterpret_cast<CT*>(cache_ptr), num_pages, P, d_c, d_r,
      rotate, rt, cache_scale, status);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_append_latent(mla_dtype act, mla_dtype cache, const void* c_kv,
                                 const void* k_pe, int T, const int32_t* req_ids,
                                 const int32_t* positions, const int32_t* block_table, int batch,
                                 int max_pages, void* cache_ptr, int num_pages, int P, int d_c,
                                 int d_r, int rotate, const RopeTable& rt, float cache_scale,
                                 int32_t* status, cudaStream_t s) {
  if (act == MLA_F32)
    return append_latent_t<float, float>(c_kv, k_pe, T, req_ids, positions, block_table, batch,
                                         max_pages, cache_ptr, num_pages, P, d_c, d_r, rotate, rt,
                                         cache_scale, status, s);
  if (cache == MLA_FP8_E4M3_B128) {
    if (T <= 0) return cudaSuccess;
    append_latent_b128_kernel<bf16><<<T, 128, 0, s>>>(
        reinterpret_cast<const bf16*>(c_kv), reinterpret_cast<const bf16*>(k_pe), (long long)d_c,
        (long long)d_r, req_ids, positions, block_table, batch, max_pages,
        reinterpret_cast<uint8_t*>(cache_ptr), num_pages, P, d_c, d_r, rotate, rt, status);
    note_launch();
    return cudaGetLastError();
  }
  if (cache == MLA_BF16)
    return append_latent_t<bf16, bf16>(c_kv, k_pe, T, req_ids, positions, block_table, batch,
                                       max_pages, cache_ptr, num_pages, P, d_c, d_r, rotate, rt,
                                       cache_scale, status, s);
  return append_latent_t<bf16, uint8_t>(c_kv, k_pe, T, req_ids, positions, block_table, batch,
                                        max_pages, cache_ptr, num_pages, P, d_c, d_r, rotate, rt,
                                        cache_scale, status, s);
}

template <typename AT, typename CT>
static cudaError_t append_from_h_t(const void* h, const void* W, int T, int d,
                                   const int32_t* req_ids, const int32_t* positions,
                                   const int32_t* block_table, int batch, int max_pages,
                                   void* cache_ptr, int num_pages, int P, int d_c, int d_r,
                                   const RopeTable& rt, float cache_scale, int32_t* status,
                                   cudaStream_t s) {
  AppendEpi<CT> epi{req_ids, positions, block_table, batch, max_pages, num_pages, P, d_c, d_r,
                    reinterpret_cast<CT*>(cache_ptr), rt, cache_scale, status};
  const int D = d_c + d_r;
  return simt_gemm(reinterpret_cast<const AT*>(h), (long long)d, 0LL,
                   reinterpret_cast<const AT*>(W), (long long)D, 0LL, T, D, d, 1, 1, epi, s);
}

cudaError_t launch_append_from_h(mla_dtype act, mla_dtype cache, const void* h, const void* W,
                                 int T, int d, const int32_t* req_ids, const int32_t* positions,
                                 const int32_t* block_table, int batch, int max_pages,
                                 void* cache_ptr, int num_pages, int P, int d_c, int d_r,
                                 const RopeTable& rt, float cache_scale, int32_t* status,
                                 cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (act == MLA_F32)
    return append_from_h_t<float, float>(h, W, T, d, req_ids, positions, block_table, batch,
                                         max_pages, cache_ptr, num_pages, P, d_c, d_r, rt,
                                         cache_scale, status, s);
  if (cache == MLA_BF16)
    return append_from_h_t<bf16, bf16>(h, W, T, d, req_ids, positions, block_table, batch,
                                       max_pages, cache_ptr, num_pages, P, d_c, d_r, rt,
                                       cache_scale, status, s);
  return append_from_h_t<bf16, uint8_t>(h, W, T, d, req_ids, positions, block_table, batch,
                                        max_pages, cache_ptr, num_pages, P, d_c, d_r, rt,
                                        cache_scale, status, s);
}

template <typename T>
static cudaError_t absorb_t(const void* W_UK, const void* W_UV, const void* W_O, void* W_UK_abs,
                           void* W_comb, int H, int d_c, int d_n, int d_v, int d, cudaStream_t s) {
  const long long n = (long long)H * d_n * d_c;
  transpose_heads_kernel<T><<<(int)min((n + 255) / 256, 8192LL), 256, 0, s>>>(
      reinterpret_cast<const T*>(W_UK), reinterpret_cast<T*>(W_UK_abs), H, d_c, d_n);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // block i of W_comb = W_UV[:, i*d_v:(i+1)*d_v] . W_O[i*d_v:(i+1)*d_v, :]; bf16 on the
  // tensor cores where the tensor maps' 16-byte row strides allow
  if (sizeof(T) == 2 && d % 8 == 0 && d_v % 8 == 0)
    return launch_fold_tc(W_UV, W_O, H, d_c, d_v, d, W_comb, nullptr, s);
  StoreEpi<T> epi{reinterpret_cast<T*>(W_comb), (long long)d, (long long)d_c * d};
  return simt_gemm(reinterpret_cast<const T*>(W_UV), (long long)H * d_v, (long long)d_v,
                   reinterpret_cast<const T*>(W_O), (long long)d, (long long)d_v * d, d_c, d, d_v,
                   H, 1, epi, s);
}

cudaError_t launch_absorb(mla_dtype act, const void* W_UK, const void* W_UV, const void* W_O,
                          void* W_UK_abs, void* W_comb, int H, int d_c, int d_n, int d_v, int d,
                          cudaStream_t s) {
  if (act == MLA_F32) return absorb_t<float>(W_UK, W_UV, W_O, W_UK_abs, W_comb, H, d_c, d_n, d_v, d, s);
  return absorb_t<bf16>(W_UK, W_UV, W_O, W_UK_abs, W_comb, H, d_c, d_n, d_v, d, s);
}

// out = o_lat . W_comb with split-K partial sums accumulated in fp32 in `acc`
// ([rows][N], zeroed here), then converted to the activation dtype.
template <typename T>
static cudaError_t output_proj_t(const void* o_lat, const void* W_comb, int rows, int K, int N,
                                 void* out, float* acc, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(acc, 0, (size_t)rows * N * sizeof(float), s);
  if (e != cudaSuccess) return e;
  // a split per 128 of K (at most 64): with a handful of rows the grid is otherwise a few
  // blocks each walking all of K
  const int splits = max(1, min(64, K / 128));
  AtomicAddEpi epi{acc, (long long)N};
  e = simt_gemm(reinterpret_cast<const T*>(o_lat), (long long)K, 0LL,
                reinterpret_cast<const T*>(W_comb), (long long)N, 0LL, rows, N, K, 1, splits, epi, s);
  if (e != cudaSuccess) return e;
  const long long n = (long long)rows * N;
  f32_to_act_kernel<T><<<(int)min((n + 255) / 256, 4096LL), 256, 0, s>>>(acc, reinterpret_cast<T*>(out), n);
  note_launch();
  return cudaGetLastError();
}

// u[r][h][0:d_v] = o_lat[r][h][:] . W_UV[:, h d_v : (h + 1) d_v], one batch entry per head.
template <typename T>
static cudaError_t lift_t(const void* o_lat, const void* W_UV, int rows, int H, int d_c, int d_v,
                          void* u, cudaStream_t s) {
  StoreEpi<T> epi{reinterpret_cast<T*>(u), (long long)H * d_v, (long long)d_v};
  return simt_gemm(reinterpret_cast<const T*>(o_lat), (long long)H * d_c, (long long)d_c,
                   reinterpret_cast<const T*>(W_UV), (long long)H * d_v, (long long)d_v, rows, d_v,
                   d_c, H, 1, epi, s);
}

cudaError_t launch_lift_simt(mla_dtype act, const void* o_lat, const void* W_UV, int rows, int H,
                             int d_c, int d_v, void* u, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (act == MLA_F32) return lift_t<float>(o_lat, W_UV, rows, H, d_c, d_v, u, s);
  return lift_t<bf16>(o_lat, W_UV, rows, H, d_c, d_v, u, s);
}

cudaError_t launch_output_proj_simt_ws(mla_dtype act, const void* o_lat, const void* W_comb,
                                       int rows, int K, int N, void* out, float* acc,
                                       cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (act == MLA_F32) return output_proj_t<float>(o_lat, W_comb, rows, K, N, out, acc, s);
  return output_proj_t<bf16>(o_lat, W_comb, rows, K, N, out, acc, s);
}

}  // namespace mla
