// The decode prologue's small jobs, shared by the kernels that run them: the split planner
// (the fp32 path's plan_kernel, the bf16 path's prep kernel or extra blocks of the query
// absorption GEMM) and the q_pe rotation.
#pragma once
#include "internal.h"

namespace mla {

// Shared memory plan_body needs for `groups` groups and `workers` workers.
inline size_t plan_smem_bytes(int groups, int workers) {
  return (size_t)(4 * (groups + 1) + 3 * (workers + 1) + 32) * sizeof(int);
}

// In-place inclusive prefix sum of a[0..n) in shared memory by one block.
__device__ inline void block_inclusive_scan(int* a, int n, int* warp_tot) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int per = (n + nt - 1) / nt;
  const int b0 = min(n, tid * per), b1 = min(n, b0 + per);
  int run = 0;
  for (int i = b0; i < b1; ++i) {
    run += a[i];
    a[i] = run;
  }
  // exclusive scan of the per-thread totals
  const int lane = tid & 31, wid = tid >> 5;
  int x = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = (lane < (nt + 31) / 32) ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_tot[lane] = w;
  }
  __syncthreads();
  const int offset = x - run + (wid > 0 ? warp_tot[wid - 1] : 0);
  for (int i = b0; i < b1; ++i) a[i] += offset;
  __syncthreads();
}

// The flattened sequence of all groups' key pages is cut into `workers` ranges of equal
// cost, where a work item costs its pages plus kItemCost start-up units (its query load
// into tensor memory and its epilogue). Measured on the tensor-core path at batch 32 x 4096,
// a worker's finishing time grows by about 1.3 us per page and 2.8 us per extra item, and 2
// units balanced the workers best (3 made the decode 0.5 us slower); worker w processes its
// range as one work item per group it touches. An item that
// covers a whole group writes the final output, the others write partials merged by the
// combine kernel.
//
// Every step is data-parallel with O(1) work per thread (the plan runs on the decode's
// critical path, where serial per-thread chains cost microseconds): per group the
// prefix sums of pages, cost and non-empty groups; each group places the cost cuts that
// fall inside it; each worker reads its item count from the non-empty prefix.
#ifndef MLA_ITEM_COST
#define MLA_ITEM_COST 2
#endif
constexpr int kItemCost = MLA_ITEM_COST;

// Largest g in [0, n) with a[g] <= x (a non-decreasing, a[0] = 0 <= x < a[n]).
__device__ __forceinline__ int last_at_most(const int* a, int n, long long x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ inline void plan_body(const PlanParams& p, int* sm, bool reset_status) {
  const int groups = p.batch * p.q_len, W = p.workers;
  int* cu = sm;                             // [groups + 1] page prefix
  int* vcu = cu + groups + 1;               // [groups + 1] cost prefix
  int* nz = vcu + groups + 1;               // [groups + 1] non-empty group prefix
  int* cutp = nz + groups + 1;              // [W + 1] page position of cut k
  int* cutg = cutp + W + 1;                 // [W + 1] group holding cut k
  int* wc = cutg + W + 1;                   // [W + 1] item prefix
  int* warp_tot = wc + W + 1;               // [32]
  int* kvs = warp_tot + 32;                 // [groups] keys per group
  const int tid = threadIdx.x, nt = blockDim.x;
  // each decode call reports its own status: clear the word before anything can flag it
  if (reset_status) {
    if (tid == 0) *p.status = 0;
    __syncthreads();
  }
  for (int g = tid; g < groups; g += nt) {
    const int b = g / p.q_len, t = g % p.q_len;
    const int S = p.seq_lens[b];
    int kv = 0;
    if (S != 0) {
      if (S < p.q_len || (long long)S > (long long)p.max_pages * p.page_size) {
        if (t == 0) flag_status(p.status, MLA_ERR_DEVICE_GUARD);
      } else {
        kv = S - p.q_len + t + 1;
      }
    }
    p.group_kv[g] = kv;
    kvs[g] = kv;
    p.group_first[g] = -1;
    p.group_last[g] = -2;
    const int pages = (kv + p.page_size - 1) / p.page_size;
    cu[g + 1] = pages;
    vcu[g + 1] = pages > 0 ? pages + kItemCost : 0;
    nz[g + 1] = pages > 0 ? 1 : 0;
  }
  if (tid == 0) {
    cu[0] = 0;
    vcu[0] = 0;
    nz[0] = 0;
    wc[0] = 0;
  }
  __syncthreads();
  block_inclusive_scan(cu + 1, groups, warp_tot);
  block_inclusive_scan(vcu + 1, groups, warp_tot);
  block_inclusive_scan(nz + 1, groups, warp_tot);
  // cut k sits at cost floor(V k / W), inside the (non-empty) group g with
  // vcu[g] <= cut < vcu[g + 1]; a cut inside a group's start-up units falls on its first page
  const long long V = vcu[groups];
  for (int k = tid; k <= W; k += nt) {
    if (k == W || V == 0) {
      cutp[k] = k == W ? cu[groups] : 0;
      cutg[k] = groups;
      continue;
    }
    const long long c = V * k / W;
    const int g = last_at_most(vcu, groups, c);
    const long long o = c - vcu[g] - kItemCost;
    cutp[k] = cu[g] + (int)(o < 0 ? 0 : o);
    cutg[k] = g;
  }
  __syncthreads();
  // worker w: pages [cutp[w], cutp[w + 1]), one item per non-empty group from cutg[w] to the
  // group of its last page
  auto last_group_end = [&](int w) {       // one past the group of page cutp[w + 1] - 1
    const int g1 = cutg[w + 1];
    return (g1 < groups && cutp[w + 1] > cu[g1]) ? g1 + 1 : g1;
  };
  for (int w = tid; w < W; w += nt)
    wc[w + 1] = cutp[w + 1] > cutp[w] ? nz[last_group_end(w)] - nz[cutg[w]] : 0;
  __syncthreads();
  block_inclusive_scan(wc + 1, W, warp_tot);
  for (int w = tid; w <= W; w += nt) p.worker_off[w] = wc[w];
  for (int w = tid; w < W; w += nt) {
    const int lo = cutp[w], hi = cutp[w + 1];
    if (hi <= lo) continue;
    const int g0 = cutg[w], g1 = last_group_end(w);
    for (int g = g0; g < g1; ++g) {
      const int a = cu[g], e = cu[g + 1];
      if (e == a) continue;
      const int idx = wc[w] + nz[g] - nz[g0];
      const int pb = max(lo, a) - a, pe = min(hi, e) - a;
      WorkItem it;
      it.group = g;
      it.page_begin = pb;
      it.page_end = pe;
      it.single = (pb == 0 && pe == e - a);
      it.kv = kvs[g];
      p.items[idx] = it;
      if (pb == 0) p.group_first[g] = idx;
      if (pe == e - a) p.group_last[g] = idx;
    }
  }
}

// One block per (group, hpb heads): the d_r/2 rotation angles of the group's position are
// computed once into shared memory, then applied to those heads' q_pe.
// A rotated query value as stored in q_lat: the activation type, or (f16 set, bf16
// activations) the bits of an f16.
template <typename T>
__device__ __forceinline__ T q_out(float v, int f16) {
  if constexpr (sizeof(T) == 2) {
    if (f16) return __ushort_as_bfloat16(__half_as_ushort(__float2half_rn(v)));
  }
  return from_f32<T>(v);
}

template <typename T>
__device__ __forceinline__ void rope_body(const T* __restrict__ q_pe, const int32_t* seq_lens,
                                          int q_len, int H, int d_c, int d_r, const RopeTable& rt,
                                          float qs, int planar, T* __restrict__ q_lat, int g, int hy,
                                          int hpb = 16, int f16 = 0) {
  __shared__ float cs[kMaxRopePairs], sn[kMaxRopePairs];
  const int h0 = hy * hpb, h1 = min(H, h0 + hpb);
  const int b = g / q_len, t = g % q_len;
  const int pos = seq_lens[b] - q_len + t;
  const int pairs = d_r / 2;
  if (threadIdx.x < pairs) {
    float s_ = 0.f, c_ = 0.f;
    if (pos >= 0) rope_sincos(rt, threadIdx.x, pos, &s_, &c_);
    sn[threadIdx.x] = s_;
    cs[threadIdx.x] = c_;
  }
  __syncthreads();
  const int D = d_c + d_r;
  for (int i = threadIdx.x; i < (h1 - h0) * pairs; i += blockDim.x) {
    const int h = h0 + i / pairs, k = i % pairs;
    const long long gh = (long long)g * H + h;
    const float x0 = to_f32(q_pe[gh * d_r + 2 * k]);
    const float x1 = to_f32(q_pe[gh * d_r + 2 * k + 1]);
    float y0 = 0.f, y1 = 0.f;
    if (pos >= 0) {
      y0 = (x0 * cs[k] - x1 * sn[k]) * qs;
      y1 = (x0 * sn[k] + x1 * cs[k]) * qs;
    }
    const long long o = planar ? (long long)g * H * D + (long long)d_c * H + (long long)h * d_r + 2 * k
                               : gh * D + d_c + 2 * k;
    q_lat[o] = q_out<T>(y0, f16);
    q_lat[o + 1] = q_out<T>(y1, f16);
  }
}

// The same for bf16 with d_r a multiple of 16, eight pairs per thread and item: each item's
// two 16-byte loads are issued before the angles are computed, and its result is written
// with two 16-byte stores (every head's rope part is a 16-byte aligned contiguous run in
// both query layouts).
__device__ __forceinline__ void rope_body_bf16x8(const bf16* __restrict__ q_pe, const int32_t* seq_lens,
                                                 int q_len, int H, int d_c, int d_r, const RopeTable& rt,
                                                 float qs, int planar, bf16* __restrict__ q_lat, int g,
                                                 int hy, int hpb, int f16) {
  __shared__ float cs[kMaxRopePairs], sn[kMaxRopePairs];
  const int h0 = hy * hpb, h1 = min(H, h0 + hpb);
  const int chunks = d_r / 16;
  const int items = (h1 - h0) * chunks;
  const int D = d_c + d_r;
  auto src = [&](int i) {
    const long long gh = (long long)g * H + h0 + i / chunks;
    return reinterpret_cast<const uint4*>(q_pe + gh * d_r + 16 * (i % chunks));
  };
  uint4 a0 = make_uint4(0u, 0u, 0u, 0u), a1 = a0;
  if ((int)threadIdx.x < items) {
    a0 = src(threadIdx.x)[0];
    a1 = src(threadIdx.x)[1];
  }
  const int b = g / q_len, t = g % q_len;
  const int pos = seq_lens[b] - q_len + t;
  if ((int)threadIdx.x < d_r / 2) {
    float s_ = 0.f, c_ = 0.f;
    if (pos >= 0) rope_sincos(rt, threadIdx.x, pos, &s_, &c_);
    sn[threadIdx.x] = s_;
    cs[threadIdx.x] = c_;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < items; i += blockDim.x) {
    if (i != (int)threadIdx.x) {
      a0 = src(i)[0];
      a1 = src(i)[1];
    }
    const int h = h0 + i / chunks, c = i % chunks;
    const uint32_t in[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    uint32_t out[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = 8 * c + j;
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&in[j]));
      float y0 = 0.f, y1 = 0.f;
      if (pos >= 0) {
        y0 = (x.x * cs[k] - x.y * sn[k]) * qs;
        y1 = (x.x * sn[k] + x.y * cs[k]) * qs;
      }
      if (f16) {
        const __half2 yh = __floats2half2_rn(y0, y1);
        out[j] = *reinterpret_cast<const uint32_t*>(&yh);
      } else {
        const __nv_bfloat162 yb = __floats2bfloat162_rn(y0, y1);
        out[j] = *reinterpret_cast<const uint32_t*>(&yb);
      }
    }
    const long long gh = (long long)g * H + h;
    const long long o = planar ? (long long)g * H * D + (long long)d_c * H + (long long)h * d_r + 16 * c
                               : gh * D + d_c + 16 * c;
    uint4* dst = reinterpret_cast<uint4*>(q_lat + o);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
}

// One rotation job: q_pe of `groups` groups into the rotated part of q_lat, one block per
// (group, 32 heads).
struct RopeJob {
  const bf16* q_pe;
  const int32_t* seq_lens;
  bf16* q_lat;
  int groups, q_len, H, d_c, d_r, planar, hblocks;
  int f16;     // store the rotated query as f16 (the tensor-core kernel on an e4m3 cache)
  float qs;
  RopeTable rt;
};

}  // namespace mla
