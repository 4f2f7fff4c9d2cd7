// Internal launch interface between the C-ABI layer (mla_api.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/mla.h"
#include "common.cuh"

namespace mla {

// One decode "group" is one (request, query token) pair: 128 heads attending over the
// request's keys 0..p_t. A work item is a contiguous page range of one group.
struct WorkItem {
  int group;
  int page_begin;   // group-relative page index
  int page_end;
  int single;       // 1: the item covers the whole group -> write the final output
  int kv;           // keys the group attends to (its last page holds kv - 64 * (pages - 1))
};

// Byte offsets of every region of the decode workspace (all 256-byte aligned).
struct DecodeWorkspace {
  size_t status;        // int32 status word (+ padding)
  size_t worker_off;    // int32 [G + 1]
  size_t items;         // WorkItem [G + groups]
  size_t group_first;   // int32 [groups]
  size_t group_last;    // int32 [groups]
  size_t group_kv;      // int32 [groups]
  size_t q_lat;         // act dtype [groups][H][D]
  size_t part_o;        // fp32 [G + groups][H][d_c]
  size_t part_lse;      // fp32 [G + groups][H]
  size_t total;
  int workers;          // G
  int groups;           // batch * q_len
  int max_items;        // G + groups
};

struct PlanParams {
  const int32_t* seq_lens;
  int batch, q_len, page_size, max_pages, workers;
  int* worker_off;
  WorkItem* items;
  int* group_first;
  int* group_last;
  int* group_kv;
  int32_t* status;
};

struct DecodeParams {
  const void* q_lat;          // [groups][H][D]
  const void* cache;          // [num_pages][P][D]
  const int32_t* block_table;
  int max_pages, num_pages;
  int batch, q_len;
  int H, d_c, d_r, D, P;
  long long row_bytes;        // bytes of one cache row (token)
  float scale_log2;           // softmax_scale * log2(e) (* cache_scale for fp8)
  float out_scale;            // cache_scale for an fp8 cache, else 1
  void* out_latent;           // [groups][H][d_c] act dtype
  float* lse;                 // [groups][H]
  const int* worker_off;
  const WorkItem* items;
  const int* group_first;
  const int* group_last;
  const int* group_kv;
  float* part_o;              // split partials; layout set by part_planar
  float* part_lse;            // [items][H]
  int32_t* status;
  int workers;
  // tensor-core kernel: the limit of every barrier wait, in ns, and the testing hook that
  // withholds page withhold_page - 1 of worker 0 (0 = off)
  unsigned long long wait_limit_ns;
  int withhold_page;
  // 0: part_o is fp32 [items][H][d_c]; 1: bf16 [items][d_c / 8][H][8] (eight latent dims of
  // every head contiguous, so a warp of consecutive heads writes one 512-byte run)
  int part_planar;
};

// Counts kernels launched through the library (read by mla_kernel_launches).
void note_launch(int n = 1);

// ---- launchers (return cudaGetLastError() of the launch) --------------------------------
cudaError_t launch_plan(const PlanParams& p, cudaStream_t s);

cudaError_t launch_query_prologue(mla_dtype act, const void* q_nope, const void* q_pe,
                                  const void* W_UK_abs, const int32_t* seq_lens, int batch,
                                  int q_len, int H, int d_n, int d_c, int d_r,
                                  const RopeTable& rt, void* q_lat, cudaStream_t s);

cudaError_t launch_decode_simt(mla_dtype act, mla_dtype cache, const DecodeParams& p,
                               cudaStream_t s);

cudaError_t launch_combine(mla_dtype act, const DecodeParams& p, int groups, cudaStream_t s);

cudaError_t launch_append_latent(mla_dtype act, mla_dtype cache, const void* c_kv,
                                 const void* k_pe, int T, const int32_t* req_ids,
                                 const int32_t* positions, const int32_t* block_table, int batch,
                                 int max_pages, void* cache_ptr, int num_pages, int P, int d_c,
                                 int d_r, int rotate, const RopeTable& rt, float cache_scale,
                                 int32_t* status, cudaStream_t s);

cudaError_t launch_append_from_h(mla_dtype act, mla_dtype cache, const void* h, const void* W,
                                 int T, int d, const int32_t* req_ids, const int32_t* positions,
                                 const int32_t* block_table, int batch, int max_pages,
                                 void* cache_ptr, int num_pages, int P, int d_c, int d_r,
                                 const RopeTable& rt, float cache_scale, int32_t* status,
                                 cudaStream_t s);

cudaError_t launch_absorb(mla_dtype act, const void* W_UK, const void* W_UV, const void* W_O,
                          void* W_UK_abs, void* W_comb, int H, int d_c, int d_n, int d_v, int d,
                          cudaStream_t s);

// Tensor-core GEMMs (bf16 in, fp32 accumulate), gemm_tc.cu.
// out[rows][N] = x[rows][K] . W[K][N] through the cluster split-K GEMM (bf16, fp32 sums).
cudaError_t launch_output_proj_tc(const void* x, const void* W, int rows, int K, int N, void* out,
                                  int32_t* status, cudaStream_t s);
// out_a = x . W_a and out_b = x . W_b (same tokens, two weights) in one launch (bf16).
cudaError_t launch_two_proj_tc(const void* x, const void* W_a, const void* W_b, int rows, int K,
                               int N_a, int N_b, void* out_a, void* out_b, int32_t* status,
                               cudaStream_t s);
// The one-time fold W_comb[h] = W_UV[:, h] . W_O[h] on the tensor cores (bf16).
cudaError_t launch_fold_tc(const void* W_UV, const void* W_O, int H, int d_c, int d_v, int d,
                           void* W_comb, int32_t* status, cudaStream_t s);
// q_scale multiplies the query before its bf16 rounding (1, or the softmax scale times
// log2(e) for the tensor-core attention, which then works in log2 units).
// Query layouts in the workspace, per group of H heads (H * D elements each):
//   row-major (planar = 0): [H][D], the latent part then the rotated k_pe part of each head;
//   planar (planar = 1, tensor-core attention): the latent part as [d_c / 8][H][8] (eight
//   dims of every head contiguous, so that a warp of consecutive heads reads 512 contiguous
//   bytes), then the rotated part as [H][d_r].
// plan / rope: if non-null, extra blocks of the GEMM run the split planner (which clears the
// status word) and the q_pe rotation, and the GEMM is the decode's first kernel; if null,
// the GEMM follows the prep kernel (which did both) with programmatic serialization.
struct RopeJob;
// f16: the query is stored as f16 instead of bf16 (the tensor-core kernel on a per-tensor
// e4m3 cache, whose MMAs take f16 operands).
cudaError_t launch_query_absorb_tc(const void* q_nope, const void* W_UK_abs, int groups, int H,
                                   int d_n, int d_c, int D, float q_scale, int planar, int f16,
                                   void* q_lat, int32_t* status, const PlanParams* plan,
                                   const RopeJob* rope, cudaStream_t s);
// Append from h in one launch: projection, RoPE, encoding and page scatter (bf16 h and W).
cudaError_t launch_append_tc(mla_dtype cache_dtype, const void* h, const void* W, int T, int d,
                             int d_c, int d_r, const int32_t* req_ids, const int32_t* positions,
                             const int32_t* block_table, int batch, int max_pages, void* cache,
                             int num_pages, int P, const RopeTable& rt, float cache_scale,
                             int32_t* status, cudaStream_t s);
// q_pe rotation in one bf16 launch, plus (if pp.workers > 0) the status reset and the
// planner in block 0, then as the decode's first kernel; without the planner it follows the
// query absorption GEMM (which planned) with programmatic serialization.
cudaError_t launch_prep(const PlanParams& pp, const void* q_pe, const int32_t* seq_lens, int q_len,
                        int H, int d_c, int d_r, const RopeTable& rt, float q_scale, int planar,
                        int f16, void* q_lat, cudaStream_t s);
cudaError_t launch_q_rope(mla_dtype act, const void* q_pe, const int32_t* seq_lens, int batch,
                          int q_len, int H, int d_c, int d_r, const RopeTable& rt, float q_scale,
                          int planar, void* q_lat, cudaStream_t s);

// u[r][h][:] = o_lat[r][h][:] . W_i^UV (the latent output lifted to the value width):
// tensor-core GEMM for bf16 (d_c and d_v multiples of 64), SIMT GEMM otherwise.
cudaError_t launch_lift_tc(const void* o_lat, const void* W_UV, int rows, int H, int d_c, int d_v,
                           void* u, int32_t* status, cudaStream_t s);
cudaError_t launch_lift_simt(mla_dtype act, const void* o_lat, const void* W_UV, int rows, int H,
                             int d_c, int d_v, void* u, cudaStream_t s);

// out = o_lat . W_comb; `acc` is an fp32 [rows][N] accumulator in the caller's workspace.
cudaError_t launch_output_proj_simt_ws(mla_dtype act, const void* o_lat, const void* W_comb,
                                       int rows, int K, int N, void* out, float* acc,
                                       cudaStream_t s);

}  // namespace mla
