// C-ABI entry points of libmla (declared in include/mla.h): argument validation,
// workspace layout, split planning and kernel dispatch. Nothing here allocates device
// memory; every launch goes to the caller's stream.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <string>

#include "internal.h"
#include "decode_tc.h"
#include "prologue.cuh"

using namespace mla;

namespace mla {
static std::atomic<unsigned long long> g_launches{0};
void note_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }
}  // namespace mla

namespace {

thread_local std::string g_last_error;

mla_status cuda_fail(cudaError_t e, const char* where) {
  g_last_error = std::string(where) + ": " + cudaGetErrorString(e);
  return MLA_ERR_CUDA;
}

mla_status invalid(const char* why) {
  g_last_error = why;
  return MLA_ERR_INVALID;
}

mla_status unsupported(const char* why) {
  g_last_error = why;
  return MLA_ERR_UNSUPPORTED;
}

// Per-device attribute cache (SM count); the only state the library keeps.
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t act_size(mla_dtype t) { return t == MLA_F32 ? 4 : 2; }
size_t cache_size(mla_dtype t) { return t == MLA_F32 ? 4 : (t == MLA_BF16 ? 2 : 1); }

mla_status check_config(const mla_config* c) {
  if (!c) return invalid("config is NULL");
  if (c->num_heads <= 0 || c->d_model <= 0 || c->d_latent <= 0 || c->d_rope <= 0 ||
      c->d_nope <= 0 || c->d_v <= 0 || c->page_size <= 0)
    return invalid("config dimensions must be positive");
  if (c->d_rope % 2) return invalid("d_rope must be even (RoPE rotates pairs)");
  if (c->d_rope / 2 > kMaxRopePairs) return unsupported("d_rope above 128");
  if (c->d_latent % 4 || c->d_rope % 4) return unsupported("d_latent and d_rope must be multiples of 4");
  if (c->page_size > 64) return unsupported("page_size above 64");
  if (c->rope_interleaved != 1) return unsupported("only interleaved RoPE pairs are implemented");
  if (c->act_dtype == MLA_F32) {
    if (c->cache_dtype != MLA_F32) return unsupported("fp32 activations need an fp32 cache");
  } else if (c->act_dtype == MLA_BF16) {
    if (c->cache_dtype != MLA_BF16 && c->cache_dtype != MLA_FP8_E4M3 &&
        c->cache_dtype != MLA_FP8_E4M3_B128)
      return unsupported("bf16 activations need a bf16, fp8_e4m3 or fp8_e4m3_b128 cache");
    if (c->cache_dtype == MLA_FP8_E4M3_B128 && c->d_latent % 128)
      return unsupported("the block-scaled fp8 cache needs d_latent a multiple of 128");
  } else {
    return invalid("act_dtype must be MLA_F32 or MLA_BF16");
  }
  if (c->cache_dtype == MLA_FP8_E4M3 && !(c->cache_scale > 0.f && isfinite(c->cache_scale)))
    return invalid("fp8 cache needs a positive finite cache_scale");
  return MLA_OK;
}

size_t cache_row_bytes(const mla_config* c) {
  if (c->cache_dtype == MLA_FP8_E4M3_B128)
    return (size_t)c->d_latent + (size_t)c->d_latent / 32 + 2 * (size_t)c->d_rope;
  return (size_t)(c->d_latent + c->d_rope) * cache_size(c->cache_dtype);
}

float softmax_scale_of(const mla_config* c) {
  return c->softmax_scale > 0.f ? c->softmax_scale
                                : (float)(1.0 / sqrt((double)(c->d_nope + c->d_rope)));
}

RopeTable rope_table(const mla_config* c) {
  RopeTable rt;
  memset(&rt, 0, sizeof(rt));
  const double theta = c->rope_theta > 0.f ? (double)c->rope_theta : 10000.0;
  rt.pairs = c->d_rope / 2;
  for (int k = 0; k < rt.pairs; ++k) rt.inv_freq[k] = pow(theta, -2.0 * k / (double)c->d_rope);
  return rt;
}

int default_workers(const mla_config* c, const mla_decode_opts* o, bool tc) {
  if (o && o->num_workers > 0) return o->num_workers;
  const int sms = device_sm_count();
  if (tc) return sms > 1 ? sms / 2 : 1;   // one worker per CTA pair
  (void)c;
  return sms > 0 ? sms : 1;
}

mla_status decode_layout(const mla_config* c, int batch, int q_len, int workers,
                         DecodeWorkspace* w) {
  const size_t groups = (size_t)batch * q_len;
  const size_t items = (size_t)workers + groups;
  const size_t D = (size_t)c->d_latent + c->d_rope;
  size_t off = 0;
  w->status = off;       off = align256(off + 16);
  w->worker_off = off;   off = align256(off + (size_t)(workers + 1) * 4);
  w->items = off;        off = align256(off + items * sizeof(WorkItem));
  w->group_first = off;  off = align256(off + groups * 4);
  w->group_last = off;   off = align256(off + groups * 4);
  w->group_kv = off;     off = align256(off + groups * 4);
  w->q_lat = off;        off = align256(off + groups * c->num_heads * D * act_size(c->act_dtype));
  w->part_o = off;       off = align256(off + items * c->num_heads * c->d_latent * 4);
  w->part_lse = off;     off = align256(off + items * c->num_heads * 4);
  w->total = off;
  w->workers = workers;
  w->groups = (int)groups;
  w->max_items = (int)items;
  return MLA_OK;
}

bool use_tc_kernel(const mla_config* c, const mla_decode_opts* o) {
  const int k = o ? o->kernel : 0;
  if (k == 1) return false;
  const bool eligible = tc_decode_supported(c);
  if (k == 2) return eligible;
  return eligible && tc_decode_default_enabled();
}

}  // namespace

namespace mla {
void set_last_error(const std::string& what) { g_last_error = what; }
}  // namespace mla

extern "C" {

int mla_version(void) { return 102; }

uint64_t mla_kernel_launches(void) { return (uint64_t)mla::g_launches.load(); }

const char* mla_last_error(void) { return g_last_error.c_str(); }

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_DEVICE_GUARD: return "device data out of range (rows skipped)";
    case MLA_ERR_TIMEOUT: return "bounded device wait gave up (work skipped)";
  }
  return "unknown status";
}

mla_status mla_absorb_weights(const mla_config* cfg, const void* W_UK, const void* W_UV,
                              const void* W_O, void* W_UK_abs, void* W_comb, void* stream) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (!W_UK || !W_UV || !W_O || !W_UK_abs || !W_comb) return invalid("null weight pointer");
  cudaError_t e = launch_absorb(cfg->act_dtype, W_UK, W_UV, W_O, W_UK_abs, W_comb, cfg->num_heads,
                                cfg->d_latent, cfg->d_nope, cfg->d_v, cfg->d_model,
                                (cudaStream_t)stream);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_absorb_weights");
}

static mla_status check_append(const mla_config* cfg, int T, const int32_t* req_ids,
                               const int32_t* positions, const int32_t* block_table, int batch,
                               int max_pages, void* cache, int num_pages) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (T < 0) return invalid("T must be >= 0");
  if (T > 0 && (!req_ids || !positions || !block_table || !cache))
    return invalid("null pointer");
  if (batch <= 0 || max_pages <= 0 || num_pages <= 0)
    return invalid("batch, max_pages and num_pages must be positive");
  return MLA_OK;
}

mla_status mla_cache_row_bytes(const mla_config* cfg, size_t* bytes) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (!bytes) return invalid("bytes is NULL");
  *bytes = cache_row_bytes(cfg);
  return MLA_OK;
}

mla_status mla_append_cache_workspace_size(const mla_config* cfg, int T, size_t* bytes) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (T < 0 || !bytes) return invalid("T must be >= 0 and bytes non-NULL");
  // the bf16 append sums its split-K partials on chip and the others use none: no scratch
  *bytes = 0;
  return MLA_OK;
}

mla_status mla_append_cache(const mla_config* cfg, const void* h, const void* W_DKV_KR, int T,
                            const int32_t* req_ids, const int32_t* positions,
                            const int32_t* block_table, int batch, int max_pages, void* cache,
                            int num_pages, int32_t* dev_status, void* workspace,
                            size_t workspace_bytes, void* stream) {
  mla_status st = check_append(cfg, T, req_ids, positions, block_table, batch, max_pages, cache,
                               num_pages);
  if (st != MLA_OK) return st;
  if (T == 0) return MLA_OK;
  if (!h || !W_DKV_KR) return invalid("null h or W_DKV_KR");
  const RopeTable rt = rope_table(cfg);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  (void)workspace;
  (void)workspace_bytes;
  if (cfg->act_dtype == MLA_BF16 && cfg->d_model % 8 == 0 &&
      (cfg->d_latent + cfg->d_rope) % 8 == 0) {
    e = launch_append_tc(cfg->cache_dtype, h, W_DKV_KR, T, cfg->d_model, cfg->d_latent, cfg->d_rope,
                         req_ids, positions, block_table, batch, max_pages, cache, num_pages,
                         cfg->page_size, rt, cfg->cache_scale, dev_status, s);
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_append_cache");
  }
  if (cfg->cache_dtype == MLA_FP8_E4M3_B128)
    return unsupported("the block-scaled cache from h needs d_model and d_latent + d_rope "
                       "multiples of 8");
  e = launch_append_from_h(cfg->act_dtype, cfg->cache_dtype, h, W_DKV_KR, T, cfg->d_model, req_ids,
                           positions, block_table, batch, max_pages, cache, num_pages,
                           cfg->page_size, cfg->d_latent, cfg->d_rope, rt, cfg->cache_scale,
                           dev_status, s);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_append_cache");
}

mla_status mla_append_cache_latent(const mla_config* cfg, const void* c_kv, const void* k_pe,
                                   int T, const int32_t* req_ids, const int32_t* positions,
                                   const int32_t* block_table, int batch, int max_pages,
                                   void* cache, int num_pages, int rotate, int32_t* dev_status,
                                   void* stream) {
  mla_status st = check_append(cfg, T, req_ids, positions, block_table, batch, max_pages, cache,
                               num_pages);
  if (st != MLA_OK) return st;
  if (T == 0) return MLA_OK;
  if (!c_kv || !k_pe) return invalid("null c_kv or k_pe");
  const RopeTable rt = rope_table(cfg);
  cudaError_t e = launch_append_latent(cfg->act_dtype, cfg->cache_dtype, c_kv, k_pe, T, req_ids,
                                       positions, block_table, batch, max_pages, cache, num_pages,
                                       cfg->page_size, cfg->d_latent, cfg->d_rope, rotate, rt,
                                       cfg->cache_scale, dev_status, (cudaStream_t)stream);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_append_cache_latent");
}

static mla_status check_decode_shape(const mla_config* cfg, int batch, int q_len) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (batch <= 0 || q_len <= 0) return invalid("batch and q_len must be positive");
  if ((long long)batch * q_len > 32768) return unsupported("batch * q_len above 32768");
  return MLA_OK;
}

mla_status mla_decode_workspace_size(const mla_config* cfg, int batch, int q_len,
                                     const mla_decode_opts* opts, size_t* bytes) {
  mla_status st = check_decode_shape(cfg, batch, q_len);
  if (st != MLA_OK) return st;
  if (!bytes) return invalid("bytes is NULL");
  const bool tc = use_tc_kernel(cfg, opts);
  DecodeWorkspace w;
  decode_layout(cfg, batch, q_len, default_workers(cfg, opts, tc), &w);
  *bytes = w.total;
  return MLA_OK;
}

mla_status mla_decode_ex(const mla_config* cfg, const void* q_nope, const void* q_pe,
                         const void* W_UK_abs, const void* cache, int num_pages,
                         const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                         int batch, int q_len, void* out_latent, float* lse, void* workspace,
                         size_t workspace_bytes, const mla_decode_opts* opts, void* stream) {
  mla_status st = check_decode_shape(cfg, batch, q_len);
  if (st != MLA_OK) return st;
  if (!q_nope || !q_pe || !W_UK_abs || !cache || !block_table || !seq_lens || !out_latent || !lse)
    return invalid("null pointer");
  if (num_pages <= 0 || max_pages <= 0) return invalid("num_pages and max_pages must be positive");
  if (opts && (opts->kernel < 0 || opts->kernel > 2 || opts->num_workers < 0))
    return invalid("bad decode options");
  if (opts && opts->kernel == 2 && !tc_decode_supported(cfg))
    return unsupported("the tensor-core decode kernel needs bf16 activations, 64-token pages and "
                       "the DeepSeek-V2 head shape (128 heads, d_c 512, d_r 64)");
  const bool tc = use_tc_kernel(cfg, opts);
  DecodeWorkspace w;
  decode_layout(cfg, batch, q_len, default_workers(cfg, opts, tc), &w);
  if (!workspace || workspace_bytes < w.total) {
    g_last_error = "workspace smaller than mla_decode_workspace_size";
    return MLA_ERR_WORKSPACE;
  }
  if (((uintptr_t)workspace & 255) != 0) return invalid("workspace must be 256-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = (char*)workspace;
  const RopeTable rt = rope_table(cfg);
  const int D = cfg->d_latent + cfg->d_rope;

  PlanParams pp;
  pp.seq_lens = seq_lens;
  pp.batch = batch;
  pp.q_len = q_len;
  pp.page_size = cfg->page_size;
  pp.max_pages = max_pages;
  pp.workers = w.workers;
  pp.worker_off = (int*)(ws + w.worker_off);
  pp.items = (WorkItem*)(ws + w.items);
  pp.group_first = (int*)(ws + w.group_first);
  pp.group_last = (int*)(ws + w.group_last);
  pp.group_kv = (int*)(ws + w.group_kv);
  pp.status = (int32_t*)(ws + w.status);
  cudaError_t e = cudaSuccess;
  if (cfg->act_dtype == MLA_BF16) {
    // the tensor-core attention takes its query pre-multiplied by softmax_scale * log2(e)
    // (and by an fp8 cache's scale: it multiplies the stored codes, converted exactly)
    const float code_scale = cfg->cache_dtype == MLA_FP8_E4M3 ? cfg->cache_scale : 1.f;
    const float q_scale = tc ? softmax_scale_of(cfg) * kLog2e * code_scale : 1.f;
    // ... and in the planar layout (see internal.h)
    const int planar = tc ? 1 : 0;
    // the tensor-core kernel on a per-tensor e4m3 cache takes an f16 query (its codes convert
    // to f16 exactly, and every MMA's two operands share one type)
    const int f16 = (tc && cfg->cache_dtype == MLA_FP8_E4M3) ? 1 : 0;
    // one launch: the query absorption GEMM with the planner (which clears the status word)
    // and the q_pe rotation as extra blocks. A plan too large for the GEMM block's shared
    // memory runs in the prep kernel, which then goes first.
    if (plan_smem_bytes(batch * q_len, w.workers) <= 32 * 1024) {
      RopeJob rj;
      rj.q_pe = reinterpret_cast<const bf16*>(q_pe);
      rj.seq_lens = seq_lens;
      rj.q_lat = reinterpret_cast<bf16*>(ws + w.q_lat);
      rj.groups = batch * q_len;
      rj.q_len = q_len;
      rj.H = cfg->num_heads;
      rj.d_c = cfg->d_latent;
      rj.d_r = cfg->d_rope;
      rj.planar = planar;
      rj.hblocks = (cfg->num_heads + 31) / 32;
      rj.f16 = f16;
      rj.qs = q_scale;
      rj.rt = rt;
      e = launch_query_absorb_tc(q_nope, W_UK_abs, batch * q_len, cfg->num_heads, cfg->d_nope,
                                 cfg->d_latent, D, q_scale, planar, f16, ws + w.q_lat, pp.status, &pp,
                                 &rj, s);
    } else {
      e = launch_prep(pp, q_pe, seq_lens, q_len, cfg->num_heads, cfg->d_latent, cfg->d_rope, rt,
                      q_scale, planar, f16, ws + w.q_lat, s);
      if (e == cudaSuccess)
        e = launch_query_absorb_tc(q_nope, W_UK_abs, batch * q_len, cfg->num_heads, cfg->d_nope,
                                   cfg->d_latent, D, q_scale, planar, f16, ws + w.q_lat, pp.status,
                                   nullptr, nullptr, s);
    }
  } else {
    e = launch_plan(pp, s);
    if (e != cudaSuccess) return cuda_fail(e, "mla_decode (plan)");
    e = launch_query_prologue(cfg->act_dtype, q_nope, q_pe, W_UK_abs, seq_lens, batch, q_len,
                              cfg->num_heads, cfg->d_nope, cfg->d_latent, cfg->d_rope, rt,
                              ws + w.q_lat, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "mla_decode (query prologue)");

  DecodeParams dp;
  dp.q_lat = ws + w.q_lat;
  dp.cache = cache;
  dp.block_table = block_table;
  dp.max_pages = max_pages;
  dp.num_pages = num_pages;
  dp.batch = batch;
  dp.q_len = q_len;
  dp.H = cfg->num_heads;
  dp.d_c = cfg->d_latent;
  dp.d_r = cfg->d_rope;
  dp.D = D;
  dp.P = cfg->page_size;
  dp.row_bytes = (long long)cache_row_bytes(cfg);
  const float cs = cfg->cache_dtype == MLA_FP8_E4M3 ? cfg->cache_scale : 1.f;
  dp.scale_log2 = tc ? cs : softmax_scale_of(cfg) * cs * kLog2e;   // tc: query pre-scaled
  dp.out_scale = cs;
  dp.out_latent = out_latent;
  dp.lse = lse;
  dp.worker_off = pp.worker_off;
  dp.items = pp.items;
  dp.group_first = pp.group_first;
  dp.group_last = pp.group_last;
  dp.group_kv = pp.group_kv;
  dp.part_o = (float*)(ws + w.part_o);
  dp.part_lse = (float*)(ws + w.part_lse);
  dp.status = pp.status;
  dp.workers = w.workers;
  dp.part_planar = tc ? 1 : 0;
  dp.wait_limit_ns = (opts && opts->wait_limit_us > 0) ? 1000ull * (unsigned long long)opts->wait_limit_us
                                                       : 2000000000ull;
  dp.withhold_page = (opts && opts->withhold_page > 0) ? opts->withhold_page : 0;
  if (opts && opts->attn_events[0]) {
    e = cudaEventRecord((cudaEvent_t)opts->attn_events[0], s);
    if (e != cudaSuccess) return cuda_fail(e, "mla_decode (timing event)");
  }
  e = tc ? launch_decode_tc(cfg->cache_dtype, dp, s)
         : launch_decode_simt(cfg->act_dtype, cfg->cache_dtype, dp, s);
  if (e != cudaSuccess) return cuda_fail(e, "mla_decode (attention)");
  if (opts && opts->attn_events[1]) {
    e = cudaEventRecord((cudaEvent_t)opts->attn_events[1], s);
    if (e != cudaSuccess) return cuda_fail(e, "mla_decode (timing event)");
  }
  e = launch_combine(cfg->act_dtype, dp, w.groups, s);
  if (e != cudaSuccess) return cuda_fail(e, "mla_decode (combine)");
  return MLA_OK;
}

mla_status mla_decode(const mla_config* cfg, const void* q_nope, const void* q_pe,
                      const void* W_UK_abs, const void* cache, int num_pages,
                      const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                      int batch, int q_len, void* out_latent, float* lse, void* workspace,
                      size_t workspace_bytes, void* stream) {
  return mla_decode_ex(cfg, q_nope, q_pe, W_UK_abs, cache, num_pages, block_table, max_pages,
                       seq_lens, batch, q_len, out_latent, lse, workspace, workspace_bytes, nullptr,
                       stream);
}

mla_status mla_output_proj_workspace_size(const mla_config* cfg, int rows, size_t* bytes) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (rows < 0 || !bytes) return invalid("rows must be >= 0 and bytes non-NULL");
  *bytes = align256((size_t)rows * cfg->d_model * 4) + 256;
  return MLA_OK;
}

mla_status mla_output_proj(const mla_config* cfg, const void* out_latent, const void* W_comb,
                           int rows, void* out, void* workspace, size_t workspace_bytes,
                           void* stream) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (rows < 0) return invalid("rows must be >= 0");
  if (rows == 0) return MLA_OK;
  if (!out_latent || !W_comb || !out) return invalid("null pointer");
  const size_t acc_bytes = align256((size_t)rows * cfg->d_model * 4);
  if (!workspace || workspace_bytes < acc_bytes + 256) {
    g_last_error = "workspace smaller than mla_output_proj_workspace_size";
    return MLA_ERR_WORKSPACE;
  }
  if (((uintptr_t)workspace & 255) != 0) return invalid("workspace must be 256-byte aligned");
  cudaError_t e;
  if (cfg->act_dtype == MLA_BF16)
    e = launch_output_proj_tc(out_latent, W_comb, rows, cfg->num_heads * cfg->d_latent,
                              cfg->d_model, out, (int32_t*)((char*)workspace + acc_bytes),
                              (cudaStream_t)stream);
  else
    e = launch_output_proj_simt_ws(cfg->act_dtype, out_latent, W_comb, rows,
                                   cfg->num_heads * cfg->d_latent, cfg->d_model, out,
                                   (float*)workspace, (cudaStream_t)stream);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_output_proj");
}

// workspace of the unfolded projection: fp32 accumulator, status word, lifted u
static size_t unfolded_acc_bytes(const mla_config* c, int rows) {
  return align256((size_t)rows * c->d_model * 4);
}
static size_t unfolded_u_bytes(const mla_config* c, int rows) {
  return align256((size_t)rows * c->num_heads * c->d_v * act_size(c->act_dtype));
}

mla_status mla_output_proj_unfolded_workspace_size(const mla_config* cfg, int rows, size_t* bytes) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (rows < 0 || !bytes) return invalid("rows must be >= 0 and bytes non-NULL");
  *bytes = unfolded_acc_bytes(cfg, rows) + 256 + unfolded_u_bytes(cfg, rows);
  return MLA_OK;
}

mla_status mla_output_proj_unfolded(const mla_config* cfg, const void* out_latent, const void* W_UV,
                                    const void* W_O, int rows, void* out, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (rows < 0) return invalid("rows must be >= 0");
  if (rows == 0) return MLA_OK;
  if (!out_latent || !W_UV || !W_O || !out) return invalid("null pointer");
  const size_t acc_bytes = unfolded_acc_bytes(cfg, rows);
  if (!workspace || workspace_bytes < acc_bytes + 256 + unfolded_u_bytes(cfg, rows)) {
    g_last_error = "workspace smaller than mla_output_proj_unfolded_workspace_size";
    return MLA_ERR_WORKSPACE;
  }
  if (((uintptr_t)workspace & 255) != 0) return invalid("workspace must be 256-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  float* acc = (float*)workspace;
  int32_t* status = (int32_t*)((char*)workspace + acc_bytes);
  void* u = (char*)workspace + acc_bytes + 256;
  const int H = cfg->num_heads, d_c = cfg->d_latent, d_v = cfg->d_v, d = cfg->d_model;
  cudaError_t e;
  if (cfg->act_dtype == MLA_BF16 && d_c % 64 == 0 && d_v % 64 == 0) {
    e = launch_lift_tc(out_latent, W_UV, rows, H, d_c, d_v, u, status, s);
    if (e == cudaSuccess) e = launch_output_proj_tc(u, W_O, rows, H * d_v, d, out, status, s);
  } else {
    e = launch_lift_simt(cfg->act_dtype, out_latent, W_UV, rows, H, d_c, d_v, u, s);
    if (e == cudaSuccess)
      e = launch_output_proj_simt_ws(cfg->act_dtype, u, W_O, rows, H * d_v, d, out, acc, s);
  }
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_output_proj_unfolded");
}

// Query side: three GEMMs through fp32 accumulators, one accumulator region reused in stream
// order (each GEMM zeroes it after the previous conversion has read it).
static size_t query_acc_bytes(const mla_config* c, int d_q, int T) {
  const size_t w = std::max<size_t>((size_t)d_q,
                                    std::max((size_t)c->num_heads * c->d_rope,
                                             (size_t)c->num_heads * c->d_nope));
  return align256((size_t)T * w * 4);
}
static size_t query_cq_bytes(const mla_config* c, int d_q, int T) {
  return align256((size_t)T * d_q * act_size(c->act_dtype));
}

mla_status mla_query_workspace_size(const mla_config* cfg, int d_q, int T, size_t* bytes) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (d_q <= 0 || T < 0 || !bytes) return invalid("d_q must be positive, T >= 0, bytes non-NULL");
  *bytes = query_acc_bytes(cfg, d_q, T) + 256 + query_cq_bytes(cfg, d_q, T);
  return MLA_OK;
}

mla_status mla_query_from_hidden(const mla_config* cfg, int d_q, const void* h, const void* W_DQ,
                                 const void* W_UQ, const void* W_QR, int T, void* q_nope,
                                 void* q_pe, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (d_q <= 0 || T < 0) return invalid("d_q must be positive and T >= 0");
  if (T == 0) return MLA_OK;
  if (!h || !W_DQ || !W_UQ || !W_QR || !q_nope || !q_pe) return invalid("null pointer");
  const size_t acc_bytes = query_acc_bytes(cfg, d_q, T);
  if (!workspace || workspace_bytes < acc_bytes + 256 + query_cq_bytes(cfg, d_q, T)) {
    g_last_error = "workspace smaller than mla_query_workspace_size";
    return MLA_ERR_WORKSPACE;
  }
  if (((uintptr_t)workspace & 255) != 0) return invalid("workspace must be 256-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  float* acc = (float*)workspace;
  int32_t* status = (int32_t*)((char*)workspace + acc_bytes);
  void* c_q = (char*)workspace + acc_bytes + 256;
  const int H = cfg->num_heads, d = cfg->d_model;
  const int n_pe = H * cfg->d_rope, n_nope = H * cfg->d_nope;
  // tensor maps need 16-byte row strides: every row length a multiple of 8 bf16 elements
  const bool tc = cfg->act_dtype == MLA_BF16 && d % 8 == 0 && d_q % 8 == 0 && n_pe % 8 == 0 &&
                  n_nope % 8 == 0;
  cudaError_t e;
  if (tc) {
    // c_q and q_pe both read h: one launch for the two weights, then q_nope from c_q
    e = launch_two_proj_tc(h, W_DQ, W_QR, T, d, d_q, n_pe, c_q, q_pe, status, s);
    if (e == cudaSuccess) e = launch_output_proj_tc(c_q, W_UQ, T, d_q, n_nope, q_nope, status, s);
  } else {
    e = launch_output_proj_simt_ws(cfg->act_dtype, h, W_DQ, T, d, d_q, c_q, acc, s);
    if (e == cudaSuccess)
      e = launch_output_proj_simt_ws(cfg->act_dtype, h, W_QR, T, d, n_pe, q_pe, acc, s);
    if (e == cudaSuccess)
      e = launch_output_proj_simt_ws(cfg->act_dtype, c_q, W_UQ, T, d_q, n_nope, q_nope, acc, s);
  }
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_query_from_hidden");
}

mla_status mla_read_device_status(const void* status_word, void* stream, int* code) {
  if (!status_word || !code) return invalid("null pointer");
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "mla_read_device_status (sync)");
  int32_t word = 0;
  e = cudaMemcpy(&word, status_word, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "mla_read_device_status (read)");
  const int32_t zero = 0;
  e = cudaMemcpy((void*)status_word, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "mla_read_device_status (reset)");
  if (word & (1 << MLA_ERR_TIMEOUT)) *code = MLA_ERR_TIMEOUT;
  else if (word & (1 << MLA_ERR_DEVICE_GUARD)) *code = MLA_ERR_DEVICE_GUARD;
  else *code = word ? MLA_ERR_CUDA : MLA_OK;
  return MLA_OK;
}

}  // extern "C"
