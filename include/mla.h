/*
 * mla.h - C ABI of libmla: weight-absorbed Multi-head Latent Attention (MLA)
 * decode on one GB300 (sm_103a).
 *
 * What the library computes (pages cited by title and section):
 *   - "DeepSeek Multi-Head Latent Attention(MLA) 해부" (blog.huny.dev), §2-1 (the
 *     latent c_t = h_t W^DKV), §2-3 (decoupled RoPE key k^R = RoPE(h_t W^KR), the
 *     concatenated query/key and the score split), §3-1 (W^UK absorbed into the
 *     query) and §3-2 (W^UV folded into W^O);
 *   - "KV Cache를 10분의 1로 줄인 MLA의 트릭" (donmain.dev), "위치 정보와 압축의 충돌":
 *     the cache stores c_t (512) and k^R_t (64) = 576 elements per token, the
 *     absorption is done once at model load;
 *   - "[vLLM] Multi-head Latent Attention" (blog.secrett2633.cloud), "FlashMLABackend"
 *     (64-token pages, bf16 or fp8_e4m3 cache), "MLA의 MQA 디코딩 경로" (decode runs
 *     as MQA: every query head over one shared latent "KV head"), "FlashMLAImpl"
 *     (query given as (q_nope, q_pe) and concatenated, LSE returned, several query
 *     tokens per request for speculative decoding).
 *
 * Conventions shared by every call
 *   - Every tensor argument is a DEVICE pointer to a contiguous row-major array
 *     owned by the caller; the library allocates no device memory and keeps no
 *     global state beyond a per-device cache of attributes and tensor-map
 *     encoders. Sizes are element counts unless stated.
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream. Every call only enqueues work on `stream` and returns; results are
 *     ready when the stream reaches that point.
 *   - Host-side validation runs before anything is enqueued: a null pointer, a
 *     bad dimension, an unsupported dtype combination or a too-small workspace
 *     returns MLA_ERR_INVALID / MLA_ERR_UNSUPPORTED / MLA_ERR_WORKSPACE and
 *     enqueues nothing. A CUDA launch failure returns MLA_ERR_CUDA.
 *   - Device-side guards: data that only the device sees (a block-table entry
 *     outside [0, num_pages), a request id outside [0, batch), a position past the
 *     request's block-table row, a seq_len below q_len or above
 *     max_pages*page_size) never causes an out-of-bounds access: the offending
 *     row or request is skipped and MLA_ERR_DEVICE_GUARD is OR-ed into a device
 *     status word, which mla_read_device_status returns.
 *
 * Dtypes: act_dtype (activations, weights, queries, outputs) is MLA_F32 or
 * MLA_BF16; cache_dtype is MLA_F32 (only with MLA_F32 activations), MLA_BF16,
 * MLA_FP8_E4M3 or MLA_FP8_E4M3_B128 (the last two only with MLA_BF16 activations).
 * bf16 and fp8 values are rounded to nearest-even; fp8 saturates to +-448.
 *   - MLA_FP8_E4M3: c_kv and k_pe as e4m3 codes, dequantised as code * cache_scale
 *     (one per-tensor scale).
 *   - MLA_FP8_E4M3_B128: the fp8 cache huny.dev §6 describes for DeepSeek-V3. c_kv is in
 *     e4m3 with one fp32 scale per 128 consecutive latent elements of each token, computed
 *     from the values when the token is written: scale = amax|x| / 448 and
 *     code = e4m3(x / scale), both divisions in IEEE fp32; a block of zeros has scale 0 and
 *     codes 0. The rotated k_pe stays in bf16. A cache row holds d_c code bytes, then d_c/128
 *     fp32 scales, then d_r bf16 values: d_c + d_c/32 + 2 d_r bytes (656 at DeepSeek-V2
 *     shapes; mla_cache_row_bytes). d_c must be a multiple of 128, and cache_scale is
 *     ignored.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID = 1,      /* bad argument (null pointer, bad size or layout)        */
  MLA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (dtype or shape combination)  */
  MLA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required              */
  MLA_ERR_CUDA = 4,         /* a CUDA runtime/driver call or a launch failed           */
  MLA_ERR_DEVICE_GUARD = 5, /* device data out of range; the bad rows were skipped     */
  MLA_ERR_TIMEOUT = 6       /* a bounded device-side wait gave up; the work was skipped */
} mla_status;

typedef enum { MLA_F32 = 0, MLA_BF16 = 1, MLA_FP8_E4M3 = 2, MLA_FP8_E4M3_B128 = 3 } mla_dtype;

/* Model dimensions and numeric options of one MLA layer.
 *   num_heads H, d_model d, d_latent d_c (c_kv width), d_rope d_r (k_pe width),
 *   d_nope d_n (per-head content query/key width), d_v (per-head value width),
 *   page_size P (tokens per cache page; 64 as in the FlashMLA backend).
 *   softmax_scale: multiplies q.k; <= 0 selects 1/sqrt(d_n + d_r).
 *   rope_theta: RoPE base; <= 0 selects 10000. Pairs (2k, 2k+1) are rotated by
 *     pos * theta^(-2k/d_r) (rope_interleaved = 1, the only supported layout).
 *   cache_scale: fp8 dequantisation scale (ignored for other cache dtypes). */
typedef struct {
  int num_heads, d_model, d_latent, d_rope, d_nope, d_v, page_size;
  float softmax_scale;
  float rope_theta;
  int rope_interleaved;
  mla_dtype act_dtype;
  mla_dtype cache_dtype;
  float cache_scale;
} mla_config;

/* Fold the up-projections into the serving weights, once at model load
 * (donmain.dev "위치 정보와 압축의 충돌"; huny.dev §3-1, §3-2).
 *   W_UK [d_c][H*d_n], W_UV [d_c][H*d_v], W_O [H*d_v][d]  (act dtype, inputs; head i
 *     owns columns i*d_n.. of W_UK, i*d_v.. of W_UV and rows i*d_v.. of W_O)
 *   W_UK_abs [H][d_n][d_c]   out: W_UK_abs[i] = (W_i^UK)^T
 *   W_comb   [H*d_c][d]      out: block i = W_i^UV W_i^O  (fp32 accumulation) */
mla_status mla_absorb_weights(const mla_config* cfg, const void* W_UK, const void* W_UV,
                              const void* W_O, void* W_UK_abs, void* W_comb, void* stream);

/* Append T new tokens from hidden states (huny.dev §2-1 and §2-3):
 *   [c | k_raw] = h W_DKV_KR,  k^R = RoPE(k_raw, position),
 * encoded in the cache dtype and written to
 *   cache[block_table[req][pos / P]][pos % P][0 : d_c + d_r] = [c | k^R].
 *   h [T][d], W_DKV_KR [d][d_c + d_r] = [W^DKV | W^KR]   (act dtype)
 *   req_ids [T], positions [T]          int32 (device)
 *   block_table [batch][max_pages]      int32 (device)
 *   cache [num_pages][P][d_c + d_r]     cache dtype, updated in place (MLA_FP8_E4M3_B128:
 *                                       bytes, [num_pages][P][mla_cache_row_bytes])
 *   dev_status                          optional int32 device word (may be NULL):
 *                                       MLA_ERR_DEVICE_GUARD is OR-ed in for skipped rows.
 *   workspace                           device buffer of mla_append_cache_workspace_size
 *                                       bytes (may be NULL when that is 0, as it is now for
 *                                       every configuration: the bf16 path sums its split-K
 *                                       partials on chip and encodes in the same kernel).
 * Rows must not share a (request, position); T == 0 is a no-op. */
mla_status mla_append_cache(const mla_config* cfg, const void* h, const void* W_DKV_KR, int T,
                            const int32_t* req_ids, const int32_t* positions,
                            const int32_t* block_table, int batch, int max_pages, void* cache,
                            int num_pages, int32_t* dev_status, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Bytes of one token's row in the paged cache: (d_c + d_r) * element size, or
 * d_c + d_c/32 + 2 d_r for MLA_FP8_E4M3_B128. A page is P rows. */
mla_status mla_cache_row_bytes(const mla_config* cfg, size_t* bytes);

/* Bytes of workspace mla_append_cache needs for T rows (currently 0). */
mla_status mla_append_cache_workspace_size(const mla_config* cfg, int T, size_t* bytes);

/* Append T tokens given their latent c_kv [T][d_c] and raw k_pe [T][d_r] (act dtype).
 * rotate != 0 applies RoPE at `positions` to k_pe before encoding; rotate == 0 stores
 * k_pe as given. Placement, encoding and guards as mla_append_cache. */
mla_status mla_append_cache_latent(const mla_config* cfg, const void* c_kv, const void* k_pe,
                                   int T, const int32_t* req_ids, const int32_t* positions,
                                   const int32_t* block_table, int batch, int max_pages,
                                   void* cache, int num_pages, int rotate, int32_t* dev_status,
                                   void* stream);

/* Decode tuning knobs (NULL = defaults). num_workers: how many independent workers
 * share the key pages (0 = one per SM pair on this GPU); kernel: 0 = best available,
 * 1 = the SIMT kernel, 2 = the tensor-core (tcgen05) kernel. attn_events: optional
 * pair of cudaEvent_t (as void*) recorded on `stream` right before and right after
 * the attention kernel, for timing it alone; NULL entries are ignored.
 * Testing hooks of the tensor-core kernel's failure path (zero-initialise them otherwise):
 * wait_limit_us: how long any of its barrier waits may last before the kernel gives up,
 * records MLA_ERR_TIMEOUT in the status word, releases its tensor memory and exits
 * (0 = the default, 2 s); withhold_page: when >= 1, the page of index withhold_page - 1 in
 * worker 0's sequence is never loaded, so that the wait for it runs out (0 = off). Both
 * leave every other worker's results intact; the call's status then reads
 * MLA_ERR_TIMEOUT and its outputs for worker 0's requests are undefined. */
typedef struct {
  int num_workers;
  int kernel;
  void* attn_events[2];
  int wait_limit_us;
  int withhold_page;
} mla_decode_opts;

/* Bytes of workspace mla_decode needs for this batch on the current device. */
mla_status mla_decode_workspace_size(const mla_config* cfg, int batch, int q_len,
                                     const mla_decode_opts* opts, size_t* bytes);

/* Weight-absorbed decode (huny.dev §3-1; secrett2633.cloud "MLA의 MQA 디코딩 경로",
 * "FlashMLAImpl"). For request b, query token t (0 <= t < q_len) sits at position
 * p = seq_lens[b] - q_len + t and attends to the cached keys 0..p of its request;
 * for every head i:
 *   q_lat = [ q_nope[b][t][i] W_UK_abs[i] ; RoPE(q_pe[b][t][i], p) ]      (d_c + d_r)
 *   s_j   = softmax_scale * q_lat . cache_row_j            (fp8: * cache_scale)
 *   out_latent[b][t][i] = sum_j softmax(s)_j c_j,  lse[b][t][i] = ln sum_j exp(s_j).
 *   q_nope [batch][q_len][H][d_n], q_pe [batch][q_len][H][d_r], W_UK_abs [H][d_n][d_c]
 *     (act dtype); cache, num_pages as in mla_append_cache;
 *   block_table [batch][max_pages], seq_lens [batch]  int32 (device); seq_lens count the
 *     cached tokens including this step's q_len tokens (appended before the call);
 *   out_latent [batch][q_len][H][d_c] (act dtype), lse [batch][q_len][H] (fp32)  outputs.
 * seq_lens[b] == 0 marks an empty request: out_latent = 0, lse = -inf.
 * workspace: device buffer of at least mla_decode_workspace_size bytes, 256-byte
 * aligned, owned by the caller, any initial contents; its first int32 is the device
 * status word, cleared by each call and then set by that call's guards. Calls that
 * share one workspace must be ordered on the GPU. */
mla_status mla_decode(const mla_config* cfg, const void* q_nope, const void* q_pe,
                      const void* W_UK_abs, const void* cache, int num_pages,
                      const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                      int batch, int q_len, void* out_latent, float* lse, void* workspace,
                      size_t workspace_bytes, void* stream);

/* mla_decode with explicit knobs (opts may be NULL). */
mla_status mla_decode_ex(const mla_config* cfg, const void* q_nope, const void* q_pe,
                         const void* W_UK_abs, const void* cache, int num_pages,
                         const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                         int batch, int q_len, void* out_latent, float* lse, void* workspace,
                         size_t workspace_bytes, const mla_decode_opts* opts, void* stream);

/* mla_decode without a caller workspace, for callers that cannot allocate device memory
 * when they decode (a plugin inside a runtime that owns all device allocations, a serving
 * loop with a frozen memory footprint, an environment that bans dynamic allocation). The
 * pages have no counterpart to this call: it is a deployment convenience of this library.
 * Its scratch is one 64 MiB array in device memory, statically part of the library and
 * held by every GPU that loads it until the process exits; a batch whose
 * mla_decode_workspace_size exceeds 64 MiB is rejected with MLA_ERR_WORKSPACE and an
 * explanation in mla_last_error(). The first call on a device looks the array up
 * (cudaGetSymbolAddress) with that device current: make it outside any stream capture.
 * All calls share the array, so calls whose GPU work overlaps (other streams, unordered
 * host threads) race; order them on one stream. Nothing in the array needs to start at
 * zero. Arguments and results are those of mla_decode; the call's device status (its
 * guards) is read with mla_decode_noalloc_status. */
mla_status mla_decode_noalloc(const mla_config* cfg, const void* q_nope, const void* q_pe,
                              const void* W_UK_abs, const void* cache, int num_pages,
                              const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                              int batch, int q_len, void* out_latent, float* lse, void* stream);

/* The device status of the last mla_decode_noalloc on the current device: waits for
 * `stream`, then reads the status word at the start of the library's scratch array into
 * *code (MLA_OK, or MLA_ERR_DEVICE_GUARD when that call's guards skipped a request) and
 * resets it to 0. The pages have no counterpart to this call. The array's address is looked
 * up once per device and kept: neither call may be used on a device after a
 * cudaDeviceReset of it in the same process. Errors: MLA_ERR_INVALID (code is NULL),
 * MLA_ERR_CUDA. */
mla_status mla_decode_noalloc_status(void* stream, int* code);

/* Bytes of workspace mla_output_proj needs for `rows` rows (may be 0). */
mla_status mla_output_proj_workspace_size(const mla_config* cfg, int rows, size_t* bytes);

/* Output projection through the folded weights (huny.dev §3-2):
 *   out[r] = sum_i out_latent[r][i] W_comb[i*d_c : (i+1)*d_c]
 *   out_latent [rows][H*d_c], W_comb [H*d_c][d], out [rows][d]  (act dtype),
 *   fp32 accumulation. workspace: 256-byte aligned device buffer of
 *   mla_output_proj_workspace_size bytes (an fp32 accumulator, used with fp32 activations,
 *   plus a status word). */
mla_status mla_output_proj(const mla_config* cfg, const void* out_latent, const void* W_comb,
                           int rows, void* out, void* workspace, size_t workspace_bytes,
                           void* stream);

/* Bytes of workspace mla_output_proj_unfolded needs for `rows` rows (may be 0). */
mla_status mla_output_proj_unfolded_workspace_size(const mla_config* cfg, int rows,
                                                   size_t* bytes);

/* Output projection without the fold, the two sides of huny.dev §3-2 read before the
 * absorption (its first equation, then the per-head output projection):
 *   u[r][i] = out_latent[r][i] W_i^UV      (per head: d_c -> d_v, rounded to the act dtype)
 *   out[r]  = sum_i u[r][i] W_i^O
 *   out_latent [rows][H*d_c]; W_UV [d_c][H*d_v] and W_O [H*d_v][d] as given to
 *   mla_absorb_weights (head i owns columns i*d_v.. of W_UV, rows i*d_v.. of W_O);
 *   out [rows][d]  (act dtype), fp32 accumulation. It streams H*d_c*d_v + H*d_v*d weight
 *   elements instead of W_comb's H*d_c*d (185 MB instead of 671 MB at DeepSeek-V2 shapes);
 *   equal to mla_output_proj up to the rounding of u. workspace: 256-byte aligned device
 *   buffer of mla_output_proj_unfolded_workspace_size bytes (an fp32 accumulator, used with
 *   fp32 activations, a status word and u). Errors as mla_output_proj. */
mla_status mla_output_proj_unfolded(const mla_config* cfg, const void* out_latent, const void* W_UV,
                                    const void* W_O, int rows, void* out, void* workspace,
                                    size_t workspace_bytes, void* stream);

/* Bytes of workspace mla_query_from_hidden needs for T query rows and query rank d_q. */
mla_status mla_query_workspace_size(const mla_config* cfg, int d_q, int T, size_t* bytes);

/* The step's queries from the hidden states, by low-rank query compression (huny.dev
 * "DeepSeek MLA 해부" §2-2) and the per-head rotary query (§2-3):
 *   c_q[t]       = h[t] W_DQ                              (d -> d_q, rounded to the act dtype)
 *   q_nope[t][i] = c_q[t] W_UQ[:, i*d_n : (i+1)*d_n]
 *   q_pe[t][i]   = h[t] W_QR[:, i*d_r : (i+1)*d_r]       (not rotated: mla_decode rotates it
 *                                                          at the query position)
 *   h [T][d]; W_DQ [d][d_q]; W_UQ [d_q][H*d_n]; W_QR [d][H*d_r]; outputs q_nope [T][H][d_n]
 *   and q_pe [T][H][d_r], the layouts mla_decode reads (row b*q_len + t), all in the act
 *   dtype, fp32 accumulation. W_UQ stays separate from W_UK: merging them per head
 *   (W_i^UQ (W_i^UK)^T, d_q x d_c) would make the step read H*d_q*d_c weight elements (201 MB at
 *   DeepSeek-V2 shapes) instead of H*d_q*d_n + H*d_n*d_c (67 MB).
 *   workspace: 256-byte aligned device buffer of mla_query_workspace_size bytes (an fp32
 *   accumulator, used with fp32 activations, a status word and c_q). d_q > 0; T == 0 is a no-op. Errors: MLA_ERR_INVALID
 *   (null pointers, bad sizes), MLA_ERR_WORKSPACE, MLA_ERR_CUDA; nothing is launched on an
 *   error found on the host. */
mla_status mla_query_from_hidden(const mla_config* cfg, int d_q, const void* h, const void* W_DQ,
                                 const void* W_UQ, const void* W_QR, int T, void* q_nope,
                                 void* q_pe, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* Wait for `stream`, then read the device status word at `status_word` (a decode
 * workspace or an append dev_status) into *code (an mla_status value, MLA_OK if clean)
 * and reset it to 0. */
mla_status mla_read_device_status(const void* status_word, void* stream, int* code);

/* Static description of a status code. */
const char* mla_status_string(mla_status status);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char* mla_last_error(void);

/* Library ABI version (major * 100 + minor). 1.02: mla_append_cache needs no workspace
 * (its size is 0). */
int mla_version(void);

/* Number of CUDA kernels the library has launched in this process so far (all
 * threads, all devices); lets a caller count the kernels of a timed region. */
uint64_t mla_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
