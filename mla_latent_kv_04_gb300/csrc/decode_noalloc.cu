// mla_decode_noalloc: the decode call for callers that must not allocate device memory.
//
// Some callers of a decode kernel cannot call cudaMalloc at the point where they decode:
// a plugin or custom op embedded in a host runtime that owns every device allocation and
// hands its kernels no allocator, a serving loop that forbids allocation after warm-up so
// that its memory footprint is fixed and latency has no allocator stalls, or a runtime
// whose rules (certification, real-time) ban dynamic allocation outright. For them this
// entry point takes its scratch from one statically sized array in device memory instead
// of a caller-provided workspace.
//
// The array is set up once per device: the first call on a device, with that device
// current, looks up the array's device address with cudaGetSymbolAddress. Make that first
// call outside any stream capture. The address is kept for the life of the process, so the
// library must not outlive a cudaDeviceReset of a device it has decoded on (the reset
// unloads the module that holds the array). The array lives as long as the library is
// loaded, on every GPU that loads it, and every call shares it: two calls whose work
// overlaps on the GPU (different streams, or different host threads without ordering) race
// on it. The decode needs no zeroed scratch (each call clears the status word it uses), so
// the contents left by the previous call are harmless.
//
// The decode's device guards (a block-table entry outside the cache, a seq_len above the
// block-table row) report through a status word at the start of the array, which the caller
// cannot address; mla_decode_noalloc_status reads and clears it.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/mla.h"

namespace mla {
void set_last_error(const std::string& what);
}

namespace {

constexpr size_t kScratchBytes = 64ull << 20;   // 64 MiB per device
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

mla_status scratch_of_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    mla::set_last_error("mla_decode_noalloc: no current CUDA device");
    return MLA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_decode_scratch);
    if (e != cudaSuccess || addr == nullptr) {
      mla::set_last_error(std::string("mla_decode_noalloc: cudaGetSymbolAddress failed: ") +
                          cudaGetErrorString(e));
      return MLA_ERR_CUDA;
    }
    g_scratch_addr[dev] = addr;
  }
  *out = g_scratch_addr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_decode_noalloc(const mla_config* cfg, const void* q_nope,
                                         const void* q_pe, const void* W_UK_abs, const void* cache,
                                         int num_pages, const int32_t* block_table, int max_pages,
                                         const int32_t* seq_lens, int batch, int q_len,
                                         void* out_latent, float* lse, void* stream) {
  size_t need = 0;
  mla_status st = mla_decode_workspace_size(cfg, batch, q_len, nullptr, &need);
  if (st != MLA_OK) return st;
  if (need > kScratchBytes) {
    mla::set_last_error("mla_decode_noalloc: this batch needs " + std::to_string(need) +
                        " bytes of scratch, above the fixed " + std::to_string(kScratchBytes) +
                        "-byte array; use mla_decode with a caller-provided workspace");
    return MLA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  st = scratch_of_current_device(&scratch);
  if (st != MLA_OK) return st;
  return mla_decode(cfg, q_nope, q_pe, W_UK_abs, cache, num_pages, block_table, max_pages,
                    seq_lens, batch, q_len, out_latent, lse, scratch, kScratchBytes, stream);
}

extern "C" mla_status mla_decode_noalloc_status(void* stream, int* code) {
  if (!code) {
    mla::set_last_error("mla_decode_noalloc_status: code is NULL");
    return MLA_ERR_INVALID;
  }
  void* scratch = nullptr;
  const mla_status st = scratch_of_current_device(&scratch);
  if (st != MLA_OK) return st;
  // the decode's status word is the first int32 of its workspace, here the array
  return mla_read_device_status(scratch, stream, code);
}
