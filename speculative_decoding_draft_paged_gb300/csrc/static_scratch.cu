// dflash_block_attn_static_ws: the attention call for callers that cannot
// allocate device memory themselves.
//
// Some callers have no way to provide a workspace: code that runs while a
// stream is being captured under a mode that forbids cudaMalloc, plugin code
// whose host framework owns every device allocation and hands the plugin no
// scratch buffer, or latency-critical paths that must not take an
// allocator's locks or its implicit synchronisation.  For them this entry
// point uses a fixed scratch array compiled into the library instead of a
// caller-provided workspace.  It allocates nothing and calls no allocating
// routine; it runs exactly the same kernels as dflash_block_attn.

#include <mutex>

#include <cuda_runtime.h>

#include "dflash.h"
#include "dflash_internal.h"

namespace dflash {
namespace {

constexpr size_t kStaticScratchBytes = DFLASH_STATIC_SCRATCH_BYTES;

// One copy per device that loads the library, held until the process exits.
// In host code this name is only a host-side stand-in: its device address is
// obtained with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxScratchDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the first call on each device does it).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) {
    cudaGetLastError();
    return DFLASH_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return DFLASH_ERR_LAUNCH;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return DFLASH_OK;
}

}  // namespace
}  // namespace dflash

extern "C" int dflash_block_attn_static_ws(const dflash_params* p, const void* q,
                                           const void* k_pages, const void* v_pages,
                                           const int32_t* page_table, const int32_t* ctx_lens,
                                           void* out, float* lse2, void* stream) {
  const size_t need = dflash_workspace_size(p);
  if (need == 0) return DFLASH_ERR_INVALID;
  if (need > dflash::kStaticScratchBytes) return DFLASH_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = dflash::scratch_address(&scratch);
  if (rc != DFLASH_OK) return rc;
  return dflash_block_attn(p, q, k_pages, v_pages, page_table, ctx_lens, out, lse2, scratch,
                           dflash::kStaticScratchBytes, stream);
}
