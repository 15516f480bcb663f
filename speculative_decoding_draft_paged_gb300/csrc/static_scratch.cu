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

#include <cuda.h>
#include <cudaTypedefs.h>
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

// The array's address belongs to the context the library's device code was
// loaded into: a context torn down and created again (cudaDeviceReset, for
// one) loads the module anew, possibly elsewhere.  So the cached address is
// keyed on the device and on the driver's id of its current context, which
// is unique for the life of the process.
constexpr int kMaxScratchDevices = 64;
struct ScratchEntry {
  unsigned long long ctx_id = 0;
  void* ptr = nullptr;
};
std::mutex g_scratch_mutex;
ScratchEntry g_scratch[kMaxScratchDevices];

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

void* driver_fn(const char* name, unsigned version) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return fn;
}

// Id of the current context, 0 if there is none (or it cannot be read).
unsigned long long current_ctx_id() {
  std::call_once(g_ctx_once, [] {
    g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(driver_fn("cuCtxGetCurrent", 4000));
    g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(driver_fn("cuCtxGetId", 12000));
  });
  if (g_ctx_current == nullptr || g_ctx_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current device's context: looked
// up with cudaGetSymbolAddress by the first call in each context (which also
// loads the library's device code there if nothing has yet), then cached.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) {
    cudaGetLastError();
    return DFLASH_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  const unsigned long long id = current_ctx_id();
  ScratchEntry& e = g_scratch[dev];
  if (e.ptr == nullptr || id == 0 || e.ctx_id != id) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return DFLASH_ERR_LAUNCH;
    }
    e.ptr = ptr;
    // The lookup makes the primary context current if it was not yet.
    e.ctx_id = id != 0 ? id : current_ctx_id();
  }
  *out = e.ptr;
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
