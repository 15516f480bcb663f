// Block placement and K/V append.
//
// The draft block's K/V rows are stored in the paged cache right after the
// request's context: block token j of request b goes to logical position
// L_b + j, i.e. page page_table[b][(L_b + j) / P], offset (L_b + j) % P
// (PR #20374: with the block's K/V appended to the pages, one key set
// serves all block queries; the fused spec-tail kernels of the DFlash
// drafter report these positions as the draft block placement).  One thread
// moves one 16-byte piece of one (request, block token, kv head) row of K or
// V, so consecutive threads write consecutive bytes of a row.  The kernel
// lets a following attention kernel launch at once (programmatic dependent
// launch); that kernel reads the pages only after this one has finished.

#include <cuda_runtime.h>

#include "device_common.cuh"

namespace dflash {
namespace {

__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a) {
  pdl_launch_dependents();
  const int cpr = a.D / 8;  // 16-byte pieces per row
  const long long total = static_cast<long long>(a.B) * a.K * a.Hkv * 2 * cpr;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % cpr);
    long long t = idx / cpr;
    const int kv = static_cast<int>(t % 2);
    t /= 2;
    const int h = static_cast<int>(t % a.Hkv);
    t /= a.Hkv;
    const int j = static_cast<int>(t % a.K);
    const int b = static_cast<int>(t / a.K);
    const bool first = h == 0 && kv == 0 && c == 0;  // one thread per (request, block token)

    int L = __ldg(&a.ctx_lens[b]);
    if (L < 0 || L > a.max_ctx_len) {
      if (first && j == 0 && a.status != nullptr) flag_status(a.status, DFLASH_STATUS_BAD_CTX_LEN);
      L = L < 0 ? 0 : a.max_ctx_len;
    }
    const int pos = L + j;
    const int slot = pos / a.P;
    const int off = pos - slot * a.P;
    const int page = __ldg(&a.page_table[static_cast<size_t>(b) * a.max_pages + slot]);
    const bool ok = page >= 0 && page < a.num_pages;
    if (first) {
      if (!ok && a.status != nullptr) flag_status(a.status, DFLASH_STATUS_BAD_PAGE);
      if (a.placement != nullptr) {
        a.placement[(static_cast<size_t>(b) * a.K + j) * 2 + 0] = ok ? page : -1;
        a.placement[(static_cast<size_t>(b) * a.K + j) * 2 + 1] = off;
      }
    }
    if (!ok || a.k_block == nullptr) continue;
    const uint16_t* src = (kv ? a.v_block : a.k_block) +
                          ((static_cast<size_t>(b) * a.K + j) * a.Hkv + h) * a.D + c * 8;
    uint16_t* dst = (kv ? a.v_pages : a.k_pages) +
                    ((static_cast<size_t>(page) * a.Hkv + h) * a.P + off) * a.D + c * 8;
    *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
  }
}

}  // namespace

int launch_append(const AppendArgs& a, cudaStream_t stream) {
  const long long total = static_cast<long long>(a.B) * a.K * a.Hkv * 2 * (a.D / 8);
  long long blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  append_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dflash
