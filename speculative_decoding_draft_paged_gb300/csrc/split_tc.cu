// tcgen05 / TMEM split kernel: not built yet.
#include "dflash_internal.h"

namespace dflash {

bool split_tc_available() { return false; }
int split_tc_tile_keys(int) { return 128; }
int split_tc_threads() { return 256; }
int split_tc_smem_bytes(int) { return 0; }
int launch_split_tc(const AttnArgs&, const KernelPlan&, const CUtensorMap&, const CUtensorMap&,
                    cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace dflash
