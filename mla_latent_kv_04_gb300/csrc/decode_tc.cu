// Tensor-core decode kernel (sm_103a): placeholder until the tcgen05 kernel lands.
#include "decode_tc.h"

namespace mla {

bool tc_decode_supported(const mla_config*) { return false; }
bool tc_decode_default_enabled() { return false; }
cudaError_t launch_decode_tc(mla_dtype, const DecodeParams&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace mla
