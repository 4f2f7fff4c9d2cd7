// Tensor-core (tcgen05 / TMEM / TMA) decode kernel interface.
#pragma once
#include "internal.h"

namespace mla {

// True when the configuration has the shape the tensor-core kernel is built for:
// bf16 activations, bf16 or fp8 cache, 64-token pages, 128 heads, d_c 512, d_r 64.
bool tc_decode_supported(const mla_config* c);

// True when the tensor-core kernel is the default choice for supported shapes.
bool tc_decode_default_enabled();

// Launches the attention over the planned work items (one worker per CTA pair).
cudaError_t launch_decode_tc(mla_dtype cache, const DecodeParams& p, cudaStream_t s);

}  // namespace mla
