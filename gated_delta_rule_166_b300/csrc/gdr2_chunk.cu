// Chunked bf16 Gated Delta Rule-2 prefill (tcgen05 / TMA / TMEM) -- placeholder
// until the tensor-core kernel lands; every bf16 call takes the recurrent kernel.
#include "gdr2_internal.cuh"
#include "gdr2.h"

namespace gdr2 {
bool chunked_bf16_supports(const ForwardArgs&) { return false; }
int launch_chunked_bf16(const ForwardArgs&, cudaStream_t, int*) { return GDR2_ERR_UNSUPPORTED; }
}  // namespace gdr2
