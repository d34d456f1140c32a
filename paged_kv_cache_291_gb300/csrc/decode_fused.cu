// decode_fused.cu -- the fused decode step's variant of the decode kernel
// (pkv_decode_step: each sequence's new row is stored and attended in the
// same launch), instantiated in a translation unit of its own so that it
// compiles beside the plain variant.
#include "decode_kernel.cuh"
#include "pkv_internal.h"

namespace pkv {

cudaError_t launch_decode_fused(const DecodeArgs& a, bool stall, cudaStream_t stream) {
    return launch_decode_t<true>(a, stall, stream);
}

}  // namespace pkv
