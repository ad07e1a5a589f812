// Instantiations of the decode kernel for 1-bit codes.
#include "qmoe_decode_kernel.cuh"

namespace qmoe {
template cudaError_t launch_decode_mma_bits<1>(const DecodeArgs& a, cudaStream_t s);
}  // namespace qmoe
