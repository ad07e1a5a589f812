// Single-launch decode forward: fc1 4-bit, fc2 3-bit codes.
#include "qmoe_fused.cuh"
namespace qmoe {
template cudaError_t launch_fused_pair<4, 3>(const FusedArgs&, bool, int, int, int, int, cudaStream_t);
}
