// Single-launch decode forward: fc1 2-bit, fc2 2-bit codes.
#include "qmoe_fused.cuh"
namespace qmoe {
template cudaError_t launch_fused_pair<2, 2>(const FusedArgs&, bool, int, int, int, int, cudaStream_t);
}
