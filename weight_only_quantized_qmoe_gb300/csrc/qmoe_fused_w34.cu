// Single-launch decode forward: fc1 3-bit, fc2 4-bit codes.
#include "qmoe_fused.cuh"
namespace qmoe {
template cudaError_t launch_fused_pair<3, 4>(const FusedArgs&, bool, int, int, int, int, cudaStream_t);
}
