// Host side of the single-launch decode forward: which layers and token
// counts it serves, the item shape and the dispatch to the width pairs
// instantiated in qmoe_fused_w*.cu.
#include "qmoe_fused.cuh"

namespace qmoe {

#define QMOE_FUSED_PAIR(b1, b2) \
  extern template cudaError_t launch_fused_pair<b1, b2>(const FusedArgs&, bool, int, int, int, int, cudaStream_t);
QMOE_FUSED_PAIR(2, 2)
QMOE_FUSED_PAIR(2, 3)
QMOE_FUSED_PAIR(2, 4)
QMOE_FUSED_PAIR(3, 2)
QMOE_FUSED_PAIR(3, 3)
QMOE_FUSED_PAIR(3, 4)
QMOE_FUSED_PAIR(4, 2)
QMOE_FUSED_PAIR(4, 3)
QMOE_FUSED_PAIR(4, 4)
#undef QMOE_FUSED_PAIR

bool fused_widths_supported(int b1, int b2) {
  auto ok = [](int b) { return b == 2 || b == 3 || b == 4; };
  return ok(b1) && ok(b2);
}

bool fused_ring_shape(int budget, int fixed_bytes, int warps, int scb1, int scb2, int* sb, int* g1, int* g2) {
  const int per = (budget - fixed_bytes) / (warps * kFusedStages);
  const int s = per / 16 * 16;
  const int mx = scb1 > scb2 ? scb1 : scb2;
  if (s < mx) return false;
  // one stage = as many whole super-chunks as fit, capped near 4 KB so every
  // warp keeps several stages in flight
  const int cap = s < 4096 ? s : 4096;
  *g1 = cap / scb1 > 0 ? cap / scb1 : 1;
  *g2 = cap / scb2 > 0 ? cap / scb2 : 1;
  const int need = (*g1 * scb1 > *g2 * scb2 ? *g1 * scb1 : *g2 * scb2);
  *sb = (need + 15) / 16 * 16;
  return true;
}

cudaError_t launch_fused(const FusedArgs& a, int b1, int b2, bool bf16, int sc, int grid, int warps, int smem,
                         cudaStream_t s) {
  switch (b1 * 10 + b2) {
    case 22: return launch_fused_pair<2, 2>(a, bf16, sc, grid, warps, smem, s);
    case 23: return launch_fused_pair<2, 3>(a, bf16, sc, grid, warps, smem, s);
    case 24: return launch_fused_pair<2, 4>(a, bf16, sc, grid, warps, smem, s);
    case 32: return launch_fused_pair<3, 2>(a, bf16, sc, grid, warps, smem, s);
    case 33: return launch_fused_pair<3, 3>(a, bf16, sc, grid, warps, smem, s);
    case 34: return launch_fused_pair<3, 4>(a, bf16, sc, grid, warps, smem, s);
    case 42: return launch_fused_pair<4, 2>(a, bf16, sc, grid, warps, smem, s);
    case 43: return launch_fused_pair<4, 3>(a, bf16, sc, grid, warps, smem, s);
    case 44: return launch_fused_pair<4, 4>(a, bf16, sc, grid, warps, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmoe
