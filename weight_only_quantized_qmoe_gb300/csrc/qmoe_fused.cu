// Host side of the single-launch decode forward: which layers and token
// counts it serves, the item shape and the dispatch to the width pairs
// instantiated in qmoe_fused_w*.cu.
#include "qmoe_fused.cuh"

namespace qmoe {

#define QMOE_FUSED_PAIR(b1, b2) \
  extern template cudaError_t launch_fused_pair<b1, b2>(const FusedArgs&, bool, int, int, int, cudaStream_t);
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

int fused_smem_bytes(int R, int E, int Kp_max) {
  return fused_plan(R, E, fused_bop_bytes(Kp_max)).total;
}

// Tiles per item (tpi) and K-splits (ks = 8 / tpi): the largest tpi that
// still leaves about three items per CTA for the expected row groups, with
// every warp holding at least two super-chunks where possible.
void fused_item_shape(int ntiles, int nkc, long long nrg_est, int grid, int* tpi, int* ks) {
  for (int t : {8, 4, 2}) {
    const int k = 8 / t;
    if (nkc < 2 * k) continue;
    if (nrg_est * ((ntiles + t - 1) / t) >= 3LL * grid) {
      *tpi = t;
      *ks = k;
      return;
    }
  }
  // few items: split K as far as the super-chunks allow
  int k = 8;
  while (k > 1 && nkc < 2 * k) k /= 2;
  *ks = k;
  *tpi = 8 / k;
}

cudaError_t launch_fused(const FusedArgs& a, int b1, int b2, bool bf16, int sc, int grid, int smem,
                         cudaStream_t s) {
  switch (b1 * 10 + b2) {
    case 22: return launch_fused_pair<2, 2>(a, bf16, sc, grid, smem, s);
    case 23: return launch_fused_pair<2, 3>(a, bf16, sc, grid, smem, s);
    case 24: return launch_fused_pair<2, 4>(a, bf16, sc, grid, smem, s);
    case 32: return launch_fused_pair<3, 2>(a, bf16, sc, grid, smem, s);
    case 33: return launch_fused_pair<3, 3>(a, bf16, sc, grid, smem, s);
    case 34: return launch_fused_pair<3, 4>(a, bf16, sc, grid, smem, s);
    case 42: return launch_fused_pair<4, 2>(a, bf16, sc, grid, smem, s);
    case 43: return launch_fused_pair<4, 3>(a, bf16, sc, grid, smem, s);
    case 44: return launch_fused_pair<4, 4>(a, bf16, sc, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmoe
