// Tensor-core grouped GEMM path (prefill): declarations.
#pragma once
#include <cuda.h>

#include "qmoe_internal.cuh"

namespace qmoe {

// GEMM (prefill) prepacked layout of one projection.
//
// A tile is 128 weight rows: fc1 rows interleaved gate/up (tile row 2p = gate
// row nt*64 + p, row 2p+1 = the matching up row), fc2 rows nt*128 + r.  Along
// K the tile is cut into steps of 64; one step is
//   codes : 128 rows x (64*bits/8) bytes; per 32-bit word the two codes of a
//           k pair sit in the low and high 16-bit halves (int3: 2-bit plane
//           words, then 1-bit plane words)
//   scales: 128 rows x nbs values of D (nbs = quantisation blocks in the step)
//   zp    : 128 rows x nbs bytes (uint8 zero points), padded to 16 bytes
// so each step is one contiguous bulk copy.  Rows past N and k past K hold
// zero codes and zero scales (weight 0).
struct GemmLayout {
  int bits, B, ksteps, ntiles, code_row, nbs, zp_bytes, stage_bytes;
  size_t tile_bytes, expert_bytes;
};

GemmLayout make_gemm_layout(int bits, int B, int fc, int N, int K, int I, int zp_mode);

struct GemmRepackArgs {
  const uint8_t* codes;
  const void* scales;
  const uint8_t* zp;
  uint8_t* out;
  int E, N, K, I, fc;
  GemmLayout L;
};
cudaError_t launch_repack_gemm(const GemmRepackArgs& a, cudaStream_t s);

struct GemmArgs {
  const uint8_t* wq;       // GEMM layout
  GemmLayout L;
  const Item* items;       // class-1 work-list (e, start, rows <= 256)
  const int* n_items;
  int max_items;
  int grid;                // persistent CTAs
  int fc, act, zp_mode, bf16;
  float zp_offset;
  void* hout;              // fc1: h [R, I] D (route order)
  float* out_acc;          // fc2: fp32 [T, H] combine accumulator
  const int* perm;
  const float* w;
  int k;
  int N_out;               // I (fc1) or H (fc2)
  WaitCfg wait;
};

cudaError_t make_token_map(CUtensorMap* map, const void* base, int rows, int K, bool bf16);
cudaError_t launch_gemm(const CUtensorMap& map, const GemmArgs& a, cudaStream_t s);
cudaError_t launch_gather(const void* x, const int* perm, int k, int R, int H, void* xg, cudaStream_t s);
cudaError_t launch_finalize_acc(float* acc, void* out, size_t n, int dtype, cudaStream_t s);

}  // namespace qmoe
