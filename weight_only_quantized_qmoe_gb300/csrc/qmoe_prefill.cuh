// Tensor-core grouped GEMM path (prefill): declarations.
#pragma once

#include "qmoe_internal.cuh"

namespace qmoe {

// GEMM (prefill) prepacked layout of one projection.
//
// A tile is 128 weight rows: fc1 rows interleaved gate/up (tile row 2p = gate
// row nt*64 + p, row 2p+1 = the matching up row), fc2 rows nt*128 + r.  Along
// K the tile is cut into steps of 64; one step is
//   codes : 128 rows x (64*bits/8) bytes; per 32-bit word the two codes of a
//           k pair sit in the low and high 16-bit halves (int3: 2-bit plane
//           words, then 1-bit plane words; int8: word i holds the pairs 2i in
//           bytes 0 and 2 and 2i+1 in bytes 1 and 3; 1-bit: bit m of word i's
//           low / high half holds codes 32i + 2m / 32i + 2m + 1)
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
  int interleaved;          // fc1 canonical rows: 0 = [gate | up], 1 = (gate f, up f) pairs
  GemmLayout L;
};
cudaError_t launch_repack_gemm(const GemmRepackArgs& a, cudaStream_t s);

// Tiled token layout (the B operand of the grouped GEMM).  Work item i of the
// GEMM class owns block i: for each k-step s of 64 values, 128 token rows of
// 128 bytes, the 16-byte chunk c of row r stored at chunk position
// c ^ (r & 7) -- the K-major 128-byte-swizzle layout the MMA reads -- so one
// (item, k-step) operand tile is one contiguous 16 KB bulk copy.
constexpr int kTokTileBytes = 128 * 128;
__host__ __device__ inline size_t tok_tile_offset(int item, int ksteps, int s) {
  return ((size_t)item * ksteps + s) * kTokTileBytes;
}

struct GemmArgs {
  const uint8_t* wq;       // GEMM layout
  GemmLayout L;
  const Item* items;       // class-1 work-list (e, start, rows <= 128; <= 64 when dec)
  const int* n_items;
  int max_items;
  int grid;                // persistent CTAs
  int dec;                 // every item has <= 64 rows: the decode ring shape (128-deep stages)
  int fc, zp_mode, bf16;
  ActParams act;
  const float* bias;       // fc1: [E, I, 2] (gate, up) pairs ; fc2: [E, H] ; or null
  float zp_offset;
  const uint8_t* btiles;   // B operand in the tiled token layout (L.ksteps steps per item)
  // fc1 with the gather overlapped (prefill shapes): the kernel's two
  // otherwise idle warps write btiles from x themselves, one (item, part)
  // unit at a time spread over the CTAs, and count each item's finished
  // units in gready; the producer waits for an item's count before its first
  // copy from it.  (Decode shapes gather in a kernel of their own first:
  // there the overlap measured slower.)
  const void* gx;          // x [T, gH] 16-bit, or null: btiles is already written
  int gH;
  int* gready;             // [max_items] unit counts, zero at launch
  float* zacc;             // fc1: the fc2 accumulator to clear meanwhile (zacc_n4 float4), or null
  size_t zacc_n4;
  uint8_t* htiles;         // fc1: h written in the tiled token layout for fc2
  int h_ksteps;            // fc1: k-steps of h (ceil(I / 64))
  float* out_acc;          // fc2: fp32 [T, H] combine accumulator (fp32 reductions of w * y)
  float* ybuf;             // fc2, or null: y rows [R, H] fp32 in grouped order instead, for the
                           // slot-ordered (deterministic) combine
  const int* perm;
  const float* w;
  int k;
  int N_out;               // I (fc1) or H (fc2)
  WaitCfg wait;
  int inject_stall;         // test hook: arm the first stage's barrier, never issue its copies
};

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s);
// x rows of every GEMM-class item into the tiled token layout (K = H padded
// to 64 with zeros).
cudaError_t launch_gather_tiles(const void* x, const int* perm, int k, int H, const Item* items,
                                const int* n_items, int max_items, uint8_t* xt, cudaStream_t s);
cudaError_t launch_finalize_acc(float* acc, void* out, size_t n, int dtype, cudaStream_t s);

}  // namespace qmoe
