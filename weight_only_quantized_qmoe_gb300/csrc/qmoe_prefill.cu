// Tensor-core grouped GEMM for experts with many routed rows (prefill):
// fc1 (+ fused gated activation) and fc2 (+ weighted scatter into the fp32
// combine accumulator) of the QMoE layer forward.
//
// What is computed is the same as the decode path (onnx-runtime-ep-cuda
// src/kernels/qmoe.rs decode_affine_weight; PR "[CUDA] QMoE: fused int2
// mixed-input GEMM ..." zero_point_offset; PR "[CUDA] Add fast INT3 QMoE
// kernels" review "Round dequantized weights before accumulation"), written as
// a dense contraction per (expert, token tile, weight-row tile).
//
// GB300 design (ours; the pages' SM80 DqMma prior art does not apply):
//   D[128 weight rows, N tokens] += A[128 rows, 64 k] * B[N tokens, 64 k]^T
//   * A = dequantised weights, written by CUDA-core warps straight into
//     tensor memory (tcgen05.st, one thread per weight row, 64 k per step;
//     three warp groups take k-steps in turn): the dequant costs no
//     shared-memory bandwidth, which the B stream needs;
//   * B = the routed token rows (x gathered per work item for fc1, h written
//     by fc1's epilogue for fc2), pre-tiled in the MMA's K-major 128-byte
//     swizzle so each 128 x 64 operand tile is one contiguous 16 KB bulk
//     copy (strided 2-D tensor loads of the same tile were ~7x slower to
//     arrive);
//   * tcgen05.mma.cta_group::1.kind::f16, fp32 accumulators in TMEM, two of
//     128 columns so the epilogue of one tile overlaps the next tile's MMAs;
//     N = the tile's rows rounded up to 16, at least 64;
//   * warp roles: 0 = bulk-copy producer, 1 = MMA issuer (the whole warp,
//     one elected lane issues) and TMEM owner, then the dequant groups,
//     then 4 epilogue warps (tcgen05.ld);
//   * persistent CTAs stride over the (item, weight-tile) list; fc1 rows are
//     interleaved gate/up so the GLU pairs sit in adjacent TMEM lanes;
//   * every wait is bounded; a timeout aborts all roles, drains in-flight
//     copies and MMAs, frees TMEM and records QMOE_ERR_TIMEOUT.
#include "qmoe_prefill.cuh"

namespace qmoe {

// ----------------------------------------------------------------------------
// Prepack: canonical -> GEMM layout (see GemmLayout).  One thread per
// (expert, tile, k-step, tile row).
// ----------------------------------------------------------------------------
__device__ __forceinline__ int canon_field(const uint8_t* row, int row_bytes, int bits, int d, int K) {
  if (d >= K) return 0;
  const int bo = d * bits;
  const int byte = bo >> 3, sh = bo & 7;
  uint32_t v = row[byte];
  if (byte + 1 < row_bytes) v |= (uint32_t)row[byte + 1] << 8;
  return (int)((v >> sh) & ((1u << bits) - 1u));
}

__global__ void repack_gemm_kernel(const GemmRepackArgs a) {
  const GemmLayout& L = a.L;
  const size_t total = (size_t)a.E * L.ntiles * L.ksteps * 128;
  const size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int r = (int)(idx % 128);
  const int ks = (int)((idx / 128) % L.ksteps);
  const int nt = (int)((idx / (128 * (size_t)L.ksteps)) % L.ntiles);
  const int e = (int)(idx / (128 * (size_t)L.ksteps * L.ntiles));
  int row;
  bool valid;
  if (a.fc == 1) {
    // tile row 2p = gate of feature n, 2p+1 = its up row; canonical rows
    // concatenated ([gate | up]) or interleaved (gate n = 2n, up n = 2n+1)
    const int n = nt * 64 + r / 2;
    valid = n < a.I;
    row = a.interleaved ? 2 * n + (r & 1) : ((r & 1) ? a.I + n : n);
  } else {
    row = nt * 128 + r;
    valid = row < a.N;
  }
  const int bits = L.bits;
  const int row_bytes = a.K * bits / 8;
  const int nblk = a.K / L.B;
  const int zrow = (nblk * bits + 7) / 8;
  const uint8_t* crow = valid ? a.codes + ((size_t)e * a.N + row) * row_bytes : nullptr;
  auto code = [&](int d) { return valid ? canon_field(crow, row_bytes, bits, d, a.K) : 0; };
  uint8_t* stage = a.out + ((((size_t)e * L.ntiles + nt) * L.ksteps) + ks) * L.stage_bytes;
  uint32_t* cw = reinterpret_cast<uint32_t*>(stage + (size_t)r * L.code_row);
  const int k0 = ks * 64;
  if (bits == 1) {
    // word i: bit m of the low / high half = codes k0 + 32 i + 2 m / + 1
    for (int i = 0; i < 2; ++i) {
      uint32_t w = 0;
      for (int m = 0; m < 16; ++m) {
        w |= (uint32_t)code(k0 + 32 * i + 2 * m) << m;
        w |= (uint32_t)code(k0 + 32 * i + 2 * m + 1) << (16 + m);
      }
      cw[i] = w;
    }
  } else if (bits == 8) {
    // word i: k pairs 2i (bytes 0 and 2) and 2i+1 (bytes 1 and 3)
    for (int i = 0; i < 16; ++i) {
      const int kk = k0 + 4 * i;
      cw[i] = (uint32_t)code(kk) | ((uint32_t)code(kk + 2) << 8) | ((uint32_t)code(kk + 1) << 16) |
              ((uint32_t)code(kk + 3) << 24);
    }
  } else if (bits == 4) {
    for (int i = 0; i < 8; ++i) {
      uint32_t w = 0;
      for (int m = 0; m < 4; ++m) {
        w |= (uint32_t)code(k0 + 8 * i + 2 * m) << (4 * m);
        w |= (uint32_t)code(k0 + 8 * i + 2 * m + 1) << (16 + 4 * m);
      }
      cw[i] = w;
    }
  } else {
    for (int i = 0; i < 4; ++i) {
      uint32_t w = 0;
      for (int m = 0; m < 8; ++m) {
        w |= (uint32_t)(code(k0 + 16 * i + 2 * m) & 3) << (2 * m);
        w |= (uint32_t)(code(k0 + 16 * i + 2 * m + 1) & 3) << (16 + 2 * m);
      }
      cw[i] = w;
    }
    if (bits == 3) {
      for (int i = 0; i < 2; ++i) {
        uint32_t w = 0;
        for (int m = 0; m < 16; ++m) {
          w |= (uint32_t)((code(k0 + 32 * i + 2 * m) >> 2) & 1) << m;
          w |= (uint32_t)((code(k0 + 32 * i + 2 * m + 1) >> 2) & 1) << (16 + m);
        }
        cw[4 + i] = w;
      }
    }
  }
  uint16_t* sc = reinterpret_cast<uint16_t*>(stage + 128 * L.code_row) + (size_t)r * L.nbs;
  uint8_t* zp = stage + 128 * L.code_row + 128 * L.nbs * 2 + (size_t)r * L.nbs;
  for (int b = 0; b < L.nbs; ++b) {
    const int kb = k0 / L.B + b;
    uint16_t s = 0;
    uint8_t z = 0;
    if (valid && kb < nblk) {
      s = reinterpret_cast<const uint16_t*>(a.scales)[((size_t)e * a.N + row) * nblk + kb];
      if (a.zp) z = (uint8_t)canon_field(a.zp + ((size_t)e * a.N + row) * zrow, zrow, bits, kb, nblk);
    }
    sc[b] = s;
    if (L.zp_bytes) zp[b] = z;
  }
}

GemmLayout make_gemm_layout(int bits, int B, int fc, int N, int K, int I, int zp_mode) {
  GemmLayout L;
  L.bits = bits;
  L.B = B;
  L.ksteps = (K + 63) / 64;
  L.ntiles = fc == 1 ? (I + 63) / 64 : (N + 127) / 128;
  L.code_row = 64 * bits / 8;
  L.nbs = B >= 64 ? 1 : 64 / B;
  L.zp_bytes = zp_mode == QMOE_ZP_UINT8 ? ((128 * L.nbs + 15) / 16) * 16 : 0;
  L.stage_bytes = 128 * L.code_row + 128 * L.nbs * 2 + L.zp_bytes;
  L.tile_bytes = (size_t)L.ksteps * L.stage_bytes;
  L.expert_bytes = L.tile_bytes * L.ntiles;
  return L;
}

cudaError_t launch_repack_gemm(const GemmRepackArgs& a, cudaStream_t s) {
  const size_t total = (size_t)a.E * a.L.ntiles * a.L.ksteps * 128;
  if (total == 0) return cudaSuccess;
  const size_t blocks = (total + 255) / 256;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  repack_gemm_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// Gather of x into the tiled token layout (fc1 B operand), and the combine of
// the fp32 accumulator.
// ----------------------------------------------------------------------------
// kGatherParts CTAs per GEMM-class item (grid y); their warps take the item's
// rows in turn; chunks past H (K padding up to 64) and rows past the item's
// count up to the next multiple of 8 (copied with the tile) are written as
// zeros, so the MMA never reads undefined values.
constexpr int kGatherParts = 8;

__global__ void __launch_bounds__(256) gather_tiles_kernel(const void* __restrict__ x, const int* __restrict__ perm,
                                                           int k, int H, const Item* __restrict__ items,
                                                           const int* __restrict__ n_items, uint8_t* __restrict__ xt) {
  pdl_wait();
  if ((int)blockIdx.x >= *n_items) return;
  const Item it = items[blockIdx.x];
  const int ksteps = (H + 63) / 64;
  const int cpr = ksteps * 8;                 // 16-byte chunks per row (padded to 64 values)
  const int hv = H / 8;                       // real chunks per row
  const int rows = (it.rows + 7) & ~7;        // rows up to a multiple of 8 (the copy unit)
  const int lane = threadIdx.x & 31;
  const int nw = (int)gridDim.y * (blockDim.x >> 5);
  const uint4* src = static_cast<const uint4*>(x);
  uint8_t* tile0 = xt + tok_tile_offset(blockIdx.x, ksteps, 0);
  // A warp copies whole rows: one token lookup per row, lanes across the row
  // (coalesced 16-byte loads; each 8-lane group stores one swizzled 128-byte
  // row of a k-step tile).
  constexpr int U = 4;
  for (int row = (int)blockIdx.y * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows; row += nw) {
    const bool real = row < it.rows;
    const uint4* srow = src + (size_t)(real ? perm[it.start + row] / k : 0) * hv;
    uint8_t* drow = tile0 + row * 128;
    for (int c0 = lane; c0 < cpr; c0 += 32 * U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        v[u] = (real && c < hv) ? srow[c] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        if (c < cpr)
          *reinterpret_cast<uint4*>(drow + (size_t)(c >> 3) * kTokTileBytes + (((c & 7) ^ (row & 7)) << 4)) = v[u];
      }
    }
  }
  pdl_launch_dependents();
}

cudaError_t launch_gather_tiles(const void* x, const int* perm, int k, int H, const Item* items,
                                const int* n_items, int max_items, uint8_t* xt, cudaStream_t s) {
  if (max_items <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(max_items, kGatherParts);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gather_tiles_kernel, x, perm, k, H, items, n_items, xt);
}

template <int DT>
__global__ void __launch_bounds__(256) finalize_acc_kernel(float* __restrict__ acc, void* __restrict__ out, size_t n4) {
  pdl_wait();
  float4* a4 = reinterpret_cast<float4*>(acc);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    store_d4<DT>(out, 4 * i, a4[i]);
  }
}

cudaError_t launch_finalize_acc(float* acc, void* out, size_t n, int dtype, cudaStream_t s) {
  const size_t n4 = n / 4;
  int grid = (int)((n4 + 255) / 256);
  if (grid > 152 * 8) grid = 152 * 8;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dtype == QMOE_F16) return cudaLaunchKernelEx(&cfg, finalize_acc_kernel<QMOE_F16>, acc, out, n4);
  if (dtype == QMOE_BF16) return cudaLaunchKernelEx(&cfg, finalize_acc_kernel<QMOE_BF16>, acc, out, n4);
  return cudaLaunchKernelEx(&cfg, finalize_acc_kernel<QMOE_F32>, acc, out, n4);
}

// ----------------------------------------------------------------------------
// tcgen05 / TMA helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// The MMA-issuing code runs on a whole converged warp and the tcgen05
// instructions are predicated on one lane chosen by elect.sync: the operands
// are then warp-uniform values.  Issued from a single divergent lane, the same
// loop reached about half the MMA rate (measured: 119 vs 65 cycles per
// 128x128x16 MMA).
__device__ __forceinline__ void tc_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
// Four K=16 MMAs of one 64-deep k-step from one asm block: A columns a0 + 8j,
// B descriptor start advanced 32 bytes per MMA; the first accumulates into D
// only when `acc` is set, the rest always do.  One elected lane issues.
__device__ __forceinline__ void umma_ts_x4_elect(uint32_t d, uint32_t a0, uint64_t b0, uint32_t idesc,
                                                 uint32_t acc) {
  const uint64_t b1 = b0 + 2, b2 = b0 + 4, b3 = b0 + 6;   // +32 bytes in 16-byte units
  asm volatile(
      "{\n\t.reg .pred e, p0, p1;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %9, 0;\n\t"
      "setp.eq.b32 p1, %9, %9;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %8, p0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %6, %8, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %7, %8, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %10, %8, p1;\n\t}" ::"r"(d),
      "r"(a0), "r"(a0 + 8), "r"(a0 + 16), "r"(a0 + 24), "l"(b0), "l"(b1), "l"(b2), "r"(idesc), "r"(acc),
      "l"(b3)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

#define TC_LD32(taddr, v)                                                                               \
  asm volatile(                                                                                         \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"  \
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                        \
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), \
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),        \
        "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),      \
        "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),      \
        "=r"(v[29]), "=r"(v[30]), "=r"(v[31])                                                           \
      : "r"(taddr)                                                                                      \
      : "memory")

#define TC_ST32(taddr, v)                                                                                \
  asm volatile(                                                                                          \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15," \
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),              \
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), \
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),    \
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),    \
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])                 \
      : "memory")

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);          // start address
  d |= (uint64_t)1 << 16;                           // leading byte offset (unused for SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;                 // stride byte offset
  d |= (uint64_t)1 << 46;                           // descriptor version
  d |= (uint64_t)2 << 61;                           // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: D f32, A/B f16 or bf16, both K-major.
__device__ __forceinline__ uint32_t idesc_f16(bool bf16, int M, int N) {
  uint32_t d = 0;
  d |= 1u << 4;                                     // D = f32
  d |= (bf16 ? 1u : 0u) << 7;                       // A type
  d |= (bf16 ? 1u : 0u) << 10;                      // B type
  d |= (uint32_t)(N >> 3) << 17;
  d |= (uint32_t)(M >> 4) << 24;
  return d;
}

// One poll of a phase whose answer is the same for the whole warp: every lane
// polls, lane 0's answer is broadcast.  (Each lane acting on its own answer
// can split the warp when the phase completes during the poll; the split
// halves would then reach different warp-synchronous instructions.)
__device__ __forceinline__ bool warp_test_wait(uint64_t* bar, uint32_t parity) {
  const int done = mbar_test_wait(bar, parity) ? 1 : 0;
  return __shfl_sync(0xffffffffu, done, 0) != 0;
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const WaitCfg& w,
                                              volatile int* abort_flag) {
  for (long long i = 0; i < w.limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63 && *abort_flag) return false;
  }
  atomicExch(w.status, DEV_TIMEOUT);
  *abort_flag = 1;
  return false;
}

// Bounded wait for a global count (acquire), giving up when another role aborted.
__device__ __forceinline__ bool count_wait_or_abort(const int* p, int target, const WaitCfg& w,
                                                    volatile int* abort_flag) {
  for (long long i = 0; i < w.limit; ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    if ((i & 63) == 63 && *abort_flag) return false;
    __nanosleep(32);
  }
  atomicExch(w.status, DEV_TIMEOUT);
  *abort_flag = 1;
  return false;
}

// Units (of 2 warps x rows) an item's overlapped gather is cut into: enough
// that the first wave's items (the first 152 tiles) are spread over every CTA.
constexpr int kGatherUnits = 32;

// The same with non-blocking polls: for the MMA-issuing thread, whose loop
// paces the whole pipeline (a parked poll costs ~250 cycles even when the
// phase has already completed).
__device__ __forceinline__ bool spin_or_abort(uint64_t* bar, uint32_t parity, const WaitCfg& w,
                                              volatile int* abort_flag) {
  const long long limit = w.limit * 64;
  for (long long i = 0; i < limit; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort_flag) return false;
  }
  atomicExch(w.status, DEV_TIMEOUT);
  *abort_flag = 1;
  return false;
}

// ----------------------------------------------------------------------------
// The grouped GEMM kernel
// ----------------------------------------------------------------------------
// One ring of Ring<>::stages stages: stage s holds KSUB consecutive 64-deep
// k-steps -- their token tiles (B, shared memory), their packed weights (W,
// shared memory, one contiguous copy) and their dequantised weights (A, 32
// TMEM columns per k-step).  Three barriers per stage, one wait per role and
// stage:
//   full[s]  the producer's copies of W and B have landed (transaction count)
//   ready[s] the 4 dequant warps of the stage have written A   (4 arrivals)
//   empty[s] the MMAs of the stage have completed                (tcgen05.commit)
// producer: empty -> copies -> full;  dequant: full -> A -> ready;
// MMA: ready -> MMAs -> commit empty.
constexpr int kTmemCols = 512;
constexpr int kEpiPitch = 36;     // fp32 words per row of an epilogue transpose tile (pad: banks)
constexpr int kEpiBytes = 4 * 32 * kEpiPitch * 4;   // one 32x32 tile per epilogue warp

// The two ring shapes.  A stage holds several 64-deep k-steps, so each
// barrier round, copy and commit covers several k-steps of MMAs (the
// hand-offs, not the MMAs, pace the ring at these shapes).  Prefill items
// carry up to 128 token rows: two 128-column accumulators leave TMEM for 4
// stages of 2 k-steps.  Decode items (T <= 64) carry at most 64 rows: two
// 64-column accumulators leave TMEM for 4 stages of 3 k-steps (6 of 2 for
// 3-bit codes, whose three dequant groups need a ring depth divisible by 3).
// Dequant warp groups (4 warps each; stage step kc -> group kc % groups):
// two, except three for the decode shape's 3-bit codes, whose two-plane
// unpack is the longest dequant (measured: two groups 147 vs three 135 µs on
// the mixed-width fc1; the other widths ran 2-4 % faster with two).
template <bool DEC, int BITS = 4>
struct Ring {
  static constexpr int stages = DEC ? (BITS == 3 ? 6 : 4) : 4;
  static constexpr int ksub = DEC ? (BITS == 3 ? 2 : 3) : 2;   // 64-deep k-steps per stage
  static constexpr int groups = (DEC && BITS == 3) ? 3 : 2;
  static constexpr int epi_warp0 = 4 + 4 * groups;  // first epilogue warp
  static constexpr int threads = (epi_warp0 + 4) * 32;
  static constexpr int tile_n = DEC ? 64 : 128;     // token rows per item (MMA N <= tile_n)
  static constexpr int bsub = tile_n * 128;         // shared bytes of one k-step's token tile
  static constexpr int acc_cols = tile_n;           // accumulators: [0, acc) and [acc, 2 acc)
  static constexpr int acol0 = 2 * acc_cols;        // first TMEM column of the A ring
  static constexpr int a_cols = 32 * ksub;          // A columns per stage
  // Each stage is always dequantised by the same group (stage s -> group
  // s % groups), so a group consumes its stages' phases in order and
  // never runs a ring ahead of a fill that has not landed (a parity test
  // could not tell those apart).
  static_assert(stages % groups == 0, "a stage belongs to one dequant group");
  static_assert(acol0 + stages * a_cols <= kTmemCols, "TMEM columns");
  // shared memory: B ring, W ring (128-byte aligned slots), epilogue tiles, barriers
  __host__ __device__ static int wslot(int stage_bytes) { return (ksub * stage_bytes + 127) / 128 * 128; }
  static constexpr int b_off = 0;
  static constexpr int w_off = stages * ksub * bsub;
  __host__ __device__ static int epi_off(int sb) { return w_off + stages * wslot(sb); }
  __host__ __device__ static int bar_off(int sb) { return epi_off(sb) + kEpiBytes; }
  __host__ __device__ static int total(int sb) { return bar_off(sb) + 1024; }
};

__device__ __forceinline__ void red_add_v4_f32(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

template <int BITS, int ZPM, bool BF16>
__device__ __forceinline__ void dequant_row(const uint8_t* stage, const GemmLayout& L, int r, uint32_t zoff2,
                                            uint32_t* v) {
  constexpr uint32_t MAGIC = BF16 ? 0x43004300u : 0x64006400u;
  const uint8_t* row = stage + r * (64 * BITS / 8);
  constexpr int NW = BITS == 8 ? 16 : (BITS == 4 ? 8 : (BITS == 3 ? 6 : (BITS == 1 ? 2 : 4)));
  uint32_t w[NW];
  if constexpr (BITS == 1) {
    const uint2 q0 = reinterpret_cast<const uint2*>(row)[0];
    w[0] = q0.x; w[1] = q0.y;
  } else if constexpr (BITS == 8) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 q = reinterpret_cast<const uint4*>(row)[i];
      w[4 * i] = q.x; w[4 * i + 1] = q.y; w[4 * i + 2] = q.z; w[4 * i + 3] = q.w;
    }
  } else if constexpr (BITS == 4) {
    const uint4 q0 = reinterpret_cast<const uint4*>(row)[0];
    const uint4 q1 = reinterpret_cast<const uint4*>(row)[1];
    w[0] = q0.x; w[1] = q0.y; w[2] = q0.z; w[3] = q0.w;
    w[4] = q1.x; w[5] = q1.y; w[6] = q1.z; w[7] = q1.w;
  } else if constexpr (BITS == 2) {
    const uint4 q0 = reinterpret_cast<const uint4*>(row)[0];
    w[0] = q0.x; w[1] = q0.y; w[2] = q0.z; w[3] = q0.w;
  } else {
    // 24-byte rows: 8-byte aligned
    const uint2 q0 = reinterpret_cast<const uint2*>(row)[0];
    const uint2 q1 = reinterpret_cast<const uint2*>(row)[1];
    const uint2 q2 = reinterpret_cast<const uint2*>(row)[2];
    w[0] = q0.x; w[1] = q0.y; w[2] = q1.x; w[3] = q1.y; w[4] = q2.x; w[5] = q2.y;
  }
  const uint16_t* sc = reinterpret_cast<const uint16_t*>(stage + 128 * L.code_row) + r * L.nbs;
  const uint8_t* zp = stage + 128 * L.code_row + 128 * L.nbs * 2 + r * L.nbs;
  // Registers 0..15 cover k 0..31 (block 0); registers 16..31 cover k 32..63,
  // block 1 when B = 32 (nbs = 2), else still block 0.  Selecting the second
  // block's scale / zero point once keeps every index below compile-time.
  const int b1 = L.nbs > 1 ? 1 : 0;
  const uint32_t ss0 = (uint32_t)sc[0] * 0x00010001u;
  const uint32_t ss1 = (uint32_t)sc[b1] * 0x00010001u;
  uint32_t zz0 = MAGIC | ((1u << (BITS - 1)) * 0x00010001u), zz1 = zz0;
  if constexpr (BITS == 8) zz0 = zz1 = code8_zq<BF16>(128u);
  if constexpr (ZPM == QMOE_ZP_UINT8) {
    if constexpr (BITS == 8) {
      zz0 = code8_zq<BF16>(zp[0]);
      zz1 = code8_zq<BF16>(zp[b1]);
    } else {
      zz0 = MAGIC | ((uint32_t)zp[0] * 0x00010001u);
      zz1 = MAGIC | ((uint32_t)zp[b1] * 0x00010001u);
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if constexpr (BITS == 8) {
      // word j/2 holds the pairs 2(j/2) and 2(j/2)+1: bytes (0, 2) and (1, 3)
      const uint32_t b = w[j >> 1] >> (8 * (j & 1));
      uint32_t x;
      if constexpr (ZPM == QMOE_ZP_OFFSET && !BF16)
        x = sub2<false>(((b & 0x00FF00FFu) << 1) | Magic<false>::half, zoff2);
      else
        x = code8_minus_zp<BF16>(b, ZPM == QMOE_ZP_OFFSET ? zoff2 : (j < 16 ? zz0 : zz1));
      v[j] = mul2<BF16>(x, j < 16 ? ss0 : ss1);
      continue;
    }
    uint32_t p;
    if constexpr (BITS == 1) p = (w[j >> 4] >> (j & 15)) & 0x00010001u;
    else if constexpr (BITS == 4) p = (w[j >> 2] >> (4 * (j & 3))) & 0x000F000Fu;
    else if constexpr (BITS == 2) p = (w[j >> 3] >> (2 * (j & 7))) & 0x00030003u;
    else p = ((w[j >> 3] >> (2 * (j & 7))) & 0x00030003u) | (((w[4 + (j >> 4)] >> (j & 15)) & 0x00010001u) << 2);
    uint32_t x;
    if constexpr (ZPM == QMOE_ZP_OFFSET) {
      x = sub2<BF16>((p << 1) | Magic<BF16>::half, zoff2);   // exact c - z, half-integer z
    } else {
      x = sub2<BF16>(p | MAGIC, j < 16 ? zz0 : zz1);
    }
    v[j] = mul2<BF16>(x, j < 16 ? ss0 : ss1);
  }
}

// Gated activations for the GEMM epilogue, from exp (CUDA's __expf):
// SwiGLU with its attributes (gate bounded by limit, linear half clamped to
// [-limit, limit], g * sigmoid(alpha g) = g / (1 + e^{-alpha g}), times
// (u + beta)); tanh(y) = 1 - 2 / (e^{2y} + 1) for GeGLU.
__device__ __forceinline__ float glu_fast(const ActParams& p, float g, float u) {
  if (p.act == QMOE_ACT_SWIGLU) {
    g = fminf(g, p.limit);
    if (!isnan(u)) u = fminf(fmaxf(u, -p.limit), p.limit);
    return __fdividef(g, 1.f + __expf(-p.alpha * g)) * (u + p.beta);
  }
  const float y = 0.7978845608028654f * (g + 0.044715f * g * g * g);
  const float t = 1.f - __fdividef(2.f, __expf(2.f * y) + 1.f);
  return 0.5f * g * (1.f + t) * u;
}

// Sources of one tile: its weight tile, its token tile and the first k-step.
// The weight tiles of one token tile run on neighbouring CTAs at the same
// time; starting each at a different k-step (rotation by nt) spreads their
// reads of the shared token tile over the L2 instead of hitting the same lines
// together.  The MMA sums the k-steps in any order.  With several k-steps per
// stage they stay aligned (no rotation): a stage's k-steps are then one
// contiguous weight copy.
struct TileSrc {
  const uint8_t* w;     // k-step kr at w + kr * stage_bytes
  const uint8_t* b;     // k-step kr at b + kr * kTokTileBytes
  uint32_t b_bytes;     // token bytes copied per k-step
  int rot;              // first k-step
};
template <bool DEC, int BITS>
__device__ __forceinline__ TileSrc tile_src(const GemmArgs& a, int tile) {
  const GemmLayout& L = a.L;
  const int item = tile / L.ntiles, nt = tile - item * L.ntiles;
  const Item it = a.items[item];
  TileSrc r;
  r.w = a.wq + (size_t)it.e * L.expert_bytes + (size_t)nt * L.tile_bytes;
  r.b = a.btiles + tok_tile_offset(item, L.ksteps, 0);
  // only the 8-row groups that hold the item's rows (the MMA reads stale
  // rows past them into columns that are never stored)
  r.b_bytes = (uint32_t)min(Ring<DEC, BITS>::bsub, ((it.rows + 7) / 8) * 1024);
  r.rot = Ring<DEC, BITS>::ksub > 1 ? 0 : (int)(((long long)nt * L.ksteps) / L.ntiles);
  return r;
}

__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)), "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s_elect(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Warp roles (8 + 4 * groups warps):
//   0      bulk-copy producer (whole warp, elect.sync): W + B of a stage into slot s
//   1      MMA issuer (whole warp, elect.sync) and TMEM owner
//   2..3   fc1: write the items' token tiles from x (overlapped gather) and
//          clear the fc2 accumulator; otherwise idle
//   4 ..   dequant groups of 4 warps; group g takes stage steps kc % groups == g,
//          warp w owns TMEM lanes 32*(w%4)
//   last 4 epilogue (TMEM lanes 32*(w%4))
// The MMA issuer polls without suspending (it paces the ring); the producer,
// dequant and epilogue warps park on their barriers.
// EPI: 0 = fc2 (weighted combine), 1 = gated fc1 (GLU), 2 = non-gated fc1.
template <int BITS, int ZPM, bool BF16, int EPI, bool DEC>
__global__ void __launch_bounds__((Ring<DEC, BITS>::threads), 1)
    gemm_kernel(const GemmArgs a) {
  constexpr bool GLU = EPI == 1;
  using RG = Ring<DEC, BITS>;
  constexpr int kDeqGroups = RG::groups;
  constexpr int kEpiWarp0 = RG::epi_warp0;
  constexpr int kStages = RG::stages;
  constexpr int KSUB = RG::ksub;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled B tiles
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const GemmLayout& L = a.L;
  const int wslot = RG::wslot(L.stage_bytes);
  uint8_t* bring = smem + RG::b_off;
  uint8_t* wring = smem + RG::w_off;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RG::bar_off(L.stage_bytes));
  uint64_t* full = bars;
  uint64_t* ready = full + kStages;
  uint64_t* empty = ready + kStages;
  uint64_t* acc_full = empty + kStages;      // [2]
  uint64_t* acc_empty = acc_full + 2;        // [2]
  uint64_t* drain_bar = acc_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  // stage steps per tile; the last one of a tile may hold fewer than KSUB k-steps
  const int nss = (L.ksteps + KSUB - 1) / KSUB;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&ready[i], 4);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], 4); }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  // The MMA reads N >= 64 token rows of a k-step, more than a small item
  // copies; the rows past the copy must hold finite values (zero here, or
  // rows of an earlier copy), never undefined shared memory.
  for (int i = threadIdx.x; i < kStages * KSUB * RG::bsub / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(bring)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  pdl_wait();
  const int n_items = *a.n_items;
  const int total_tiles = n_items * L.ntiles;

  if (warp == 0) {
    // ---------------- producer: the whole warp, one elected lane copies ----------------
    int kc = 0, issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
      // (An L2 bulk prefetch a ring's depth ahead of each copy made the
      // kernel twice as slow: the copies queue behind the prefetches.)
      const TileSrc src = tile_src<DEC, BITS>(a, tile);
      if (a.gx) {
        // the item's token tile is written by the gathering warps (of any
        // CTA): wait for all of its units, then make those generic-proxy
        // writes visible to this thread's bulk copies
        int okw = 1;
        if (lane == 0)
          okw = count_wait_or_abort(a.gready + tile / L.ntiles, 2 * kGatherUnits, a.wait, abort_flag) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, okw, 0) != 0;
        if (!ok) break;
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      int kr = src.rot;
      for (int j = 0; j < nss; ++j, ++kc) {
        const int s = kc % kStages;
        const uint32_t par = ((uint32_t)(kc / kStages) & 1u) ^ 1u;
        const int nk = KSUB == 1 ? 1 : min(KSUB, L.ksteps - j * KSUB);
        // Parked (not spinning) wait: the producer runs a ring's depth ahead
        // of the MMAs, and a spinning poll competes with them for the
        // barrier unit.  The first poll is one warp-wide instruction (a
        // lane-0 broadcast here cost 4-9 % of the kernel time).
        if (!mbar_test_wait(&empty[s], par)) {
          ok = wait_or_abort(&empty[s], par, a.wait, abort_flag);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
        mbar_arrive_expect_tx_elect(&full[s], (uint32_t)nk * ((uint32_t)L.stage_bytes + src.b_bytes));
        // Test hook: stage 0's barrier is armed but its copies are never
        // issued, so the waits on it can only run out (host-injected failure).
        if (!(a.inject_stall && kc == 0)) {
          // the stage's k-steps are consecutive in the weight tile: one copy
          bulk_g2s_elect(wring + s * wslot, src.w + (size_t)kr * L.stage_bytes, (uint32_t)(nk * L.stage_bytes),
                         &full[s]);
#pragma unroll
          for (int h = 0; h < KSUB; ++h)
            if (h < nk)
              bulk_g2s_elect(bring + (s * KSUB + h) * RG::bsub, src.b + (size_t)(kr + h) * kTokTileBytes,
                             src.b_bytes, &full[s]);
        }
        issued = kc + 1;
        kr += nk;
        if (kr == L.ksteps) kr = 0;
      }
    }
    if (!ok) {
      // Drain: the last copy issued into each stage must land before the CTA
      // leaves (fixed large bound).  A stage's phase completes on the bytes
      // alone, whatever the consumers did.
      const WaitCfg drain{a.wait.status, kDrainWaitLimit};
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i) {
        if (a.inject_stall && i == 0) continue;   // no copy was issued for it
        mbar_wait_bounded(&full[i % kStages], (i / kStages) & 1, drain);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: the whole warp, one elected lane issues ----------------
    const uint32_t a0 = tmem + RG::acol0;
    const uint64_t bdesc0 = smem_desc_sw128(smem_u32(bring));
    int st = 0, tc = 0;       // ring stage of the next stage step, tile count
    uint32_t ph = 0;          // phase parity of that stage's current use
    bool ok = true;
    for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++tc) {
      const Item it = a.items[tile / L.ntiles];
      // N >= 64: below that the MMA takes as long as at 64 (measured) and
      // the extra columns are never stored
      const int N = max(64, (it.rows + 15) & ~15);
      const uint32_t idesc = idesc_f16(BF16, 128, N);
      const int ab = tc & 1;
      ok = spin_or_abort(&acc_empty[ab], ((tc >> 1) & 1) ^ 1, a.wait, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t dacc = tmem + ab * RG::acc_cols;
      // The stage-step loop is unrolled over the ring stage u, so every
      // stage's operands are compile-time offsets from a0 / bdesc0 and the
      // code between two MMA batches is a single barrier poll and a commit:
      // with more work there (index arithmetic, a general wait loop) the
      // tensor pipe idled between batches (measured: 257 vs 700 cycles per
      // k-step).
      int j = 0;
      while (j < nss && ok) {
#pragma unroll
        for (int u = 0; u < kStages; ++u) {
          if (u == st && j < nss && ok) {
            if (!warp_test_wait(&ready[u], ph)) {
              ok = spin_or_abort(&ready[u], ph, a.wait, abort_flag);
              ok = __shfl_sync(0xffffffffu, ok, 0);
            }
            if (ok) {
              tc_fence_after();
              const int nk = KSUB == 1 ? 1 : min(KSUB, L.ksteps - j * KSUB);
#pragma unroll
              for (int h = 0; h < KSUB; ++h)
                if (h < nk)
                  umma_ts_x4_elect(dacc, a0 + RG::a_cols * u + 32 * h,
                                   bdesc0 + (uint64_t)(((u * KSUB + h) * RG::bsub) >> 4), idesc,
                                   (j != 0 || h != 0) ? 1u : 0u);
              tc_commit_elect(&empty[u]);
              ++j;
              if (++st == kStages) {
                st = 0;
                ph ^= 1u;
              }
            }
          }
        }
      }
      if (ok) tc_commit_elect(&acc_full[ab]);
    }
    // All MMAs issued by this warp have completed once drain_bar flips.
    tc_commit_elect(drain_bar);
    const WaitCfg drain{a.wait.status, kDrainWaitLimit};
    mbar_wait_bounded(drain_bar, 0, drain);
  } else if (warp == 2 || warp == 3) {
    // ---------------- fc1: the token tiles from x, overlapped with the MMAs ----------------
    // Unit u = (item u / kGatherUnits, part u % kGatherUnits) goes to CTA
    // u % gridDim.x, so the first wave's items are written by many CTAs at
    // once.  A part is 2 x RPW rows, RPW per warp: a warp copies whole rows
    // (one token lookup per row, lanes across the row, 16-byte loads, each
    // 8-lane group storing one swizzled 128-byte row of a k-step tile), rows
    // past the item's count up to the next multiple of 8 and chunks past H
    // as zeros.  Then (with or without the gather) the fc2 accumulator is
    // cleared, a slice per CTA.
    if (a.gx) {
      constexpr int RPW = RG::tile_n / (2 * kGatherUnits);
      // 16-byte loads in flight per lane (a 4096-wide row per pass); the
      // decode ring shape never gathers (and has fewer registers to spare)
      constexpr int U = DEC ? 4 : 16;
      const int cpr = L.ksteps * 8;
      const int hv = a.gH / 8;
      const uint4* xsrc = static_cast<const uint4*>(a.gx);
      const int nunits = n_items * kGatherUnits;
      for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
        const int item = u / kGatherUnits, part = u - item * kGatherUnits;
        const Item it = a.items[item];
        const int rows8 = (it.rows + 7) & ~7;
        uint8_t* tile0 = const_cast<uint8_t*>(a.btiles) + tok_tile_offset(item, L.ksteps, 0);
        for (int rr = 0; rr < RPW; ++rr) {
          const int row = part * 2 * RPW + (warp - 2) * RPW + rr;
          if (row >= rows8) break;
          const bool real = row < it.rows;
          const uint4* srow = xsrc + (size_t)(real ? a.perm[it.start + row] / a.k : 0) * hv;
          uint8_t* drow = tile0 + row * 128;
          for (int c0 = lane; c0 < cpr; c0 += 32 * U) {
            uint4 v[U];
#pragma unroll
            for (int q = 0; q < U; ++q) {
              const int c = c0 + 32 * q;
              v[q] = (real && c < hv) ? srow[c] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int q = 0; q < U; ++q) {
              const int c = c0 + 32 * q;
              if (c < cpr)
                *reinterpret_cast<uint4*>(drow + (size_t)(c >> 3) * kTokTileBytes + (((c & 7) ^ (row & 7)) << 4)) =
                    v[q];
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __threadfence();
          atomicAdd(a.gready + item, 1);
        }
      }
    }
    if (a.zacc) {
      const size_t n4 = a.zacc_n4;
      const size_t i0 = n4 * blockIdx.x / gridDim.x, i1 = n4 * (blockIdx.x + 1) / gridDim.x;
      float4* z4 = reinterpret_cast<float4*>(a.zacc);
      for (size_t i = i0 + (size_t)(warp - 2) * 32 + lane; i < i1; i += 64) z4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  } else if (warp >= 4 && warp < kEpiWarp0) {
    // ---------------- dequant: packed weights -> 16-bit pairs in TMEM ----------------
    // full[s] also means the A slot is free: the producer refilled stage s
    // only after the MMAs that read it had completed (empty[s]).
    const int q = warp & 3;
    const int grp = (warp - 4) >> 2;      // dequant group
    const int r = q * 32 + lane;          // TMEM lane = weight row of the tile
    // offset zero point: the half-unit magic pair, or for bf16 8-bit codes
    // (whose accepted offsets are integers) the pair (z, z)
    uint32_t zoff2 = 0u;
    if constexpr (ZPM == QMOE_ZP_OFFSET)
      zoff2 = (BITS == 8 && BF16) ? (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a.zp_offset)) * 0x00010001u
                                  : half_magic_offset<BF16>(a.zp_offset);
    // stage steps are numbered across tiles (kc); this group takes kc = grp,
    // grp + kDeqGroups, ...
    const int n_steps = ((total_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x) * nss;
    bool ok = true;
    for (int kc = grp; kc < n_steps && ok; kc += kDeqGroups) {
      // kStages is a multiple of kDeqGroups, so every use of stage s falls
      // to this one group, in order: the parity of full[s] names one phase.
      const int s = kc % kStages;
      ok = wait_or_abort(&full[s], (kc / kStages) & 1, a.wait, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int jj = KSUB == 1 ? 0 : kc % nss;
      const int nk = KSUB == 1 ? 1 : min(KSUB, L.ksteps - jj * KSUB);
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + RG::acol0 + s * RG::a_cols;
#pragma unroll
      for (int h = 0; h < KSUB; ++h) {
        if (h < nk) {
          uint32_t v[32];
          dequant_row<BITS, ZPM, BF16>(wring + s * wslot + h * L.stage_bytes, L, r, zoff2, v);
          TC_ST32(taddr + 32 * h, v);
          tc_wait_st();   // v is reused by the next k-step of the stage
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ready[s]);
    }
  } else if (warp >= kEpiWarp0) {
    // ---------------- epilogue: TMEM -> GLU / act -> h (fc1) | weighted scatter (fc2) ----------------
    // Each warp owns TMEM lanes 32q..32q+31 (its 32 weight rows) and a 32x32
    // shared tile in which it turns its (row, token) values around, so that
    // global memory sees 16-byte stores (fc1) / 16-byte reductions (fc2)
    // along the contiguous feature axis.
    const int q = warp & 3;
    float* tile32 = reinterpret_cast<float*>(smem + RG::epi_off(L.stage_bytes)) + q * 32 * kEpiPitch;
    int tc = 0;
    bool ok = true;
    constexpr int NCH = RG::tile_n / 32;   // 32-token chunks of a tile
    for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++tc) {
      const Item it = a.items[tile / L.ntiles];
      const int nt = tile % L.ntiles;
      const int ab = tc & 1;
      // fc2 scatter: the token and weight of each of this lane's token
      // columns, loaded while the tile's MMAs still run
      int tok_c[NCH];
      float w_c[NCH];
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        tok_c[ch] = 0;
        w_c[ch] = 0.f;
        if (EPI == 0 && !a.ybuf && ch * 32 + lane < it.rows) tok_c[ch] = a.perm[it.start + ch * 32 + lane];
      }
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        if (EPI == 0 && !a.ybuf && ch * 32 + lane < it.rows) {
          w_c[ch] = a.w[tok_c[ch]];
          tok_c[ch] /= a.k;
        }
      }
      ok = wait_or_abort(&acc_full[ab], (tc >> 1) & 1, a.wait, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      for (int c0 = 0; c0 < it.rows; c0 += 32) {
        uint32_t v[32];
        TC_LD32(tmem + ((uint32_t)(q * 32) << 16) + ab * RG::acc_cols + c0, v);
        // token and weight of token column c0 + lane
        int my_tok = 0;
        float my_w = 0.f;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch)
          if (ch * 32 == c0) {
            my_tok = tok_c[ch];
            my_w = w_c[ch];
          }
        const bool col_ok = c0 + lane < it.rows;
        __syncwarp();   // converged again before the warp-wide tcgen05.wait
        tc_wait_ld();
        if (GLU) {
          // lanes 2p / 2p+1 hold gate / up of feature n = nt*64 + q*16 + p
          const bool odd = lane & 1;
          const int jbeg = odd ? 16 : 0;
          if (a.bias) {   // fp32 projection bias of this lane's row (gate or up of n)
            const int n = nt * 64 + q * 16 + (lane >> 1);
            const float b = n < a.N_out ? a.bias[((size_t)it.e * a.N_out + n) * 2 + (lane & 1)] : 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + b);
          }
          uint16_t* t16 = reinterpret_cast<uint16_t*>(tile32);   // [32 tokens][16 features]
          // Even lanes take tokens 0..15 of the chunk (own gate, partner's
          // up), odd lanes tokens 16..31 (partner's gate, own up): one
          // exchange and one activation per lane and token pair, no divergence.
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float lo = __uint_as_float(v[j]), hi = __uint_as_float(v[16 + j]);
            const float other = __shfl_xor_sync(0xffffffffu, odd ? lo : hi, 1);
            const float h = glu_fast(a.act, odd ? other : lo, odd ? hi : other);
            t16[(jbeg + j) * 16 + (lane >> 1)] = BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(h))
                                                      : __half_as_ushort(__float2half_rn(h));
          }
          __syncwarp();
          // h chunk (token c0+tok, features nbase + 8*hv .. +7) -> tiled token
          // layout of fc2's B operand; chunks past I are the K padding: zeros.
          const int nbase = nt * 64 + q * 16;
          const int item = tile / L.ntiles;
#pragma unroll
          for (int u2 = 0; u2 < 2; ++u2) {
            const int vec = lane + 32 * u2, tok = vec >> 1, hv = vec & 1;
            const int c = c0 + tok, n = nbase + 8 * hv;
            // rows up to the next multiple of 8 are copied with the tile:
            // the ones past the item's count are written as zeros
            if (c < ((it.rows + 7) & ~7) && n < a.h_ksteps * 64) {
              uint4 val = make_uint4(0u, 0u, 0u, 0u);
              if (c < it.rows && n < a.N_out) val = *reinterpret_cast<const uint4*>(t16 + tok * 16 + hv * 8);
              uint8_t* dst = a.htiles + tok_tile_offset(item, a.h_ksteps, n >> 6) + c * 128 +
                             ((((n & 63) >> 3) ^ (c & 7)) << 4);
              *reinterpret_cast<uint4*>(dst) = val;
            }
          }
          __syncwarp();
        } else {
          // transpose: tile32[token j][row] = D[row][c0 + j] (+ the row's fp32 bias)
          const int mrow = nt * 128 + q * 32 + lane;
          const float b = a.bias && mrow < a.N_out ? a.bias[(size_t)it.e * a.N_out + mrow] : 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) tile32[j * kEpiPitch + lane] = __uint_as_float(v[j]) + b;
          __syncwarp();
          const int mbase = nt * 128 + q * 32;
          const float* src = tile32 + lane * kEpiPitch;
          if (EPI == 0) {
            if (col_ok && mbase < a.N_out) {
              if (a.ybuf) {
                // slot-ordered combine later: the y row of this route, grouped order
                float* dst = a.ybuf + (size_t)(it.start + c0 + lane) * a.N_out + mbase;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  *reinterpret_cast<float4*>(dst + 4 * i) = *reinterpret_cast<const float4*>(src + 4 * i);
              } else {
                float* dst = a.out_acc + (size_t)my_tok * a.N_out + mbase;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float4 y = *reinterpret_cast<const float4*>(src + 4 * i);
                  red_add_v4_f32(dst + 4 * i, my_w * y.x, my_w * y.y, my_w * y.z, my_w * y.w);
                }
              }
            }
          } else {
            // non-gated fc1: h = act(fc1 output) of token c0 + lane, features
            // mbase .. mbase + 31 -> the tiled token layout of fc2's B operand
            // (rows up to the next multiple of 8 and features past I as zeros)
            const int c = c0 + lane, item = tile / L.ntiles;
            if (c < ((it.rows + 7) & ~7)) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int n = mbase + 8 * i;
                if (n < a.h_ksteps * 64) {
                  uint32_t w4[4] = {0u, 0u, 0u, 0u};
                  if (c < it.rows && n < a.N_out) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                      const float h0 = act_single(a.act, src[8 * i + 2 * m]);
                      const float h1 = act_single(a.act, src[8 * i + 2 * m + 1]);
                      const uint32_t lo = BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(h0))
                                               : __half_as_ushort(__float2half_rn(h0));
                      const uint32_t hi = BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(h1))
                                               : __half_as_ushort(__float2half_rn(h1));
                      w4[m] = lo | (hi << 16);
                    }
                  }
                  uint8_t* dst = a.htiles + tok_tile_offset(item, a.h_ksteps, n >> 6) + c * 128 +
                                 ((((n & 63) >> 3) ^ (c & 7)) << 4);
                  *reinterpret_cast<uint4*>(dst) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
              }
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
  }
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
template <int BITS, int ZPM, bool BF16, int EPI, bool DEC>
static cudaError_t launch_g(const GemmArgs& a, cudaStream_t s) {
  const int smem = Ring<DEC, BITS>::total(a.L.stage_bytes) + 1024;  // + alignment slack
  auto kern = gemm_kernel<BITS, ZPM, BF16, EPI, DEC>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(Ring<DEC, BITS>::threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int BITS, int ZPM, bool BF16, int EPI>
static cudaError_t launch_g_ring(const GemmArgs& a, cudaStream_t s) {
  return a.dec ? launch_g<BITS, ZPM, BF16, EPI, true>(a, s) : launch_g<BITS, ZPM, BF16, EPI, false>(a, s);
}
template <int BITS, int ZPM, bool BF16>
static cudaError_t launch_g_glu(const GemmArgs& a, cudaStream_t s) {
  if (a.fc != 1) return launch_g_ring<BITS, ZPM, BF16, 0>(a, s);
  return act_gated(a.act.act) ? launch_g_ring<BITS, ZPM, BF16, 1>(a, s) : launch_g_ring<BITS, ZPM, BF16, 2>(a, s);
}
template <int BITS, int ZPM>
static cudaError_t launch_g_dt(const GemmArgs& a, cudaStream_t s) {
  return a.bf16 ? launch_g_glu<BITS, ZPM, true>(a, s) : launch_g_glu<BITS, ZPM, false>(a, s);
}
template <int BITS>
static cudaError_t launch_g_zp(const GemmArgs& a, cudaStream_t s) {
  if (a.zp_mode == QMOE_ZP_UINT8) return launch_g_dt<BITS, QMOE_ZP_UINT8>(a, s);
  if (a.zp_mode == QMOE_ZP_OFFSET) return launch_g_dt<BITS, QMOE_ZP_OFFSET>(a, s);
  return launch_g_dt<BITS, QMOE_ZP_SYMMETRIC>(a, s);
}

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s) {
  if (a.max_items <= 0 || a.grid <= 0) return cudaSuccess;
  switch (a.L.bits) {
    case 1: return launch_g_zp<1>(a, s);
    case 2: return launch_g_zp<2>(a, s);
    case 3: return launch_g_zp<3>(a, s);
    case 4: return launch_g_zp<4>(a, s);
    case 8: return launch_g_zp<8>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmoe
