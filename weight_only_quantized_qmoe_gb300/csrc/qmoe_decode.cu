// Weight-streaming expert projections for experts with few routed rows
// (decode).  fc1 and fc2 of the QMoE layer forward.
//
// What is computed (onnx-runtime-ep-cuda src/kernels/qmoe.rs, CUDA_SRC
// qmoe_linear_impl / decode_affine_weight; zero_point_offset from the PR
// "[CUDA] QMoE: fused int2 mixed-input GEMM + GeGLU activation + fractional
// zero-point"; weight rounding from the PR "[CUDA] Add fast INT3 QMoE
// kernels", review "Round dequantized weights before accumulation"):
//   W[n, d] = R_D((code - zp) * scale[n, d / B]),  acc = sum_d W[n, d] x[d]
// with fp32 accumulation; fc1 fuses the gated activation h = act(gate) * up.
//
// GB300 design (ours, not the pages' SM80 interleaved GEMV):
//   * prepack re-lays every 16-row tile in mma.sync fragment order, split in
//     super-chunks of max(64, B) values along K, scales (and packed zero
//     points) interleaved right after the codes they belong to, so each
//     tile's weights are ONE contiguous byte stream;
//   * each warp streams its tile with 1-D bulk copies (cp.async.bulk, TMA
//     engine) into a private ring of shared-memory stages completed by
//     mbarriers (bounded waits), so many KB per SM are in flight with no
//     register cost;
//   * codes become 16-bit pairs with one LOP (magic-exponent trick), then
//     packed sub (c - zp, exact) and mul (one RNE rounding into D) -- exactly
//     the rounded weight of the definition -- and feed mma.m16n8k16 with
//     fp32 accumulation; tokens (<= 32) are the N side;
//   * the routed rows of the expert (x for fc1, h for fc2) are staged once
//     per CTA in shared memory in B-fragment order;
//   * split-K across the warps of a CTA when there are few tiles.
#include "qmoe_internal.cuh"

namespace qmoe {

DecodeLayout make_decode_layout(int bits, int B, int N_rows_per_sub, int K, int nsub,
                                int zp_mode, int dsize) {
  DecodeLayout L;
  L.bits = bits;
  L.B = B;
  L.SC = B > 64 ? B : 64;
  L.nkc = (K + L.SC - 1) / L.SC;
  L.nsub = nsub;
  L.ntiles = N_rows_per_sub / 16;
  L.code_bytes = 16 * L.SC * bits / 8;
  const int nb = L.SC / B;
  L.scale_bytes = nb * 8 * 2 * dsize;
  // uint8 zero points of rows g and g+8 per block: two nibbles in one byte,
  // or two bytes for 8-bit codes
  L.zp_bytes = zp_mode == QMOE_ZP_UINT8 ? ((nb * (bits == 8 ? 16 : 8) + 15) / 16) * 16 : 0;
  L.scb = nsub * (L.code_bytes + L.scale_bytes + L.zp_bytes);
  L.tile_bytes = (size_t)L.nkc * L.scb;
  L.expert_bytes = L.tile_bytes * L.ntiles;
  return L;
}

// ----------------------------------------------------------------------------
// Repack: canonical -> decode layout.  One CTA per (expert, tile, super-chunk).
// ----------------------------------------------------------------------------
__device__ __forceinline__ int canon_code(const uint8_t* row, int row_bytes, int bits, int d,
                                          int K) {
  if (d >= K) return 0;
  const int bo = d * bits;
  const int byte = bo >> 3, sh = bo & 7;
  uint32_t v = row[byte];
  if (byte + 1 < row_bytes) v |= (uint32_t)row[byte + 1] << 8;
  return (int)((v >> sh) & ((1u << bits) - 1u));
}

__global__ void repack_decode_kernel(const RepackArgs a) {
  const DecodeLayout& L = a.L;
  const int kc = blockIdx.x % L.nkc;
  const int tile = (blockIdx.x / L.nkc) % L.ntiles;
  const int e = blockIdx.x / (L.nkc * L.ntiles);
  const int bits = L.bits;
  const int row_bytes = a.K * bits / 8;
  const int nblk_row = a.K / L.B;
  const int zrow_bytes = (nblk_row * bits + 7) / 8;
  uint8_t* out = a.out + (size_t)e * L.expert_bytes + (size_t)tile * L.tile_bytes + (size_t)kc * L.scb;
  const int nb = L.SC / L.B;
  const int ktiles = L.SC / 16;

  for (int s = 0; s < L.nsub; ++s) {
    // canonical row of local row `off` of this 16-row sub-tile: fc1 gate
    // (s = 0) / up (s = 1) row of feature f = tile*16 + off, concatenated
    // ([gate | up]) or interleaved (gate f = 2f, up f = 2f+1); fc2 row f.
    auto crow = [&](int off) {
      const int f = tile * 16 + off;
      if (a.I_or_0 == 0) return f;
      return a.interleaved ? 2 * f + s : f + s * a.I_or_0;
    };
    auto code = [&](int row, int d) {
      const uint8_t* rp = a.codes + ((size_t)e * a.N + row) * row_bytes;
      return canon_code(rp, row_bytes, bits, d, a.K);
    };
    // k index of pair r, element e2 of k-tile j for lane (g, t)
    auto kidx = [&](int j, int t, int r, int e2) {
      return kc * L.SC + j * 16 + 2 * t + ((r & 2) ? 8 : 0) + e2;
    };
    uint32_t* cw = reinterpret_cast<uint32_t*>(out + s * L.code_bytes);
    if (bits == 1) {
      // one word per lane and four k-tiles: bit 4 (j & 3) + r of the low half
      // holds element 0 of pair r of k-tile j, the same bit of the high half
      // element 1
      const int W = ktiles / 4;
      for (int i = threadIdx.x; i < 32 * W; i += blockDim.x) {
        const int lane = i / W, wj = i % W, g = lane >> 2, t = lane & 3;
        uint32_t w = 0;
        for (int jj = 0; jj < 4; ++jj)
          for (int r = 0; r < 4; ++r) {
            const int j = 4 * wj + jj, row = crow(g + ((r & 1) ? 8 : 0));
            w |= (uint32_t)code(row, kidx(j, t, r, 0)) << (4 * jj + r);
            w |= (uint32_t)code(row, kidx(j, t, r, 1)) << (16 + 4 * jj + r);
          }
        cw[lane * W + wj] = w;
      }
    } else if (bits == 8) {
      // two words per lane and k-tile: word 2j + (r >> 1) holds pair r in
      // bytes (r & 1) and 2 + (r & 1)
      const int W = 2 * ktiles;
      for (int i = threadIdx.x; i < 32 * W; i += blockDim.x) {
        const int lane = i / W, wj = i % W, g = lane >> 2, t = lane & 3;
        const int j = wj >> 1;
        uint32_t w = 0;
        for (int rr = 0; rr < 2; ++rr) {
          const int r = 2 * (wj & 1) + rr;
          const int row = crow(g + ((r & 1) ? 8 : 0));
          w |= (uint32_t)code(row, kidx(j, t, r, 0)) << (8 * rr);
          w |= (uint32_t)code(row, kidx(j, t, r, 1)) << (16 + 8 * rr);
        }
        cw[lane * W + wj] = w;
      }
    } else if (bits == 4) {
      const int W = ktiles;  // words per lane
      for (int i = threadIdx.x; i < 32 * W; i += blockDim.x) {
        const int lane = i / W, j = i % W, g = lane >> 2, t = lane & 3;
        uint32_t w = 0;
        for (int r = 0; r < 4; ++r)
          for (int e2 = 0; e2 < 2; ++e2) {
            const int row = crow(g + ((r & 1) ? 8 : 0));
            w |= (uint32_t)code(row, kidx(j, t, r, e2)) << (4 * (r + 4 * e2));
          }
        cw[lane * W + j] = w;
      }
    } else {
      // 2-bit plane (bits 2, or the low bits of 3): one word = 2 k-tiles.
      const int W = ktiles / 2;
      for (int i = threadIdx.x; i < 32 * W; i += blockDim.x) {
        const int lane = i / W, wj = i % W, g = lane >> 2, t = lane & 3;
        uint32_t w = 0;
        for (int pi = 0; pi < 8; ++pi) {
          const int j = 2 * wj + pi / 4, r = pi % 4;
          const int row = crow(g + ((r & 1) ? 8 : 0));
          for (int e2 = 0; e2 < 2; ++e2)
            w |= (uint32_t)(code(row, kidx(j, t, r, e2)) & 3) << (2 * (pi + 8 * e2));
        }
        cw[lane * W + wj] = w;
      }
      if (bits == 3) {
        // 1-bit plane of bit 2: one word = 4 k-tiles.
        const int Wh = ktiles / 4;
        uint32_t* hw = cw + 32 * W;
        for (int i = threadIdx.x; i < 32 * Wh; i += blockDim.x) {
          const int lane = i / Wh, wj = i % Wh, g = lane >> 2, t = lane & 3;
          uint32_t w = 0;
          for (int pi = 0; pi < 16; ++pi) {
            const int j = 4 * wj + pi / 4, r = pi % 4;
            const int row = crow(g + ((r & 1) ? 8 : 0));
            for (int e2 = 0; e2 < 2; ++e2)
              w |= (uint32_t)((code(row, kidx(j, t, r, e2)) >> 2) & 1) << (pi + 16 * e2);
          }
          hw[lane * Wh + wj] = w;
        }
      }
    }
    // scales: [blk][g][2]
    const int ds = a.dsize;
    uint8_t* sp = out + L.nsub * L.code_bytes + s * L.scale_bytes;
    for (int i = threadIdx.x; i < nb * 16; i += blockDim.x) {
      const int blk = i / 16, g = (i % 16) / 2, hi = i % 2;
      const int row = crow(g + 8 * hi);
      const int kb = kc * nb + blk;
      uint16_t v = 0;
      if (kb < nblk_row)
        v = reinterpret_cast<const uint16_t*>(a.scales)[((size_t)e * a.N + row) * nblk_row + kb];
      if (ds == 2) reinterpret_cast<uint16_t*>(sp)[i] = v;
    }
    if (L.zp_bytes) {
      uint8_t* zp = out + L.nsub * (L.code_bytes + L.scale_bytes) + s * L.zp_bytes;
      for (int i = threadIdx.x; i < L.zp_bytes; i += blockDim.x) {
        uint8_t v = 0;
        if (bits == 8 && i < nb * 16) {
          // [blk][g][row g, row g+8]
          const int blk = i / 16, g = (i % 16) / 2, hi = i % 2, kb = kc * nb + blk;
          if (kb < nblk_row)
            v = (uint8_t)canon_code(a.zp + ((size_t)e * a.N + crow(g + 8 * hi)) * zrow_bytes, zrow_bytes, bits,
                                    kb, nblk_row);
        } else if (bits != 8 && i < nb * 8) {
          const int blk = i / 8, g = i % 8, kb = kc * nb + blk;
          if (kb < nblk_row) {
            const uint8_t* z0 = a.zp + ((size_t)e * a.N + crow(g)) * zrow_bytes;
            const uint8_t* z1 = a.zp + ((size_t)e * a.N + crow(g + 8)) * zrow_bytes;
            const int lo = canon_code(z0, zrow_bytes, bits, kb, nblk_row);
            const int hi = canon_code(z1, zrow_bytes, bits, kb, nblk_row);
            v = (uint8_t)(lo | (hi << 4));
          }
        }
        zp[i] = v;
      }
    }
  }
}

cudaError_t launch_repack_decode(const RepackArgs& a, cudaStream_t s) {
  const size_t nblocks = (size_t)a.E * a.L.ntiles * a.L.nkc;
  if (nblocks == 0) return cudaSuccess;
  if (nblocks > 0x7fffffff) return cudaErrorInvalidValue;
  repack_decode_kernel<<<(unsigned)nblocks, 128, 0, s>>>(a);
  return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_decode_mma_bits(const DecodeArgs& a, cudaStream_t s);
extern template cudaError_t launch_decode_mma_bits<1>(const DecodeArgs&, cudaStream_t);
extern template cudaError_t launch_decode_mma_bits<2>(const DecodeArgs&, cudaStream_t);
extern template cudaError_t launch_decode_mma_bits<3>(const DecodeArgs&, cudaStream_t);
extern template cudaError_t launch_decode_mma_bits<4>(const DecodeArgs&, cudaStream_t);
extern template cudaError_t launch_decode_mma_bits<8>(const DecodeArgs&, cudaStream_t);

cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t s) {
  if (a.max_items <= 0) return cudaSuccess;
  if (a.ng < 1 || a.ng > 4) return cudaErrorInvalidValue;
  switch (a.L.bits) {
    case 1: return launch_decode_mma_bits<1>(a, s);
    case 2: return launch_decode_mma_bits<2>(a, s);
    case 3: return launch_decode_mma_bits<3>(a, s);
    case 4: return launch_decode_mma_bits<4>(a, s);
    case 8: return launch_decode_mma_bits<8>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

// ----------------------------------------------------------------------------
// SIMT path (fp32 activations): canonical layout, one warp per output row
// (fc1: the gate row and its up row), all rows of a work item (<= 4 tokens),
// plain fp32 FMAs.  W is rounded into D exactly as in the definition.
// ----------------------------------------------------------------------------
constexpr int kSimtRows = 4;

template <int DT>
__device__ __forceinline__ float simt_weight(const SimtArgs& a, int e, int row, int d) {
  // canonical rows per expert: 2I for a gated fc1, else the output rows
  const int N = a.fc == 1 && act_gated(a.act.act) ? 2 * a.I_or_0 : a.N_out;
  const int row_bytes = a.K * a.bits / 8;
  const int nblk = a.K / a.B;
  const size_t er = (size_t)e * N + row;
  const int q = canon_code(a.codes + er * row_bytes, row_bytes, a.bits, d, a.K);
  const int kb = d / a.B;
  float z;
  if (a.zp_mode == QMOE_ZP_UINT8)
    z = (float)canon_code(a.zp + er * a.zp_bytes_row, a.zp_bytes_row, a.bits, kb, nblk);
  else if (a.zp_mode == QMOE_ZP_OFFSET)
    z = a.zp_offset;
  else
    z = (float)(1 << (a.bits - 1));
  const float sc = load_d<DT>(a.scales, er * nblk + kb);
  return round_d<DT>(__fmul_rn((float)q - z, sc));
}

template <int DT>
__global__ void __launch_bounds__(256) simt_kernel(const SimtArgs a) {
  extern __shared__ float xs[];  // [kSimtRows][K]
  pdl_wait();
  if ((int)blockIdx.y >= *a.n_items) return;
  const Item it = a.items[blockIdx.y];
  const int K = a.K;
  for (int idx = threadIdx.x; idx < kSimtRows * K; idx += blockDim.x) {
    const int n = idx / K, d = idx % K;
    float v = 0.f;
    if (n < it.rows) {
      const size_t row = a.fc == 1 ? (size_t)(a.perm[it.start + n] / a.k) : (size_t)(it.start + n);
      v = load_d<DT>(a.src, row * K + d);
    }
    xs[idx] = v;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;
  if (n >= a.N_out) return;
  const bool glu_fc = a.fc == 1 && act_gated(a.act.act);
  const bool act_fc = a.fc == 1 && !glu_fc;   // non-gated fc1
  float ag[kSimtRows] = {0.f, 0.f, 0.f, 0.f}, au[kSimtRows] = {0.f, 0.f, 0.f, 0.f};
  // fc1 rows of feature n: concatenated [gate | up] or interleaved pairs
  const int grow = glu_fc && a.interleaved ? 2 * n : n;
  const int urow = glu_fc ? (a.interleaved ? 2 * n + 1 : a.I_or_0 + n) : 0;
  for (int d = lane; d < K; d += 32) {
    const float wg = simt_weight<DT>(a, it.e, grow, d);
    const float wu = glu_fc ? simt_weight<DT>(a, it.e, urow, d) : 0.f;
#pragma unroll
    for (int r = 0; r < kSimtRows; ++r) {
      ag[r] = fmaf(wg, xs[r * K + d], ag[r]);
      if (glu_fc) au[r] = fmaf(wu, xs[r * K + d], au[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < kSimtRows; ++r) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ag[r] += __shfl_xor_sync(0xffffffffu, ag[r], o);
      au[r] += __shfl_xor_sync(0xffffffffu, au[r], o);
    }
  }
  if (lane == 0) {
    // fp32 projection bias [qmoe.rs qmoe_linear_impl]: fc1 (gate, up) pairs, fc2 rows
    float bg = 0.f, bu = 0.f;
    if (a.bias) {
      if (glu_fc) {
        bg = a.bias[((size_t)it.e * a.N_out + n) * 2];
        bu = a.bias[((size_t)it.e * a.N_out + n) * 2 + 1];
      } else {
        bg = a.bias[(size_t)it.e * a.N_out + n];
      }
    }
    for (int r = 0; r < it.rows && r < kSimtRows; ++r) {
      const size_t o = (size_t)(it.start + r) * a.N_out + n;
      if (glu_fc) store_d<DT>(a.dst, o, glu(a.act, ag[r] + bg, au[r] + bu));
      else if (act_fc) store_d<DT>(a.dst, o, act_single(a.act, ag[r] + bg));
      else static_cast<float*>(a.dst)[o] = ag[r] + bg;
    }
  }
}

cudaError_t launch_simt(const SimtArgs& a, cudaStream_t s) {
  if (a.max_items <= 0) return cudaSuccess;
  const size_t smem = (size_t)kSimtRows * a.K * sizeof(float);
  if (smem > 220 * 1024) return cudaErrorInvalidConfiguration;
  dim3 grid((a.N_out + 7) / 8, a.max_items);
  cudaError_t err;
  switch (a.dtype) {
    case QMOE_F32:
      err = cudaFuncSetAttribute(simt_kernel<QMOE_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      simt_kernel<QMOE_F32><<<grid, 256, smem, s>>>(a);
      break;
    case QMOE_F16:
      err = cudaFuncSetAttribute(simt_kernel<QMOE_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      simt_kernel<QMOE_F16><<<grid, 256, smem, s>>>(a);
      break;
    default:
      err = cudaFuncSetAttribute(simt_kernel<QMOE_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      simt_kernel<QMOE_BF16><<<grid, 256, smem, s>>>(a);
      break;
  }
  return cudaGetLastError();
}

}  // namespace qmoe
