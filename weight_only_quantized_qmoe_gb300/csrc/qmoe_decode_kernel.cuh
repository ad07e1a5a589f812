// The weight-streaming mma decode kernel (template), instantiated per code
// width in qmoe_decode_b{2,3,4}.cu.  See qmoe_decode.cu for the design.
#pragma once
#include "qmoe_internal.cuh"

namespace qmoe {

// ----------------------------------------------------------------------------
// The mma decode kernel
// ----------------------------------------------------------------------------
constexpr int kWarps = 8;

struct DecodeSmem {
  int bar_off, ring_off, stage_bytes, stages, g_chunks, bop_off, total;
};

__host__ __device__ inline DecodeSmem decode_smem(const DecodeLayout& L, int NG, int stages, int g_chunks,
                                                  int ksplit) {
  DecodeSmem m;
  m.stages = stages;
  m.g_chunks = g_chunks;
  m.stage_bytes = g_chunks * L.scb;
  m.bar_off = 0;
  m.ring_off = 1024;
  int ring = kWarps * stages * m.stage_bytes;
  const int red = ksplit > 1 ? kWarps * 32 * (L.nsub * 4 * 4) * 4 : 0;
  if (red > ring) ring = red;
  m.bop_off = m.ring_off + ((ring + 127) / 128) * 128;
  const int ktiles = L.nkc * L.SC / 16;
  m.total = m.bop_off + ktiles * NG * 256;
  return m;
}


// Fragment pair r (0..3) of k-tile j of this lane's code words (pairs of
// 16-bit fields, low element in bits 0.., high element in bits 16..).
template <int BITS>
__device__ __forceinline__ uint32_t code_pair(const uint32_t* cw, const uint32_t* hw, int j, int r) {
  if (BITS == 8) {
    return cw[2 * j + (r >> 1)] >> (8 * (r & 1));   // bytes 0 and 2 (bits above ignored)
  } else if (BITS == 1) {
    return (cw[j >> 2] >> (4 * (j & 3) + r)) & 0x00010001u;
  } else if (BITS == 4) {
    return (cw[j] >> (4 * r)) & 0x000F000Fu;
  } else if (BITS == 2) {
    return (cw[j >> 1] >> (2 * ((j & 1) * 4 + r))) & 0x00030003u;
  } else {
    const uint32_t lo = (cw[j >> 1] >> (2 * ((j & 1) * 4 + r))) & 0x00030003u;
    const uint32_t hi = (hw[j >> 2] >> ((j & 3) * 4 + r)) & 0x00010001u;
    return lo | (hi << 2);
  }
}

// EPI: 0 = fc2, 1 = gated fc1 (gate and up sub-tiles), 2 = non-gated fc1.
template <int BITS, int ZPM, bool BF16, int EPI, int BLK>
__global__ void __launch_bounds__(kWarps * 32, 1)
    decode_mma_kernel(const DecodeArgs a, int tpc, int ksplit, int stages, int g_chunks) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr bool GLU = EPI == 1;
  constexpr int NSUB = GLU ? 2 : 1;
  constexpr int SC = BLK > 64 ? BLK : 64;  // super-chunk length along K
  constexpr int KT = SC / 16;              // k-tiles per super-chunk
  constexpr int NBK = SC / BLK;            // quantisation blocks per super-chunk
  constexpr int KTB = BLK / 16;            // k-tiles per block
  const DecodeLayout& L = a.L;
  constexpr int NGM = 4;               // max token groups (accumulator size)
  const int NG = a.ng;
  const DecodeSmem sm = decode_smem(L, NG, stages, g_chunks, ksplit);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + sm.bar_off);
  uint8_t* ring_base = smem + sm.ring_off;
  uint32_t* bop = reinterpret_cast<uint32_t*>(smem + sm.bop_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  pdl_wait();
  const int n_items = *a.n_items;
  if ((int)blockIdx.y >= n_items) return;  // uniform across the CTA
  const Item it = a.items[blockIdx.y];

  const int tile = blockIdx.x * tpc + warp / ksplit;
  const int ks = warp % ksplit;
  const bool active = warp < tpc * ksplit && tile < L.ntiles;
  const int kc0 = ks * L.nkc / ksplit, kc1 = (ks + 1) * L.nkc / ksplit;
  const int nchunks = kc1 - kc0;
  const int nst = active ? (nchunks + g_chunks - 1) / g_chunks : 0;
  uint64_t* bar = bars + warp * stages;
  uint8_t* ring = ring_base + (size_t)warp * stages * sm.stage_bytes;
  const uint8_t* src = a.wpk + (size_t)it.e * L.expert_bytes + (size_t)(active ? tile : 0) * L.tile_bytes +
                       (size_t)kc0 * L.scb;

  auto issue = [&](int i) {
    const int slot = i % stages;
    const int nck = min(g_chunks, nchunks - i * g_chunks);
    const uint32_t bytes = (uint32_t)(nck * L.scb);
    mbar_arrive_expect_tx(&bar[slot], bytes);
    // Test hook: the barrier of stage 0 is armed but its copy never issued,
    // so the wait on it can only run out (host-injected failure).
    if (a.inject_stall && i == 0) return;
    bulk_g2s(ring + slot * sm.stage_bytes, src + (size_t)i * g_chunks * L.scb, bytes, &bar[slot]);
  };
  int issued = 0;
  if (active && lane == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
    for (; issued < min(stages, nst); ++issued) issue(issued);
  }
  issued = __shfl_sync(0xffffffffu, issued, 0);
  __syncwarp();

  // Stage the item's rows (B operand) in fragment order:
  // bop[((kt * NG + ng) * 32 + g*4 + t) * 2 + hi] = (row ng*8+g, k = kt*16 + hi*8 + 2t, +1)
  // Only the item's rows are loaded (16 bytes per thread, all loads of a pass
  // in flight before any store); token columns past it.rows are never stored
  // by the epilogue, so their fragments may hold anything.  The K padding
  // (when K is not a multiple of SC) must be zero: it meets zero weights.
  {
    const int K = a.K;                 // multiple of 32
    const int Kp = L.nkc * SC;
    const int vrow = K / 8;            // 16-byte vectors per row
    const int nvec = it.rows * vrow;
    const uint16_t* src16 = static_cast<const uint16_t*>(a.src);
    constexpr int U = 4;
    for (int base = threadIdx.x; base < nvec; base += U * blockDim.x) {
      uint4 v[U];
      int nn[U], kv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int idx = base + u * blockDim.x;
        nn[u] = -1;
        if (idx < nvec) {
          nn[u] = idx / vrow;
          kv[u] = idx % vrow;
          const size_t row = a.fc == 1 ? (size_t)(a.perm[it.start + nn[u]] / a.k)
                                       : (size_t)(it.start + nn[u]);
          v[u] = ld_nc_v4(src16 + row * K + kv[u] * 8);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (nn[u] < 0) continue;
        const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int kk = kv[u] * 8 + 2 * w, kt = kk >> 4, within = kk & 15;
          const int tt = (within & 7) >> 1, hi = within >> 3;
          bop[((kt * NG + (nn[u] >> 3)) * 32 + (nn[u] & 7) * 4 + tt) * 2 + hi] = w4[w];
        }
      }
    }
    if (Kp > K) {
      const int pad2 = (Kp - K) / 2;   // 32-bit pairs of padding per row
      for (int idx = threadIdx.x; idx < NG * 8 * pad2; idx += blockDim.x) {
        const int n = idx / pad2, kk = K + 2 * (idx % pad2);
        const int kt = kk >> 4, within = kk & 15;
        const int tt = (within & 7) >> 1, hi = within >> 3;
        bop[((kt * NG + (n >> 3)) * 32 + (n & 7) * 4 + tt) * 2 + hi] = 0u;
      }
    }
  }
  __syncthreads();

  float acc[NSUB][NGM][4];
#pragma unroll
  for (int s = 0; s < NSUB; ++s)
#pragma unroll
    for (int n = 0; n < NGM; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[s][n][i] = 0.f;

  const int ng_act = (it.rows + 7) >> 3;
  constexpr uint32_t MAGIC = Magic<BF16>::v;
  // offset zero point: the half-unit magic pair, or for bf16 8-bit codes
  // (whose accepted offsets are integers) the pair (z, z)
  uint32_t zoff2 = 0u;
  if constexpr (ZPM == QMOE_ZP_OFFSET)
    zoff2 = (BITS == 8 && BF16) ? (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a.zp_offset)) * 0x00010001u
                                : half_magic_offset<BF16>(a.zp_offset);
  const uint32_t ZSYM = BITS == 8 ? code8_zq<BF16>(128u) : MAGIC | ((1u << (BITS - 1)) * 0x00010001u);

  bool ok = true;
  int i = 0;
  for (; i < nst; ++i) {
    const int slot = i % stages;
    // every lane polls; the warp continues (or gives up) as one
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bar[slot], (uint32_t)((i / stages) & 1), a.wait))) {
      ok = false;
      break;
    }
    const uint8_t* st = ring + slot * sm.stage_bytes;
    const int nck = min(g_chunks, nchunks - i * g_chunks);
    for (int c = 0; c < nck; ++c) {
      const uint8_t* ch = st + c * L.scb;
      const int kc = kc0 + i * g_chunks + c;
      // this lane's code words for each sub-tile
      constexpr int WPL = BITS == 8 ? SC / 8 : (BITS == 4 ? SC / 16 : (BITS == 1 ? SC / 64 : SC / 32));   // (low-plane) words per lane
      constexpr int WPH = BITS == 3 ? SC / 64 : 1;
      uint32_t cw[NSUB][WPL];
      uint32_t hw[NSUB][WPH];
#pragma unroll
      for (int s = 0; s < NSUB; ++s) {
        const uint32_t* base = reinterpret_cast<const uint32_t*>(ch + s * L.code_bytes);
        if constexpr (WPL % 4 == 0) {
#pragma unroll
          for (int w = 0; w < WPL; w += 4) {
            const uint4 q4 = *reinterpret_cast<const uint4*>(base + lane * WPL + w);
            cw[s][w] = q4.x; cw[s][w + 1] = q4.y; cw[s][w + 2] = q4.z; cw[s][w + 3] = q4.w;
          }
        } else if constexpr (WPL % 2 == 0) {
#pragma unroll
          for (int w = 0; w < WPL; w += 2) {
            const uint2 q2 = *reinterpret_cast<const uint2*>(base + lane * WPL + w);
            cw[s][w] = q2.x; cw[s][w + 1] = q2.y;
          }
        } else {
          static_assert(WPL == 1, "code words per lane");
          cw[s][0] = base[lane];
        }
        if constexpr (BITS == 3) {
#pragma unroll
          for (int w = 0; w < WPH; ++w) hw[s][w] = base[32 * WPL + lane * WPH + w];
        }
      }
#pragma unroll
      for (int blk = 0; blk < NBK; ++blk) {
        uint32_t ss[NSUB][2], zz[NSUB][2];
#pragma unroll
        for (int s = 0; s < NSUB; ++s) {
          const uint32_t sp = *reinterpret_cast<const uint32_t*>(
              ch + NSUB * L.code_bytes + s * L.scale_bytes + (blk * 8 + g) * 4);
          ss[s][0] = __byte_perm(sp, 0, 0x1010);   // (s_g, s_g)
          ss[s][1] = __byte_perm(sp, 0, 0x3232);   // (s_g8, s_g8)
          if (ZPM == QMOE_ZP_UINT8) {
            const uint8_t* zpp = ch + NSUB * (L.code_bytes + L.scale_bytes) + s * L.zp_bytes;
            if constexpr (BITS == 8) {
              zz[s][0] = code8_zq<BF16>(zpp[blk * 16 + 2 * g]);
              zz[s][1] = code8_zq<BF16>(zpp[blk * 16 + 2 * g + 1]);
            } else {
              const uint32_t zb = zpp[blk * 8 + g];
              zz[s][0] = MAGIC | ((zb & 15u) * 0x00010001u);
              zz[s][1] = MAGIC | ((zb >> 4) * 0x00010001u);
            }
          } else {
            zz[s][0] = zz[s][1] = ZSYM;
          }
        }
#pragma unroll
        for (int jj = 0; jj < KTB; ++jj) {
          const int j = blk * KTB + jj;   // k-tile within the super-chunk
          uint32_t afrag[NSUB][4];
#pragma unroll
          for (int s = 0; s < NSUB; ++s) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              uint32_t v;
              if constexpr (BITS == 8) {
                const uint32_t b = code_pair<BITS>(cw[s], hw[s], j, r);
                if constexpr (ZPM == QMOE_ZP_OFFSET && !BF16)
                  v = sub2<false>(((b & 0x00FF00FFu) << 1) | Magic<false>::half, zoff2);
                else
                  v = code8_minus_zp<BF16>(b, ZPM == QMOE_ZP_OFFSET ? zoff2 : zz[s][r & 1]);
              } else if constexpr (ZPM == QMOE_ZP_OFFSET) {
                // half-unit magic: (M/2 + c) - (M/2 + z) = c - z, exact for
                // half-integer z (the only centres the API accepts)
                v = (code_pair<BITS>(cw[s], hw[s], j, r) << 1) | Magic<BF16>::half;
                v = sub2<BF16>(v, zoff2);
              } else {
                v = code_pair<BITS>(cw[s], hw[s], j, r) | MAGIC;
                v = sub2<BF16>(v, zz[s][r & 1]);
              }
              afrag[s][r] = mul2<BF16>(v, ss[s][r & 1]);
            }
          }
          const int ktg = kc * KT + j;
#pragma unroll
          for (int n = 0; n < NGM; ++n) {
            if (n < ng_act) {
              const uint2 b = *reinterpret_cast<const uint2*>(bop + ((ktg * NG + n) * 32 + lane) * 2);
#pragma unroll
              for (int s = 0; s < NSUB; ++s) mma16816<BF16>(acc[s][n], afrag[s], b.x, b.y);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0 && i + stages < nst) {
      fence_proxy_async_smem();
      issue(i + stages);
    }
    issued = min(nst, max(issued, i + stages + 1));
  }
  if (!ok) {
    // Drain the copies still in flight into this warp's ring before the CTA
    // can exit.  This uses the fixed default bound, not the (possibly tiny)
    // configured one, so the copies have landed when the CTA leaves.
    const WaitCfg drain{a.wait.status, kDrainWaitLimit};
    for (int d = i; d < issued; ++d) {
      if (a.inject_stall && d == 0) continue;   // no copy was issued for it
      mbar_wait_bounded(&bar[d % stages], (uint32_t)((d / stages) & 1), drain);
    }
  }
  pdl_launch_dependents();

  // Split-K reduction over the ksplit warps of a tile (deterministic order).
  if (ksplit > 1) {
    __syncthreads();
    float* red = reinterpret_cast<float*>(ring_base);
    constexpr int NACC = NSUB * NGM * 4;
    if (ks != 0) {
      float* dst = red + (warp * 32 + lane) * NACC;
#pragma unroll
      for (int s = 0; s < NSUB; ++s)
#pragma unroll
        for (int n = 0; n < NGM; ++n)
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[(s * NGM + n) * 4 + q] = acc[s][n][q];
    }
    __syncthreads();
    if (ks == 0) {
      for (int o = 1; o < ksplit; ++o) {
        const float* srcr = red + ((warp + o) * 32 + lane) * NACC;
#pragma unroll
        for (int s = 0; s < NSUB; ++s)
#pragma unroll
          for (int n = 0; n < NGM; ++n)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[s][n][q] += srcr[(s * NGM + n) * 4 + q];
      }
    }
  }
  if (!active || ks != 0) return;

  // Epilogue.  acc[s][n][q]: row g + 8*(q>>1), token n*8 + 2t + (q&1).
  // fp32 projection biases [qmoe.rs qmoe_linear_impl]: fc1 (gate, up) pairs
  // per feature, fc2 per row.
  float bias_g[2] = {0.f, 0.f}, bias_u[2] = {0.f, 0.f};
  if (a.bias) {
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
      const int row = tile * 16 + g + 8 * hi;
      if (GLU) {
        bias_g[hi] = a.bias[((size_t)it.e * a.N_out + row) * 2];
        bias_u[hi] = a.bias[((size_t)it.e * a.N_out + row) * 2 + 1];
      } else {
        bias_g[hi] = a.bias[(size_t)it.e * a.N_out + row];
      }
    }
  }
#pragma unroll
  for (int n = 0; n < NGM; ++n) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int tok = n * 8 + 2 * t + (q & 1);
      const int row = tile * 16 + g + 8 * (q >> 1);
      acc[0][n][q] += bias_g[q >> 1];
      if (GLU) acc[NSUB - 1][n][q] += bias_u[q >> 1];
      if (tok < it.rows) {
        const size_t o = (size_t)(it.start + tok) * a.N_out + row;
        if (EPI != 0) {
          const float h = GLU ? glu(a.act, acc[0][n][q], acc[1][n][q]) : act_single(a.act, acc[0][n][q]);
          if (BF16) static_cast<__nv_bfloat16*>(a.dst)[o] = __float2bfloat16_rn(h);
          else static_cast<__half*>(a.dst)[o] = __float2half_rn(h);
        } else if (a.atomic) {
          const int route = a.perm[it.start + tok];
          atomicAdd(a.out_acc + (size_t)(route / a.k) * a.N_out + row, a.w[route] * acc[0][n][q]);
        } else {
          static_cast<float*>(a.dst)[o] = acc[0][n][q];
        }
      }
    }
  }
}

template <int BITS, int ZPM, bool BF16, int EPI, int BLK>
static cudaError_t launch_dm(const DecodeArgs& a, cudaStream_t s) {
  const DecodeLayout& L = a.L;
  // Split-K when the tiles alone would not fill the GPU.
  const int sms = 152;
  int ksplit = 1;
  const long long est_items = a.max_items;
  while (ksplit < 8 && est_items * ((L.ntiles + (kWarps / ksplit) - 1) / (kWarps / ksplit)) < 2LL * sms &&
         L.nkc / (ksplit * 2) >= 2)
    ksplit *= 2;
  const int tpc = kWarps / ksplit;
  // Stages of >= ~1 KB, ring of ~4 stages per warp within the smem budget.
  int g_chunks = L.scb >= 1024 ? 1 : (1024 + L.scb - 1) / L.scb;
  int stages = 4;
  DecodeSmem sm = decode_smem(L, a.ng, stages, g_chunks, ksplit);
  while (sm.total > 220 * 1024 && stages > 2) {
    --stages;
    sm = decode_smem(L, a.ng, stages, g_chunks, ksplit);
  }
  while (sm.total > 220 * 1024 && g_chunks > 1) {
    --g_chunks;
    sm = decode_smem(L, a.ng, stages, g_chunks, ksplit);
  }
  if (sm.total > 227 * 1024) return cudaErrorInvalidConfiguration;
  auto kern = decode_mma_kernel<BITS, ZPM, BF16, EPI, BLK>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, sm.total);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((L.ntiles + tpc - 1) / tpc, a.max_items);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = sm.total;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, tpc, ksplit, stages, g_chunks);
}

template <int BITS, int ZPM, bool BF16, int EPI>
static cudaError_t dispatch_blk(const DecodeArgs& a, cudaStream_t s) {
  if (a.L.B == 32) return launch_dm<BITS, ZPM, BF16, EPI, 32>(a, s);
  if (a.L.B == 64) return launch_dm<BITS, ZPM, BF16, EPI, 64>(a, s);
  return launch_dm<BITS, ZPM, BF16, EPI, 128>(a, s);
}
template <int BITS, int ZPM, bool BF16>
static cudaError_t dispatch_glu(const DecodeArgs& a, cudaStream_t s) {
  if (a.fc == 1) {
    if (act_gated(a.act.act)) return dispatch_blk<BITS, ZPM, BF16, 1>(a, s);
    return dispatch_blk<BITS, ZPM, BF16, 2>(a, s);
  }
  return dispatch_blk<BITS, ZPM, BF16, 0>(a, s);
}
template <int BITS, int ZPM>
static cudaError_t dispatch_dt(const DecodeArgs& a, cudaStream_t s) {
  if (a.bf16) return dispatch_glu<BITS, ZPM, true>(a, s);
  return dispatch_glu<BITS, ZPM, false>(a, s);
}
template <int BITS>
cudaError_t launch_decode_mma_bits(const DecodeArgs& a, cudaStream_t s) {
  if (a.zp_mode == QMOE_ZP_UINT8) return dispatch_dt<BITS, QMOE_ZP_UINT8>(a, s);
  if (a.zp_mode == QMOE_ZP_OFFSET) return dispatch_dt<BITS, QMOE_ZP_OFFSET>(a, s);
  return dispatch_dt<BITS, QMOE_ZP_SYMMETRIC>(a, s);
}

}  // namespace qmoe
