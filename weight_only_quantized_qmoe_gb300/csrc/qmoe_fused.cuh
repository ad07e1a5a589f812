// Single-launch decode forward of the QMoE layer (template; instantiated per
// code-width pair in qmoe_fused_w*.cu, launched from qmoe_fused.cu).
//
// One persistent kernel runs the whole layer for small token counts:
//   routing (top-k on the fp32 logits under the total-order key, ties to the
//   lower expert index; softmax weights, optionally renormalised over the k
//   chosen)  [onnx-runtime-ep-cuda src/kernels/qmoe.rs, CUDA_SRC
//   total_order_key / route_value_is_better / qmoe_route]
//   -> grouping (counts, offsets, stable permutation)  [qmoe.rs launch_grouping]
//   -> fc1 + gated (or plain) activation -> fc2
//   -> out[t] = R_D(sum_j w[t,j] y[t*k+j]), slots j in ascending order
//   [qmoe.rs qmoe_combine_impl]
// with W = R_D((q - zp) * s) rounded once before it is multiplied [onnxruntime
// PR "fast INT3 QMoE kernels", review "Round dequantized weights before
// accumulation"; zero_point_offset from PR "fused int2 mixed-input GEMM +
// GeGLU + fractional zero-point"].  The pages motivate the fusion: the
// single-CTA fused route of the "fast INT3" PR and the single-token direct
// path of ferrum moe.rs (SingleTokenDirectMarlin).
//
// GB300 design (ours):
//   * every CTA routes all tokens itself (a warp per token, warp-wide
//     redux.sync arg-max per slot) and builds the grouping in shared memory,
//     so no CTA waits on another before it streams weights;
//   * work items are handed out by one atomic ticket counter in a fixed order
//     (all fc1 items expert by expert, then all fc2 items): an item only ever
//     waits on items with smaller tickets, which running CTAs hold, so the
//     kernel needs no co-residency guarantee;
//   * an item = (expert, group of <= 16 routed rows, group of 16-row weight
//     tiles); its 8 warps split the tiles and K; each warp streams its part of
//     the prepacked tile straight from HBM into registers (128-bit
//     non-coherent loads, a ring of 2 super-chunks in flight) and feeds
//     mma.m16n8k16 with fp32 accumulation, the routed rows staged once per item
//     in shared memory in B-fragment order;
//   * fc2 items of an expert start as soon as that expert's fc1 items are done
//     (a per-expert counter, bounded wait); the last fc2 item of each group of
//     output rows adds the k slots in order and rounds into D;
//   * the last CTA to leave clears the counters for the next launch.
#pragma once
#include <climits>

#include "qmoe_internal.cuh"
#include "qmoe_decode_kernel.cuh"

namespace qmoe {

// Limits of the single-launch path (checked on the host).
constexpr int kFusedMaxTokens = 64;
constexpr int kFusedMaxExperts = 256;
constexpr int kFusedMaxRoutes = 512;
constexpr int kFusedMaxK = 32;
constexpr int kFusedThreads = 256;   // 8 warps
constexpr int kFusedRowsPerGroup = 16;
// Counters in the sync buffer: [0] ticket, [1] exit, [2] a flag nothing sets
// (the injected stall waits on it), then done1[E], then done2[M-groups].
constexpr int kSyncHeader = 4;

struct FusedProj {
  const uint8_t* wpk;   // decode layout
  DecodeLayout L;
  int K;                // real K
  int ntiles;           // 16-row tiles (fc1: feature tiles, gate + up when gated)
  int tpi, ks;          // weight tiles per item, K-splits (tpi * ks == 8)
  const float* bias;    // fc1 gated: [E, I, 2]; fc1 plain: [E, I]; fc2: [E, H]; or null
};

struct FusedArgs {
  const float* logits;
  const void* x;        // [T, H] D
  void* out;            // [T, H] D
  int T, E, k, normalize, H, I;
  int gated;
  FusedProj p[2];
  ActParams act;
  int zp_mode;
  float zp_offset;
  // outputs of routing kept for qmoe_get_routing / qmoe_get_worklist (CTA 0)
  int* ids;
  float* w;
  int* counts;
  int* offsets;
  int* perm;
  Item* items0;
  int* n_items;
  void* hbuf;           // [R, I] D, by route
  float* ybuf;          // [R, H] f32, by route
  int* sync;            // kSyncHeader + E + n_mg ints, zero between launches
  int n_mg;             // fc2 groups of output rows (= ceil(fc2 tiles / fc2 tpi))
  WaitCfg wait;
  int inject_stall;
};

// Shared-memory plan of one CTA (the front of dynamic shared memory).
struct FusedPlan {
  int ids_off, w_off, perm_off, cnt_off, off_off, cur_off, act_off, rgb_off, bop_off, total;
};

__host__ __device__ inline int fused_align16(int v) { return (v + 15) & ~15; }

__host__ __device__ inline FusedPlan fused_plan(int R, int E, int bop_bytes) {
  FusedPlan p;
  int o = 64;   // a few broadcast ints first
  p.ids_off = o;  o = fused_align16(o + 4 * R);
  p.w_off = o;    o = fused_align16(o + 4 * R);
  p.perm_off = o; o = fused_align16(o + 4 * R);
  p.cnt_off = o;  o = fused_align16(o + 4 * E);
  p.off_off = o;  o = fused_align16(o + 4 * (E + 1));
  p.cur_off = o;  o = fused_align16(o + 4 * E);
  p.act_off = o;  o = fused_align16(o + 4 * E);
  p.rgb_off = o;  o = fused_align16(o + 4 * (E + 1));
  o = (o + 127) & ~127;
  p.bop_off = o;
  p.total = o + bop_bytes;
  return p;
}

// Bytes of the B-operand staging (>= the split-K reduction it is reused for).
__host__ __device__ inline int fused_bop_bytes(int Kp_max) {
  const int bop = Kp_max / 16 * 2 * 32 * 8;           // k-tiles x 2 token groups x 32 lanes x 8 B
  const int red = 8 * 32 * (2 * 2 * 4) * 4;           // 8 warps x 32 lanes x acc[2][2][4] floats
  return bop > red ? bop : red;
}

__device__ __forceinline__ int redux_max_s32(int v) {
  int r;
  asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}
__device__ __forceinline__ int redux_min_s32(int v) {
  int r;
  asm volatile("redux.sync.min.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

__device__ __forceinline__ int fused_order_key(float v) {
  const int b = __float_as_int(v);
  return b ^ ((b >> 31) & 0x7fffffff);
}

// One warp ranks the E (<= 256) logits of one token: ids[0..k) in rank order
// and their weights.
__device__ __forceinline__ void fused_route_token(const float* __restrict__ lg, int E, int k, int normalize,
                                                  int* ids, float* w) {
  constexpr int NPL = kFusedMaxExperts / 32;
  const int lane = threadIdx.x & 31;
  int key[NPL];
  uint32_t taken = 0;
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float v = lg[e];
      key[i] = fused_order_key(v);
      mx = fmaxf(mx, v);
    } else {
      key[i] = INT_MIN;
      taken |= 1u << i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum_all = 0.f;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) sum_all += expf(lg[e] - mx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum_all += __shfl_xor_sync(0xffffffffu, sum_all, o);

  for (int slot = 0; slot < k; ++slot) {
    int bk = INT_MIN, bi = INT_MAX;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      if (!((taken >> i) & 1u) && (key[i] > bk || (key[i] == bk && e < bi))) {
        bk = key[i];
        bi = e;
      }
    }
    const int m = redux_max_s32(bk);
    const int sel = redux_min_s32(bk == m ? bi : INT_MAX);
    if ((sel & 31) == lane) taken |= 1u << (sel >> 5);
    if (lane == 0) ids[slot] = sel;
  }
  __syncwarp();
  const float p = lane < k ? expf(lg[ids[lane]] - mx) : 0.f;
  float sum_sel = p;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum_sel += __shfl_xor_sync(0xffffffffu, sum_sel, o);
  if (lane < k) w[lane] = p / (normalize ? sum_sel : sum_all);
}

// ----------------------------------------------------------------------------
// Weight streaming of one warp's part of a tile.
// ----------------------------------------------------------------------------
template <int BITS, int SC, int NSUB>
struct FusedChunk {
  static constexpr int WPL = BITS == 8 ? SC / 8 : (BITS == 4 ? SC / 16 : (BITS == 1 ? SC / 64 : SC / 32));
  static constexpr int WPH = BITS == 3 ? SC / 64 : 1;
  static constexpr int NBKM = SC == 64 ? 2 : 1;
  uint32_t cw[NSUB][WPL];
  uint32_t hw[NSUB][WPH];
  uint32_t sp[NSUB][NBKM];
  uint32_t zb[NSUB][NBKM];
};

__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ld_nc_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ld_nc_u8(const void* p) {
  uint16_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

struct FusedGeom {
  int code_bytes, scale_bytes, zp_bytes, scb;
  int nbk;        // quantisation blocks per super-chunk (1 or 2)
  bool has_zp;    // packed uint8 zero points present
};

template <int BITS, int SC, int NSUB>
__device__ __forceinline__ void fused_load_chunk(FusedChunk<BITS, SC, NSUB>& c, const uint8_t* ch,
                                                 const FusedGeom& gm, int lane) {
  using C = FusedChunk<BITS, SC, NSUB>;
  const int g = lane >> 2;
#pragma unroll
  for (int s = 0; s < NSUB; ++s) {
    const uint32_t* base = reinterpret_cast<const uint32_t*>(ch + s * gm.code_bytes);
    if constexpr (C::WPL % 4 == 0) {
#pragma unroll
      for (int w = 0; w < C::WPL; w += 4) {
        const uint4 q = ld_nc_v4(base + lane * C::WPL + w);
        c.cw[s][w] = q.x; c.cw[s][w + 1] = q.y; c.cw[s][w + 2] = q.z; c.cw[s][w + 3] = q.w;
      }
    } else if constexpr (C::WPL == 2) {
      const uint2 q = ld_nc_v2(base + lane * 2);
      c.cw[s][0] = q.x; c.cw[s][1] = q.y;
    } else {
      static_assert(C::WPL == 1, "code words per lane");
      c.cw[s][0] = ld_nc_u32(base + lane);
    }
    if constexpr (BITS == 3) {
      if constexpr (C::WPH == 2) {
        const uint2 q = ld_nc_v2(base + 32 * C::WPL + lane * 2);
        c.hw[s][0] = q.x; c.hw[s][1] = q.y;
      } else {
        c.hw[s][0] = ld_nc_u32(base + 32 * C::WPL + lane);
      }
    }
    const uint8_t* sp = ch + NSUB * gm.code_bytes + s * gm.scale_bytes;
    c.sp[s][0] = ld_nc_u32(sp + g * 4);
    if constexpr (C::NBKM == 2) c.sp[s][1] = gm.nbk == 2 ? ld_nc_u32(sp + 32 + g * 4) : c.sp[s][0];
    if (gm.has_zp) {
      const uint8_t* zp = ch + NSUB * (gm.code_bytes + gm.scale_bytes) + s * gm.zp_bytes;
#pragma unroll
      for (int b = 0; b < C::NBKM; ++b) {
        if (b == 0 || gm.nbk == 2) {
          if constexpr (BITS == 8)
            c.zb[s][b] = ld_nc_u8(zp + b * 16 + 2 * g) | (ld_nc_u8(zp + b * 16 + 2 * g + 1) << 8);
          else
            c.zb[s][b] = ld_nc_u8(zp + b * 8 + g);
        } else {
          c.zb[s][b] = c.zb[s][0];
        }
      }
    }
  }
}

// Dequantise one super-chunk held in registers and run its MMAs.
//   bop_chunk: this lane's B fragments of the chunk's first k-tile
//              (bop + (kt * NG) * 64 + lane * 2 words).
template <int BITS, bool BF16, int SC, int NSUB, bool OFFS>
__device__ __forceinline__ void fused_compute_chunk(const FusedChunk<BITS, SC, NSUB>& c,
                                                    const uint32_t* __restrict__ bop_chunk, int NG,
                                                    bool uint8_zp, uint32_t zoff2, float (&acc)[2][2][4]) {
  using C = FusedChunk<BITS, SC, NSUB>;
  constexpr int KT = SC / 16;
  constexpr uint32_t MAGIC = Magic<BF16>::v;
  const uint32_t ZSYM = BITS == 8 ? code8_zq<BF16>(128u) : MAGIC | ((1u << (BITS - 1)) * 0x00010001u);
  uint32_t ss[NSUB][C::NBKM][2], zz[NSUB][C::NBKM][2];
#pragma unroll
  for (int s = 0; s < NSUB; ++s)
#pragma unroll
    for (int b = 0; b < C::NBKM; ++b) {
      ss[s][b][0] = __byte_perm(c.sp[s][b], 0, 0x1010);   // (s_g, s_g)
      ss[s][b][1] = __byte_perm(c.sp[s][b], 0, 0x3232);   // (s_g8, s_g8)
      if (!OFFS && uint8_zp) {
        if constexpr (BITS == 8) {
          zz[s][b][0] = code8_zq<BF16>(c.zb[s][b] & 0xffu);
          zz[s][b][1] = code8_zq<BF16>(c.zb[s][b] >> 8);
        } else {
          zz[s][b][0] = MAGIC | ((c.zb[s][b] & 15u) * 0x00010001u);
          zz[s][b][1] = MAGIC | ((c.zb[s][b] >> 4) * 0x00010001u);
        }
      } else {
        zz[s][b][0] = zz[s][b][1] = ZSYM;
      }
    }
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    const int b = (C::NBKM == 2 && j >= KT / 2) ? 1 : 0;
    uint32_t afrag[NSUB][4];
#pragma unroll
    for (int s = 0; s < NSUB; ++s) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t pr = code_pair<BITS>(c.cw[s], c.hw[s], j, r);
        uint32_t v;
        if constexpr (BITS == 8) {
          if constexpr (OFFS && !BF16)
            v = sub2<false>(((pr & 0x00FF00FFu) << 1) | Magic<false>::half, zoff2);
          else
            v = code8_minus_zp<BF16>(pr, OFFS ? zoff2 : zz[s][b][r & 1]);
        } else if constexpr (OFFS) {
          v = sub2<BF16>((pr << 1) | Magic<BF16>::half, zoff2);
        } else {
          v = sub2<BF16>(pr | MAGIC, zz[s][b][r & 1]);
        }
        afrag[s][r] = mul2<BF16>(v, ss[s][b][r & 1]);
      }
    }
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      if (n < NG) {
        const uint2 bf = *reinterpret_cast<const uint2*>(bop_chunk + (j * NG + n) * 64);
#pragma unroll
        for (int s = 0; s < NSUB; ++s) mma16816<BF16>(acc[s][n], afrag[s], bf.x, bf.y);
      }
    }
  }
}

// Accumulators of one warp: [sub-tile][token group][mma fragment].
struct FusedAcc {
  float v[2][2][4];
};

// Stream nck super-chunks starting at `src` (a ring of U chunks in flight).
// Not inlined: the hot loop then gets the registers to itself and the item
// loop's state is saved once per call instead of competing with the ring.
template <int BITS, bool BF16, int SC, int NSUB, bool OFFS>
__device__ __noinline__ FusedAcc fused_stream(const uint8_t* __restrict__ src, int nck, FusedGeom gm,
                                              const uint32_t* __restrict__ bop_lane, int NG, bool uint8_zp,
                                              uint32_t zoff2) {
  constexpr int U = 2;
  constexpr int KT = SC / 16;
  const int lane = threadIdx.x & 31;
  float acc[2][2][4];
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[s][n][q] = 0.f;
  FusedChunk<BITS, SC, NSUB> ring[U];
#pragma unroll
  for (int u = 0; u < U; ++u)
    if (u < nck) fused_load_chunk<BITS, SC, NSUB>(ring[u], src + (size_t)u * gm.scb, gm, lane);
  for (int c0 = 0; c0 < nck; c0 += U) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u;
      if (c < nck) {
        fused_compute_chunk<BITS, BF16, SC, NSUB, OFFS>(ring[u], bop_lane + c * KT * NG * 64, NG, uint8_zp,
                                                         zoff2, acc);
        if (c + U < nck) fused_load_chunk<BITS, SC, NSUB>(ring[u], src + (size_t)(c + U) * gm.scb, gm, lane);
      }
    }
  }
  FusedAcc r;
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int q = 0; q < 4; ++q) r.v[s][n][q] = acc[s][n][q];
  return r;
}

template <int BITS, bool BF16, int SC, int NSUB>
__device__ __forceinline__ FusedAcc fused_stream_zp(const uint8_t* src, int nck, const FusedGeom& gm,
                                                    const uint32_t* bop_lane, int NG, int zp_mode,
                                                    uint32_t zoff2) {
  if (zp_mode == QMOE_ZP_OFFSET)
    return fused_stream<BITS, BF16, SC, NSUB, true>(src, nck, gm, bop_lane, NG, false, zoff2);
  return fused_stream<BITS, BF16, SC, NSUB, false>(src, nck, gm, bop_lane, NG, zp_mode == QMOE_ZP_UINT8, zoff2);
}

__device__ __forceinline__ FusedGeom fused_geom(const DecodeLayout& L) {
  FusedGeom g;
  g.code_bytes = L.code_bytes;
  g.scale_bytes = L.scale_bytes;
  g.zp_bytes = L.zp_bytes;
  g.scb = L.scb;
  g.nbk = L.SC / L.B;
  g.has_zp = L.zp_bytes > 0;
  return g;
}

// Bounded wait of one thread until *p >= target; false (and DEV_TIMEOUT
// recorded) if it ran out, or at once if the layer already timed out.
__device__ __forceinline__ bool fused_wait_geq(const int* p, int target, const WaitCfg& w) {
  for (long long i = 0; i < w.limit; ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    if ((i & 63) == 63 && *reinterpret_cast<volatile int*>(w.status) != 0) return false;
    __nanosleep(64);
  }
  atomicExch(w.status, DEV_TIMEOUT);
  return false;
}

__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ----------------------------------------------------------------------------
// The kernel.
// ----------------------------------------------------------------------------
template <int B1, int B2, bool BF16, int SC>
__global__ void __launch_bounds__(kFusedThreads, 2) fused_decode_kernel(const FusedArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, E = a.E, k = a.k, R = T * k;
  const int Kp_max = (a.p[0].L.nkc > a.p[1].L.nkc ? a.p[0].L.nkc : a.p[1].L.nkc) * SC;
  const FusedPlan pl = fused_plan(R, E, fused_bop_bytes(Kp_max));
  int* bc = reinterpret_cast<int*>(smem);                       // broadcast ints
  int* ids_s = reinterpret_cast<int*>(smem + pl.ids_off);
  float* w_s = reinterpret_cast<float*>(smem + pl.w_off);
  int* perm_s = reinterpret_cast<int*>(smem + pl.perm_off);
  int* cnt_s = reinterpret_cast<int*>(smem + pl.cnt_off);
  int* off_s = reinterpret_cast<int*>(smem + pl.off_off);
  int* cur_s = reinterpret_cast<int*>(smem + pl.cur_off);
  int* act_s = reinterpret_cast<int*>(smem + pl.act_off);      // active experts, ascending
  int* rgb_s = reinterpret_cast<int*>(smem + pl.rgb_off);      // row-group prefix over active experts
  uint32_t* bop = reinterpret_cast<uint32_t*>(smem + pl.bop_off);
  float* red = reinterpret_cast<float*>(smem + pl.bop_off);
  int* done1 = a.sync + kSyncHeader;
  int* done2 = done1 + E;

  // ---- routing (every CTA, all tokens) ----
  for (int t = warp; t < T; t += kFusedThreads / 32)
    fused_route_token(a.logits + (size_t)t * E, E, k, a.normalize, ids_s + t * k, w_s + t * k);
  for (int i = tid; i < E; i += kFusedThreads) cnt_s[i] = 0;
  __syncthreads();
  for (int r = tid; r < R; r += kFusedThreads) atomicAdd(&cnt_s[ids_s[r]], 1);
  __syncthreads();
  // ---- grouping: offsets, active experts, row-group prefix (warp 0) ----
  if (warp == 0) {
    const unsigned lt = (1u << lane) - 1u;
    int run = 0, nact = 0, nrg = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? cnt_s[e] : 0;
      const int g = (c + kFusedRowsPerGroup - 1) / kFusedRowsPerGroup;
      int ic = c, ig = g;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int nc = __shfl_up_sync(0xffffffffu, ic, o);
        const int ng = __shfl_up_sync(0xffffffffu, ig, o);
        if (lane >= o) { ic += nc; ig += ng; }
      }
      const unsigned act = __ballot_sync(0xffffffffu, c > 0);
      if (e < E) {
        off_s[e] = run + ic - c;
        cur_s[e] = run + ic - c;
      }
      if (c > 0) {
        const int ai = nact + __popc(act & lt);
        act_s[ai] = e;
        rgb_s[ai] = nrg + ig - g;
      }
      run += __shfl_sync(0xffffffffu, ic, 31);
      nrg += __shfl_sync(0xffffffffu, ig, 31);
      nact += __popc(act);
    }
    if (lane == 0) {
      off_s[E] = run;
      rgb_s[nact] = nrg;
      bc[0] = nact;
      bc[1] = nrg;
    }
    __syncwarp();
    // stable permutation: routes of an expert in ascending route order
    for (int base = 0; base < R; base += 32) {
      const int r = base + lane;
      const int e = r < R ? ids_s[r] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0) perm_s[cur_s[e] + __popc(peers & lt)] = r;
      __syncwarp();
      if (e >= 0 && lane == __ffs(peers) - 1) cur_s[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  const int nact = bc[0], NRG = bc[1];

  // CTA 0 keeps the routing and the row-group work-list for the host.
  if (blockIdx.x == 0) {
    for (int r = tid; r < R; r += kFusedThreads) {
      a.ids[r] = ids_s[r];
      a.w[r] = w_s[r];
      a.perm[r] = perm_s[r];
    }
    for (int e = tid; e <= E; e += kFusedThreads) {
      a.offsets[e] = off_s[e];
      if (e < E) a.counts[e] = cnt_s[e];
    }
    for (int ai = tid; ai < nact; ai += kFusedThreads) {
      const int e = act_s[ai], c = cnt_s[e];
      for (int g = 0; g * kFusedRowsPerGroup < c; ++g) {
        Item it;
        it.e = e;
        it.start = off_s[e] + g * kFusedRowsPerGroup;
        it.rows = min(kFusedRowsPerGroup, c - g * kFusedRowsPerGroup);
        it.pad = 0;
        a.items0[rgb_s[ai] + g] = it;
      }
    }
    if (tid == 0) {
      a.n_items[0] = NRG;
      a.n_items[1] = 0;
    }
  }

  // ---- the work-item loop ----
  const int ntg1 = (a.p[0].ntiles + a.p[0].tpi - 1) / a.p[0].tpi;
  const int ntg2 = a.n_mg;
  const int n1 = NRG * ntg1, n2 = NRG * ntg2;
  // Fractional zero point: the half-unit magic offset (M/2 + z, M/2 + z);
  // 8-bit codes in bf16 take the integer pair (z, z) instead.
  uint32_t zoff_half = 0u, zoff_int = 0u;
  if (a.zp_mode == QMOE_ZP_OFFSET) {
    zoff_half = half_magic_offset<BF16>(a.zp_offset);
    zoff_int = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a.zp_offset)) * 0x00010001u;
  }
  int staged = -1;   // (phase, row group) whose rows are in bop
  for (;;) {
    if (tid == 0) bc[2] = atomicAdd(&a.sync[0], 1);
    __syncthreads();
    const int ticket = bc[2];
    if (ticket >= n1 + n2) break;
    const int ph = ticket < n1 ? 0 : 1;
    const int tt = ph == 0 ? ticket : ticket - n1;
    const int ntg = ph == 0 ? ntg1 : ntg2;
    const int rgg = tt / ntg, tg = tt % ntg;
    // active expert of row group rgg (binary search over the prefix)
    int lo = 0, hi = nact - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (rgb_s[mid] <= rgg) lo = mid; else hi = mid - 1;
    }
    const int ai = lo, e = act_s[ai], c = cnt_s[e];
    const int rg = rgg - rgb_s[ai];
    const int j0 = rg * kFusedRowsPerGroup;
    const int nrows = min(kFusedRowsPerGroup, c - j0);
    const int NG = (nrows + 7) >> 3;
    const FusedProj& P = a.p[ph];
    const int K = P.K;
    const int Kp = P.L.nkc * SC;
    bool ok = true;

    if (ph == 1) {
      // fc2 of this expert needs all its fc1 items
      const int nrg_e = rgb_s[ai + 1] - rgb_s[ai];
      if (tid == 0) {
        const bool w8 = a.inject_stall ? fused_wait_geq(a.sync + 2, 1, a.wait)
                                       : fused_wait_geq(done1 + e, nrg_e * ntg1, a.wait);
        bc[3] = w8 ? 1 : 0;
      }
      __syncthreads();
      ok = bc[3] != 0;
    }

    // ---- stage the item's rows (x for fc1, h for fc2) in B-fragment order ----
    const int key = ph * 65536 + rgg;
    if (ok && key != staged) {
      const int vrow = K / 8;   // 16-byte vectors per row
      const int nvec = nrows * vrow;
      for (int i = tid; i < nvec; i += kFusedThreads) {
        const int n = i / vrow, kv = i % vrow;
        const int r = perm_s[off_s[e] + j0 + n];
        uint4 v;
        if (ph == 0)
          v = ld_nc_v4(static_cast<const uint16_t*>(a.x) + (size_t)(r / k) * K + kv * 8);
        else
          v = ld_cg_v4(static_cast<const uint16_t*>(a.hbuf) + (size_t)r * K + kv * 8);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int kk = kv * 8 + 2 * q, kt = kk >> 4, within = kk & 15;
          const int t4 = (within & 7) >> 1, h8 = within >> 3;
          bop[((kt * NG + (n >> 3)) * 32 + (n & 7) * 4 + t4) * 2 + h8] = w4[q];
        }
      }
      if (Kp > K) {
        // K padding meets zero-code weights that are not zero: zero it
        const int pad2 = (Kp - K) / 2;
        for (int i = tid; i < NG * 8 * pad2; i += kFusedThreads) {
          const int n = i / pad2, kk = K + 2 * (i % pad2);
          const int kt = kk >> 4, within = kk & 15;
          const int t4 = (within & 7) >> 1, h8 = within >> 3;
          bop[((kt * NG + (n >> 3)) * 32 + (n & 7) * 4 + t4) * 2 + h8] = 0u;
        }
      }
      staged = key;
    }
    __syncthreads();

    // ---- stream this warp's share of the item's tiles ----
    const int tile = tg * P.tpi + warp / P.ks;
    const int ksl = warp % P.ks;
    const bool gated1 = ph == 0 && a.gated;
    const bool act_warp = ok && tile < P.ntiles;
    FusedAcc fa;
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int q = 0; q < 4; ++q) fa.v[s][n][q] = 0.f;
    if (act_warp) {
      const int kc0 = ksl * P.L.nkc / P.ks, kc1 = (ksl + 1) * P.L.nkc / P.ks;
      const uint8_t* src = P.wpk + (size_t)e * P.L.expert_bytes + (size_t)tile * P.L.tile_bytes +
                           (size_t)kc0 * P.L.scb;
      const FusedGeom gm = fused_geom(P.L);
      const uint32_t* bop_lane = bop + (size_t)kc0 * (SC / 16) * NG * 64 + lane * 2;
      if (ph == 0) {
        const uint32_t zo = (B1 == 8 && BF16) ? zoff_int : zoff_half;
        if (gated1)
          fa = fused_stream_zp<B1, BF16, SC, 2>(src, kc1 - kc0, gm, bop_lane, NG, a.zp_mode, zo);
        else
          fa = fused_stream_zp<B1, BF16, SC, 1>(src, kc1 - kc0, gm, bop_lane, NG, a.zp_mode, zo);
      } else {
        const uint32_t zo = (B2 == 8 && BF16) ? zoff_int : zoff_half;
        fa = fused_stream_zp<B2, BF16, SC, 1>(src, kc1 - kc0, gm, bop_lane, NG, a.zp_mode, zo);
      }
    }
    __syncthreads();   // every warp is done with bop
    if (P.ks > 1) staged = -1;   // the split-K reduction reuses bop
    auto& acc = fa.v;

    // ---- split-K reduction (fixed order) ----
    if (P.ks > 1) {
      if (act_warp && ksl != 0) {
        float* dst = red + (warp * 32 + lane) * 16;
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[(s * 2 + n) * 4 + q] = acc[s][n][q];
      }
      __syncthreads();
      if (act_warp && ksl == 0) {
        for (int o = 1; o < P.ks; ++o) {
          const float* srcr = red + ((warp + o) * 32 + lane) * 16;
#pragma unroll
          for (int s = 0; s < 2; ++s)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
              for (int q = 0; q < 4; ++q) acc[s][n][q] += srcr[(s * 2 + n) * 4 + q];
        }
      }
    }

    // ---- epilogue: acc[s][n][q] = row g + 8 (q >> 1) of the tile, routed row n*8 + 2t + (q & 1) ----
    if (act_warp && ksl == 0) {
      const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
      for (int n = 0; n < 2; ++n) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int row = n * 8 + 2 * t4 + (q & 1);
          const int f = tile * 16 + g + 8 * (q >> 1);
          if (n < NG && row < nrows) {
            const int r = perm_s[off_s[e] + j0 + row];
            if (ph == 0) {
              float hv;
              if (gated1) {
                float gv = acc[0][n][q], uv = acc[1][n][q];
                if (P.bias) {
                  gv += P.bias[((size_t)e * a.I + f) * 2];
                  uv += P.bias[((size_t)e * a.I + f) * 2 + 1];
                }
                hv = glu(a.act, gv, uv);
              } else {
                float v = acc[0][n][q];
                if (P.bias) v += P.bias[(size_t)e * a.I + f];
                hv = act_single(a.act, v);
              }
              if (BF16) static_cast<__nv_bfloat16*>(a.hbuf)[(size_t)r * a.I + f] = __float2bfloat16_rn(hv);
              else static_cast<__half*>(a.hbuf)[(size_t)r * a.I + f] = __float2half_rn(hv);
            } else {
              float v = acc[0][n][q];
              if (P.bias) v += P.bias[(size_t)e * a.H + f];
              a.ybuf[(size_t)r * a.H + f] = v;
            }
          }
        }
      }
      __threadfence();
    }
    __syncthreads();

    // ---- completion: fc1 -> per-expert counter; fc2 -> per output-row group,
    //      the last item of a group adds the k slots in order ----
    if (tid == 0) {
      __threadfence();
      if (ph == 0) {
        atomicAdd(done1 + e, 1);
        bc[4] = 0;
      } else {
        bc[4] = atomicAdd(done2 + tg, 1) == NRG - 1 ? 1 : 0;
      }
    }
    __syncthreads();
    if (bc[4]) {
      __threadfence();
      const int m0 = tg * a.p[1].tpi * 16;
      const int m1 = min(a.H, m0 + a.p[1].tpi * 16);
      const int w4n = (m1 - m0) / 4;
      for (int i = tid; i < T * w4n; i += kFusedThreads) {
        const int t = i / w4n, m = m0 + 4 * (i % w4n);
        float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
          const int r = t * k + j;
          const float wr = w_s[r];
          const uint4 u = ld_cg_v4(a.ybuf + (size_t)r * a.H + m);
          s4.x = fmaf(wr, __uint_as_float(u.x), s4.x);
          s4.y = fmaf(wr, __uint_as_float(u.y), s4.y);
          s4.z = fmaf(wr, __uint_as_float(u.z), s4.z);
          s4.w = fmaf(wr, __uint_as_float(u.w), s4.w);
        }
        const size_t o = (size_t)t * a.H + m;
        if (BF16) {
          store_d<QMOE_BF16>(a.out, o, s4.x); store_d<QMOE_BF16>(a.out, o + 1, s4.y);
          store_d<QMOE_BF16>(a.out, o + 2, s4.z); store_d<QMOE_BF16>(a.out, o + 3, s4.w);
        } else {
          store_d<QMOE_F16>(a.out, o, s4.x); store_d<QMOE_F16>(a.out, o + 1, s4.y);
          store_d<QMOE_F16>(a.out, o + 2, s4.z); store_d<QMOE_F16>(a.out, o + 3, s4.w);
        }
      }
    }
    __syncthreads();
  }

  // ---- the last CTA out clears the counters for the next launch ----
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    bc[5] = atomicAdd(&a.sync[1], 1) == (int)gridDim.x - 1 ? 1 : 0;
  }
  __syncthreads();
  if (bc[5]) {
    __threadfence();
    const int n = kSyncHeader + E + a.n_mg;
    for (int i = tid; i < n; i += kFusedThreads) a.sync[i] = 0;
    __threadfence();
  }
}

}  // namespace qmoe

namespace qmoe {

// Launch of one instantiated width pair (explicitly instantiated in
// qmoe_fused_w<b1><b2>.cu).
template <int B1, int B2>
cudaError_t launch_fused_pair(const FusedArgs& a, bool bf16, int sc, int grid, int smem, cudaStream_t s) {
  auto go = [&](auto kern) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    kern<<<grid, kFusedThreads, smem, s>>>(a);
    return cudaGetLastError();
  };
  if (bf16) return sc == 64 ? go(fused_decode_kernel<B1, B2, true, 64>) : go(fused_decode_kernel<B1, B2, true, 128>);
  return sc == 64 ? go(fused_decode_kernel<B1, B2, false, 64>) : go(fused_decode_kernel<B1, B2, false, 128>);
}

}  // namespace qmoe

namespace qmoe {
// Host side (qmoe_fused.cu).
bool fused_widths_supported(int b1, int b2);
int fused_smem_bytes(int R, int E, int Kp_max);
void fused_item_shape(int ntiles, int nkc, long long nrg_est, int grid, int* tpi, int* ks);
cudaError_t launch_fused(const FusedArgs& a, int b1, int b2, bool bf16, int sc, int grid, int smem,
                         cudaStream_t s);
}  // namespace qmoe
