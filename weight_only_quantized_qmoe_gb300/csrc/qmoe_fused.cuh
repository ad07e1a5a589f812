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
//   * one CTA of 16 warps per SM, launched cooperatively (all CTAs resident:
//     fc2 waits on other CTAs' fc1 results);
//   * every CTA routes all tokens itself (qmoe_topk.cuh: a warp per two
//     tokens, per-lane sorted logits, redux.sync per rank) and builds the
//     grouping in shared memory with every warp at once, so no CTA waits on
//     another before it streams weights;
//   * the work is a list of 16-row weight tiles per phase (fc1 tiles of every
//     (expert, group of <= 16 routed rows) segment, then the fc2 tiles);
//     each CTA takes a contiguous, equal share of each phase, cut at segment
//     boundaries into blocks; a block's tiles, laid end to end with K inside,
//     are cut into equal runs of super-chunks, one per warp;
//   * each warp streams its tiles through a private shared-memory ring of
//     cp.async stages that runs ahead across blocks and phases (weights never
//     wait on anything), dequantises in registers and feeds mma.m16n8k16 with
//     fp32 accumulation; the routed rows of the block's segment are staged
//     once per block in B-fragment order;
//   * a warp finishes the tiles it holds whole; a tile cut between warps is
//     finished, after one CTA barrier, by the warp that holds its first
//     super-chunk, adding the later warps' parked pieces in warp order; then
//     fc1 publishes h and bumps the segment's counter (release), fc2 writes y;
//   * once every CTA is done with fc2 (a grid-wide arrival counter), each CTA
//     adds the k slots in order for an equal share of the outputs and rounds
//     into D;
//   * the last CTA to leave clears the counters for the next launch.
#pragma once
#include <climits>

#include "qmoe_internal.cuh"
#include "qmoe_decode_kernel.cuh"
#include "qmoe_topk.cuh"

namespace qmoe {

// Limits of the single-launch path (checked on the host).
constexpr int kFusedMaxTokens = 64;
constexpr int kFusedMaxExperts = 256;
constexpr int kFusedMaxRoutes = 512;
constexpr int kFusedMaxK = 32;
constexpr int kFusedMaxWarps = 16;   // warps per CTA: 16 (one CTA per SM) or 8 (two)
constexpr int kFusedRowsPerGroup = 16;
constexpr int kFusedStages = 4;      // cp.async ring stages per warp (3 in flight)
// Counters in the sync buffer: [0] launches so far (the epoch), [1] unused,
// [2] a flag nothing sets (the injected stall waits on it), [3] CTAs done
// with fc2 over all launches (launch e waits for gridDim * (e + 1)), then
// done1[segment] (zero between launches).
constexpr int kSyncHeader = 4;

struct FusedProj {
  const uint8_t* wpk;   // decode layout
  DecodeLayout L;
  int K;                // real K
  int ntiles;           // 16-row tiles (fc1: feature tiles, gate + up when gated)
  int g;                // super-chunks per ring stage
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
  int* sync;            // kSyncHeader + max segments ints (zero before the first launch)
  int max_seg;          // capacity of done1
  int ng_max;           // token groups of 8 the B staging is sized for (1 or 2)
  int sb;               // bytes per ring stage
  WaitCfg wait;
  int inject_stall;
  int prefetch_l2;      // every expert's prepacked weights fit the L2: prefetch them during routing
};

// Shared-memory plan of one CTA (the front of dynamic shared memory).
struct FusedPlan {
  int ids_off, w_off, perm_off, cnt_off, off_off, act_off, rgb_off, bop_off, slot_off, ring_off, total;
};

__host__ __device__ inline int fused_align16(int v) { return (v + 15) & ~15; }

// Bytes of the B-operand staging: k-tiles x token groups x 32 lanes x 8 B.
__host__ __device__ inline int fused_bop_bytes(int Kp_max, int ng_max) { return Kp_max / 16 * ng_max * 32 * 8; }

// fp32 partial sums one warp parks for another (a tile piece that does not
// start the tile): per lane acc[sub][group][4] for 2 sub-tiles x ng_max groups.
__host__ __device__ inline int fused_slot_floats(int ng_max) { return 2 * ng_max * 4; }

// Shared memory: broadcast ints, routing and grouping, the B staging, the
// warps' partial-sum slots, then one ring of kFusedStages stages of sb bytes
// per warp.
__host__ __device__ inline FusedPlan fused_plan(int R, int E, int Kp_max, int ng_max, int sb, int warps) {
  FusedPlan p;
  int o = 64;
  p.ids_off = o;  o = fused_align16(o + 4 * R);
  p.w_off = o;    o = fused_align16(o + 4 * R);
  p.perm_off = o; o = fused_align16(o + 4 * R);
  p.cnt_off = o;  o = fused_align16(o + 4 * E);
  p.off_off = o;  o = fused_align16(o + 4 * (E + 1));
  p.act_off = o;  o = fused_align16(o + 4 * E);
  p.rgb_off = o;  o = fused_align16(o + 4 * (E + 1));
  o = (o + 127) & ~127;
  p.bop_off = o;
  o += fused_bop_bytes(Kp_max, ng_max);
  p.slot_off = o;
  o += warps * 32 * fused_slot_floats(ng_max) * 4;
  o = (o + 127) & ~127;
  p.ring_off = o;
  p.total = o + warps * kFusedStages * sb;
  return p;
}

// Scratch of the routing and grouping, in the ring area before the rings
// start: the logits [T, E], the per-chunk expert counts [ceil(R / 32), E]
// (a chunk = 32 consecutive routes), the per-warp totals of the offset scan
// (3 x 8 ints).
struct FusedPrologue {
  int cntw_off, tot_off, total;
};
__host__ __device__ inline FusedPrologue fused_prologue(int T, int E, int R) {
  FusedPrologue q;
  q.cntw_off = fused_align16(T * E * 4);
  q.tot_off = fused_align16(q.cntw_off + (R + 31) / 32 * E * 4);
  q.total = q.tot_off + 3 * 8 * 4;
  return q;
}

// Every token of the forward, two per warp pass, with the key count per
// lane fixed at compile time for E's size class.
template <int NPL>
__device__ __noinline__ void fused_route_all(const float* lg_s, int T, int E, int k, int normalize, int* ids_s,
                                             float* w_s, int warp, int W) {
  for (int t = 2 * warp; t < T; t += 2 * W) topk_route_tokens<NPL, 2>(lg_s, t, T, E, k, normalize, ids_s, w_s);
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

// One super-chunk of the ring (shared memory) into registers.
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
        const uint4 q = *reinterpret_cast<const uint4*>(base + lane * C::WPL + w);
        c.cw[s][w] = q.x; c.cw[s][w + 1] = q.y; c.cw[s][w + 2] = q.z; c.cw[s][w + 3] = q.w;
      }
    } else if constexpr (C::WPL == 2) {
      const uint2 q = *reinterpret_cast<const uint2*>(base + lane * 2);
      c.cw[s][0] = q.x; c.cw[s][1] = q.y;
    } else {
      static_assert(C::WPL == 1, "code words per lane");
      c.cw[s][0] = base[lane];
    }
    if constexpr (BITS == 3) {
#pragma unroll
      for (int w = 0; w < C::WPH; ++w) c.hw[s][w] = base[32 * C::WPL + lane * C::WPH + w];
    }
    const uint8_t* sp = ch + NSUB * gm.code_bytes + s * gm.scale_bytes;
    c.sp[s][0] = *reinterpret_cast<const uint32_t*>(sp + g * 4);
    if constexpr (C::NBKM == 2) c.sp[s][1] = gm.nbk == 2 ? *reinterpret_cast<const uint32_t*>(sp + 32 + g * 4) : c.sp[s][0];
    if (gm.has_zp) {
      const uint8_t* zp = ch + NSUB * (gm.code_bytes + gm.scale_bytes) + s * gm.zp_bytes;
#pragma unroll
      for (int b = 0; b < C::NBKM; ++b) {
        const int bb = (b == 0 || gm.nbk == 2) ? b : 0;
        if constexpr (BITS == 8)
          c.zb[s][b] = (uint32_t)zp[bb * 16 + 2 * g] | ((uint32_t)zp[bb * 16 + 2 * g + 1] << 8);
        else
          c.zb[s][b] = zp[bb * 8 + g];
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
  // fp16 with 2- or 4-bit codes: each code is masked where it sits (one shift
  // per four pairs) over the magic exponent, giving M + m q for a power of two
  // m; one exact fma by 1/m minus (M/m + z) leaves q - z.  cz[s][b][i] holds
  // -(M/m_i + z) of position i (i = 1..3 for 2-bit, i = 1 for 4-bit codes).
  constexpr bool MASKED = !BF16 && (BITS == 2 || BITS == 4);
  uint32_t cz[NSUB][C::NBKM][4];
  if constexpr (MASKED) {
    // -(M/m) for m = 4, 16, 64 (2-bit) or 16 (4-bit); M = 1024, or 512 for
    // the half-unit magic of a fractional zero point
    constexpr uint32_t NEG2[3] = {OFFS ? 0xD800D800u : 0xDC00DC00u, OFFS ? 0xD000D000u : 0xD400D400u,
                                  OFFS ? 0xC800C800u : 0xCC00CC00u};
    constexpr uint32_t NEG4 = OFFS ? 0xD000D000u : 0xD400D400u;
#pragma unroll
    for (int s = 0; s < NSUB; ++s)
#pragma unroll
      for (int b = 0; b < C::NBKM; ++b) {
        // z of row g (even pairs) and row g + 8 (odd pairs), exact in fp16
        const uint32_t zg = OFFS ? sub2<false>(zoff2, Magic<false>::half) : sub2<false>(zz[s][b][0], MAGIC);
        const uint32_t zg8 = OFFS ? zg : sub2<false>(zz[s][b][1], MAGIC);
        if constexpr (BITS == 2) {
          cz[s][b][1] = sub2<false>(NEG2[0], zg8);
          cz[s][b][2] = sub2<false>(NEG2[1], zg);
          cz[s][b][3] = sub2<false>(NEG2[2], zg8);
        } else {
          cz[s][b][1] = sub2<false>(NEG4, zg8);
        }
        cz[s][b][0] = OFFS ? zoff2 : zz[s][b][0];
      }
  }
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    const int b = (C::NBKM == 2 && j >= KT / 2) ? 1 : 0;
    uint32_t afrag[NSUB][4];
    if constexpr (MASKED) {
      constexpr uint32_t BASE = OFFS ? Magic<false>::half : MAGIC;
#pragma unroll
      for (int s = 0; s < NSUB; ++s) {
        uint32_t v[4];
        if constexpr (BITS == 2) {
          // positions 0-3 (even k-tile) or 4-7 (odd) of the word, brought to
          // bits 0-7 (bits 1-8 for the half-unit magic)
          const uint32_t wd = c.cw[s][j >> 1];
          const uint32_t W = (j & 1) ? (OFFS ? wd >> 7 : wd >> 8) : (OFFS ? wd << 1 : wd);
          constexpr uint32_t M0 = OFFS ? 0x00060006u : 0x00030003u;
          constexpr uint32_t SC2[4] = {0u, 0x34003400u, 0x2C002C00u, 0x24002400u};   // 1, 1/4, 1/16, 1/64
          v[0] = sub2<false>((W & M0) | BASE, cz[s][b][0]);
#pragma unroll
          for (int i = 1; i < 4; ++i) v[i] = fma2<false>((W & (M0 << (2 * i))) | BASE, SC2[i], cz[s][b][i]);
        } else {
          const uint32_t wd = c.cw[s][j];
          const uint32_t W0 = OFFS ? wd << 1 : wd, W1 = OFFS ? wd >> 7 : wd >> 8;
          constexpr uint32_t M0 = OFFS ? 0x001E001Eu : 0x000F000Fu;
          v[0] = sub2<false>((W0 & M0) | BASE, cz[s][b][0]);
          v[1] = fma2<false>((W0 & (M0 << 4)) | BASE, 0x2C002C00u, cz[s][b][1]);
          v[2] = sub2<false>((W1 & M0) | BASE, cz[s][b][0]);
          v[3] = fma2<false>((W1 & (M0 << 4)) | BASE, 0x2C002C00u, cz[s][b][1]);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) afrag[s][r] = mul2<false>(v[r], ss[s][b][r & 1]);
      }
    } else {
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
// Bounded acquire wait until *p reaches target (wrap-around safe: the grid
// arrival counter only grows).
__device__ __forceinline__ bool fused_wait_geq(const int* p, int target, const WaitCfg& w) {
  for (long long i = 0; i < w.limit; ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if ((int)((unsigned)v - (unsigned)target) >= 0) return true;
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

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Super-chunk range of warp w in a block of `total` super-chunks: the block's
// tiles laid end to end (tile-major, K inside) and cut into equal runs.
__device__ __forceinline__ int fused_warp_begin(int w, int total, int warps) { return w * total / warps; }

// Active expert of segment `seg` (binary search over the row-group prefix).
__device__ __forceinline__ int fused_seg_expert(int seg, const int* rgb_s, int nact) {
  int lo = 0, hi = nact - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (rgb_s[mid] <= seg) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The ring stages one warp consumes, in order: for phase fc1 then fc2, for
// each block of this CTA's range (a block = tiles of one segment), the
// warp's equal run of the block's super-chunks, cut at tile boundaries into
// pieces, each piece g super-chunks at a time.  The producer runs the same
// walk kFusedStages - 1 stages ahead; the tiles of an expert are contiguous
// in the prepacked layout, so a stage is a pointer bump.
struct FusedCursor {
  int p;                  // phase; 2 = exhausted
  int u, u_end;           // block start (tile index within the phase) and range end
  int c, c_end;           // next super-chunk of the warp's run in the block, run end; c = -1: block not entered
  const uint8_t* src;     // next byte of the current piece
  int left;               // bytes of the piece not yet issued
};

struct FusedRanges {
  int u0[2], u1[2];       // this CTA's tile range per phase
  int ntiles[2], nkc[2];
  int stage_bytes[2];     // g * scb of each phase
};

// Element p (0 or 1) of a two-entry array without a runtime-indexed access
// (which would move the array, or the kernel parameters, to local memory).
template <typename X>
__device__ __forceinline__ X sel2(const X (&v)[2], int p) {
  return p == 0 ? v[0] : v[1];
}

// Move to the next piece at or after the cursor that exists; sets src / left.
__device__ __forceinline__ void fused_cursor_settle(FusedCursor& q, const FusedRanges& rg, const FusedArgs& a,
                                                    int warp, int warps, const int* rgb_s, const int* act_s,
                                                    int nact) {
  for (;;) {
    if (q.p >= 2) return;
    if (q.u >= q.u_end) {
      ++q.p;
      if (q.p < 2) {
        q.u = rg.u0[1];
        q.u_end = rg.u1[1];
        q.c = -1;
      }
      continue;
    }
    const int nt = sel2(rg.ntiles, q.p), nkc = sel2(rg.nkc, q.p);
    const int seg = q.u / nt, t0 = q.u - seg * nt;
    const int n = min(q.u_end - q.u, nt - t0);
    if (q.c < 0) {
      q.c = fused_warp_begin(warp, n * nkc, warps);
      q.c_end = fused_warp_begin(warp + 1, n * nkc, warps);
    }
    if (q.c >= q.c_end) {
      q.u += n;
      q.c = -1;
      continue;
    }
    const int e = act_s[fused_seg_expert(seg, rgb_s, nact)];
    const int tile = q.c / nkc;
    const int pend = min(q.c_end, (tile + 1) * nkc);
    const bool f1 = q.p == 0;
    const uint8_t* wpk = f1 ? a.p[0].wpk : a.p[1].wpk;
    const size_t eb = f1 ? a.p[0].L.expert_bytes : a.p[1].L.expert_bytes;
    const size_t tb = f1 ? a.p[0].L.tile_bytes : a.p[1].L.tile_bytes;
    const int scb = f1 ? a.p[0].L.scb : a.p[1].L.scb;
    q.src = wpk + (size_t)e * eb + (size_t)(t0 + tile) * tb + (size_t)(q.c - tile * nkc) * scb;
    q.left = (pend - q.c) * scb;
    q.c = pend;
    return;
  }
}

// Issue the producer's next stage into `slot` (every lane copies 16-byte
// pieces) and advance; commits one cp.async group either way.
__device__ __forceinline__ void fused_issue(FusedCursor& q, const FusedRanges& rg, const FusedArgs& a, uint8_t* slot,
                                            int lane, int warp, int warps, const int* rgb_s, const int* act_s,
                                            int nact) {
  if (q.p < 2) {
    const int bytes = min(sel2(rg.stage_bytes, q.p), q.left);
    for (int off = lane * 16; off < bytes; off += 512) cp_async16(slot + off, q.src + off);
    q.src += bytes;
    q.left -= bytes;
    if (q.left == 0) fused_cursor_settle(q, rg, a, warp, warps, rgb_s, act_s, nact);
  }
  cp_async_commit();
}

// ----------------------------------------------------------------------------
// The kernel.
// ----------------------------------------------------------------------------
template <int B1, int B2, bool BF16, int SC>
__global__ void __launch_bounds__(kFusedMaxWarps * 32, 1) fused_decode_kernel(const FusedArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int KT = SC / 16;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NT = blockDim.x, W = NT >> 5;
  const int T = a.T, E = a.E, k = a.k, R = T * k;
  const int Kp_max = (a.p[0].L.nkc > a.p[1].L.nkc ? a.p[0].L.nkc : a.p[1].L.nkc) * SC;
  const FusedPlan pl = fused_plan(R, E, Kp_max, a.ng_max, a.sb, W);
  int* bc = reinterpret_cast<int*>(smem);                       // broadcast ints
  int* ids_s = reinterpret_cast<int*>(smem + pl.ids_off);
  float* w_s = reinterpret_cast<float*>(smem + pl.w_off);
  int* perm_s = reinterpret_cast<int*>(smem + pl.perm_off);
  int* cnt_s = reinterpret_cast<int*>(smem + pl.cnt_off);
  int* off_s = reinterpret_cast<int*>(smem + pl.off_off);
  int* act_s = reinterpret_cast<int*>(smem + pl.act_off);      // active experts, ascending
  int* rgb_s = reinterpret_cast<int*>(smem + pl.rgb_off);      // row-group prefix over active experts
  uint32_t* bop = reinterpret_cast<uint32_t*>(smem + pl.bop_off);
  float* slot_s = reinterpret_cast<float*>(smem + pl.slot_off);
  const int SLOTF = fused_slot_floats(a.ng_max);
  uint8_t* ring = smem + pl.ring_off + (size_t)warp * kFusedStages * a.sb;
  int* done1 = a.sync + kSyncHeader;

  // ---- routing (every CTA, all tokens): the logits first land in the
  //      (still empty) ring area with one coalesced pass ----
  float* lg_s = reinterpret_cast<float*>(smem + pl.ring_off);
  // the token rows every CTA stages for fc1 come from the L2 by then: each
  // CTA prefetches an equal 16-byte-aligned slice of x while it routes
  if (tid == NT - 32 && (reinterpret_cast<uintptr_t>(a.x) & 15) == 0) {
    const size_t total = (size_t)T * a.H * 2;   // 16-bit activations; H is a multiple of 32
    const size_t per = ((total + gridDim.x - 1) / gridDim.x + 15) & ~(size_t)15;
    const size_t b0 = per * blockIdx.x;
    if (b0 < total) {
      const uint32_t bytes = (uint32_t)(total - b0 < per ? total - b0 : per);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<const uint8_t*>(a.x) + b0),
                   "r"(bytes)
                   : "memory");
    }
  }
  {
    const int n4 = T * E / 4;   // E is a multiple of 4 on this path
    const float4* src4 = reinterpret_cast<const float4*>(a.logits);
    for (int i = tid; i < n4; i += NT) reinterpret_cast<float4*>(lg_s)[i] = __ldg(src4 + i);
  }
  const FusedPrologue pq = fused_prologue(T, E, R);
  int* cntw_s = reinterpret_cast<int*>(smem + pl.ring_off + pq.cntw_off);
  int* tot_s = reinterpret_cast<int*>(smem + pl.ring_off + pq.tot_off);
  const int NCH = (R + 31) / 32;   // route chunks (<= warps: R <= 32 * warps)
  for (int i = tid; i < NCH * E; i += NT) cntw_s[i] = 0;
  if (tid == 0) bc[6] = *reinterpret_cast<volatile const int*>(a.sync);   // this launch's epoch
  __syncthreads();
  // ---- a layer whose weights fit the L2 many times over (small decode
  //      layers) has them pulled into the L2 while the CTAs route (issued
  //      once the logits are in, so it does not delay them): each CTA
  //      prefetches its equal slice of every expert's prepacked bytes ----
  if (a.prefetch_l2 && tid == NT - 32) {   // one thread of the last warp (it routes last, if at all)
    for (int p = 0; p < 2; ++p) {
      const size_t total = (size_t)E * a.p[p].L.expert_bytes;
      const size_t per = ((total + gridDim.x - 1) / gridDim.x + 15) & ~(size_t)15;
      const size_t b0 = per * blockIdx.x;
      if (b0 < total) {
        const uint32_t bytes = (uint32_t)(total - b0 < per ? total - b0 : per);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.p[p].wpk + b0), "r"(bytes) : "memory");
      }
    }
  }

  if (E <= 32) fused_route_all<1>(lg_s, T, E, k, a.normalize, ids_s, w_s, warp, W);
  else if (E <= 64) fused_route_all<2>(lg_s, T, E, k, a.normalize, ids_s, w_s, warp, W);
  else if (E <= 128) fused_route_all<4>(lg_s, T, E, k, a.normalize, ids_s, w_s, warp, W);
  else fused_route_all<8>(lg_s, T, E, k, a.normalize, ids_s, w_s, warp, W);
  __syncthreads();
  // ---- grouping, every warp at once ----
  // (1) each route chunk's count per expert, and each route's rank among the
  //     chunk's routes of its expert (ballot-built peer masks)
  const unsigned lt = (1u << lane) - 1u;
  const int nb = id_bits(E);
  int my_e = -1, my_rank = 0;
  if (warp < NCH) {
    const int r = warp * 32 + lane;
    my_e = r < R ? ids_s[r] : -1;
    const unsigned peers = peers_of(my_e, nb);
    my_rank = __popc(peers & lt);
    if (my_e >= 0 && my_rank == 0) cntw_s[warp * E + my_e] = __popc(peers);
  }
  __syncthreads();
  // (2) a lane per expert: counts = sum over chunks (chunk entries become
  //     exclusive prefixes); per 32 experts, scans of rows and row groups
  //     and the ballot of active experts
  const int NEW = (E + 31) / 32;
  int sc_c = 0, sc_g = 0, my_c = 0, my_g = 0;
  unsigned act_mask = 0;
  if (warp < NEW) {
    const int e = warp * 32 + lane;
    if (e < E) {
      for (int ch = 0; ch < NCH; ++ch) {
        const int v = cntw_s[ch * E + e];
        cntw_s[ch * E + e] = my_c;
        my_c += v;
      }
      cnt_s[e] = my_c;
    }
    my_g = (my_c + kFusedRowsPerGroup - 1) / kFusedRowsPerGroup;
    sc_c = my_c;
    sc_g = my_g;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nc = __shfl_up_sync(0xffffffffu, sc_c, o);
      const int ng = __shfl_up_sync(0xffffffffu, sc_g, o);
      if (lane >= o) { sc_c += nc; sc_g += ng; }
    }
    act_mask = __ballot_sync(0xffffffffu, my_c > 0);
    if (lane == 31) {
      tot_s[warp] = sc_c;
      tot_s[8 + warp] = sc_g;
      tot_s[16 + warp] = __popc(act_mask);
    }
  }
  __syncthreads();
  // (3) offsets, the active-expert list and the row-group prefix
  if (warp < NEW) {
    int pc = 0, pg = 0, pa = 0;
    for (int w2 = 0; w2 < warp; ++w2) {
      pc += tot_s[w2];
      pg += tot_s[8 + w2];
      pa += tot_s[16 + w2];
    }
    const int e = warp * 32 + lane;
    if (e < E) off_s[e] = pc + sc_c - my_c;
    if (my_c > 0) {
      const int ai = pa + __popc(act_mask & lt);
      act_s[ai] = e;
      rgb_s[ai] = pg + sc_g - my_g;
    }
    if (warp == NEW - 1 && lane == 31) {
      const int nact = pa + __popc(act_mask), nrg = pg + sc_g;
      off_s[E] = pc + sc_c;
      rgb_s[nact] = nrg;
      bc[0] = nact;
      bc[1] = nrg;
    }
  }
  __syncthreads();
  // (4) the stable permutation: routes of an expert in ascending route order
  if (my_e >= 0) perm_s[off_s[my_e] + cntw_s[warp * E + my_e] + my_rank] = warp * 32 + lane;
  __syncthreads();
  const int nact = bc[0], NRG = bc[1];

  // ---- this CTA's share of the tiles of each phase; start the weight ring ----
  FusedRanges rg;
  for (int p = 0; p < 2; ++p) {
    rg.ntiles[p] = a.p[p].ntiles;
    rg.nkc[p] = a.p[p].L.nkc;
    rg.stage_bytes[p] = a.p[p].g * a.p[p].L.scb;
    // N <= (E + R / 16 + 1) * 512 and gridDim.x <= 152 * 2: the products fit 32 bits
    const unsigned N = (unsigned)NRG * (unsigned)rg.ntiles[p];
    rg.u0[p] = (int)(N * blockIdx.x / gridDim.x);
    rg.u1[p] = (int)(N * (blockIdx.x + 1) / gridDim.x);
  }
  FusedCursor prod;
  prod.p = 0;
  prod.u = rg.u0[0];
  prod.u_end = rg.u1[0];
  prod.c = -1;
  prod.c_end = 0;
  prod.src = nullptr;
  prod.left = 0;
  fused_cursor_settle(prod, rg, a, warp, W, rgb_s, act_s, nact);
  for (int s = 0; s < kFusedStages - 1; ++s)
    fused_issue(prod, rg, a, ring + s * a.sb, lane, warp, W, rgb_s, act_s, nact);
  int stage = 0;   // ring stages this warp has consumed

  // CTA 0 keeps the routing and the row-group work-list for the host.
  if (blockIdx.x == 0) {
    for (int r = tid; r < R; r += NT) {
      a.ids[r] = ids_s[r];
      a.w[r] = w_s[r];
      a.perm[r] = perm_s[r];
    }
    for (int e = tid; e <= E; e += NT) {
      a.offsets[e] = off_s[e];
      if (e < E) a.counts[e] = cnt_s[e];
    }
    for (int ai = tid; ai < nact; ai += NT) {
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

  // Fractional zero point: the half-unit magic offset (M/2 + z, M/2 + z);
  // 8-bit codes in bf16 take the integer pair (z, z) instead.
  uint32_t zoff_half = 0u, zoff_int = 0u;
  if (a.zp_mode == QMOE_ZP_OFFSET) {
    zoff_half = half_magic_offset<BF16>(a.zp_offset);
    zoff_int = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a.zp_offset)) * 0x00010001u;
  }
  const bool offs = a.zp_mode == QMOE_ZP_OFFSET;
  const bool uint8_zp = a.zp_mode == QMOE_ZP_UINT8;
  int staged = -1;   // (phase, segment) whose rows are in bop

#pragma unroll   // compile-time phase: the projection's parameters stay in the constant bank
  for (int ph = 0; ph < 2; ++ph) {
    const FusedProj& P = a.p[ph];
    const int nt = P.ntiles, nkc = P.L.nkc, K = P.K, Kp = nkc * SC;
    const FusedGeom gm = fused_geom(P.L);
    for (int u = rg.u0[ph]; u < rg.u1[ph];) {
      // ---- one block: tiles [t0, t0 + n) of segment seg ----
      const int seg = u / nt, t0 = u % nt;
      const int n = min(rg.u1[ph] - u, nt - t0);
      const int ai = fused_seg_expert(seg, rgb_s, nact);
      const int e = act_s[ai], c = cnt_s[e];
      const int j0 = (seg - rgb_s[ai]) * kFusedRowsPerGroup;
      const int nrows = min(kFusedRowsPerGroup, c - j0);
      const int NG = (nrows + 7) >> 3;

      if (ph == 1) {
        // the h rows of this segment: every fc1 tile of the segment done
        if (tid == 0)
          bc[3] = (a.inject_stall ? fused_wait_geq(a.sync + 2, 1, a.wait)
                                  : fused_wait_geq(done1 + seg, rg.ntiles[0], a.wait)) ? 1 : 0;
        __syncthreads();
      }
      const int key = ph * 65536 + seg;
      if (key != staged) {
        const int vrow = K / 8;   // 16-byte vectors per row
        const int nvec = nrows * vrow;
        for (int i = tid; i < nvec; i += NT) {
          const int nn = i / vrow, kv = i % vrow;
          const int r = perm_s[off_s[e] + j0 + nn];
          const uint4 v = ph == 0 ? ld_nc_v4(static_cast<const uint16_t*>(a.x) + (size_t)(r / k) * K + kv * 8)
                                  : ld_cg_v4(static_cast<const uint16_t*>(a.hbuf) + (size_t)r * K + kv * 8);
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int kk = kv * 8 + 2 * q, kt = kk >> 4, within = kk & 15;
            const int t4 = (within & 7) >> 1, h8 = within >> 3;
            bop[((kt * NG + (nn >> 3)) * 32 + (nn & 7) * 4 + t4) * 2 + h8] = w4[q];
          }
        }
        if (Kp > K) {
          // K padding meets zero-code weights that are not zero: zero it
          const int pad2 = (Kp - K) / 2;
          for (int i = tid; i < NG * 8 * pad2; i += NT) {
            const int nn = i / pad2, kk = K + 2 * (i % pad2);
            const int kt = kk >> 4, within = kk & 15;
            const int t4 = (within & 7) >> 1, h8 = within >> 3;
            bop[((kt * NG + (nn >> 3)) * 32 + (nn & 7) * 4 + t4) * 2 + h8] = 0u;
          }
        }
        staged = key;
      }
      __syncthreads();

      const bool gated1 = ph == 0 && a.gated;
      const uint32_t zo = ((ph == 0 ? B1 : B2) == 8 && BF16) ? zoff_int : zoff_half;
      float acc[2][2][4];
      auto epilogue = [&](int tile) {
        const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int nn = 0; nn < 2; ++nn) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int row = nn * 8 + 2 * t4 + (q & 1);
            const int f = tile * 16 + g + 8 * (q >> 1);
            if (nn < NG && row < nrows) {
              const int r = perm_s[off_s[e] + j0 + row];
              if (ph == 0) {
                float hv;
                if (gated1) {
                  float gv = acc[0][nn][q], uv = acc[1][nn][q];
                  if (P.bias) {
                    gv += P.bias[((size_t)e * a.I + f) * 2];
                    uv += P.bias[((size_t)e * a.I + f) * 2 + 1];
                  }
                  hv = glu(a.act, gv, uv);
                } else {
                  float vv = acc[0][nn][q];
                  if (P.bias) vv += P.bias[(size_t)e * a.I + f];
                  hv = act_single(a.act, vv);
                }
                if (BF16) static_cast<__nv_bfloat16*>(a.hbuf)[(size_t)r * a.I + f] = __float2bfloat16_rn(hv);
                else static_cast<__half*>(a.hbuf)[(size_t)r * a.I + f] = __float2half_rn(hv);
              } else {
                float vv = acc[0][nn][q];
                if (P.bias) vv += P.bias[(size_t)e * a.H + f];
                a.ybuf[(size_t)r * a.H + f] = vv;
              }
            }
          }
        }
      };

      // ---- this warp's run of the block's super-chunks, piece by piece ----
      const int total = n * nkc;
      const int cb1 = fused_warp_begin(warp + 1, total, W);
      int own_tile = -1;   // a tile this warp started but did not finish
      for (int ci = fused_warp_begin(warp, total, W); ci < cb1;) {
        const int tile = ci / nkc, kc0 = ci - tile * nkc;
        const int pend = min(cb1, (tile + 1) * nkc), len = pend - ci;
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
          for (int nn = 0; nn < 2; ++nn)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[s][nn][q] = 0.f;
        for (int cc = 0; cc < len;) {
          const int nck = min(P.g, len - cc);
          // stage `stage` of the ring holds super-chunks [kc0 + cc, kc0 + cc + nck) of the tile
          // stages 0..stage have landed (the kFusedStages - 2 newer ones may not)
          cp_async_wait<kFusedStages - 2>();
          __syncwarp();
          const uint8_t* slot = ring + (stage % kFusedStages) * a.sb;
          // refill the stage consumed last (the slot before this one)
          fused_issue(prod, rg, a, ring + ((stage + kFusedStages - 1) % kFusedStages) * a.sb, lane, warp, W, rgb_s,
                      act_s, nact);
          for (int x = 0; x < nck; ++x) {
            const uint8_t* ch = slot + x * gm.scb;
            const uint32_t* bl = bop + (size_t)(kc0 + cc + x) * KT * NG * 64 + lane * 2;
            if (ph == 0) {
              if (gated1) {
                FusedChunk<B1, SC, 2> cr;
                fused_load_chunk<B1, SC, 2>(cr, ch, gm, lane);
                if (offs) fused_compute_chunk<B1, BF16, SC, 2, true>(cr, bl, NG, false, zo, acc);
                else fused_compute_chunk<B1, BF16, SC, 2, false>(cr, bl, NG, uint8_zp, zo, acc);
              } else {
                FusedChunk<B1, SC, 1> cr;
                fused_load_chunk<B1, SC, 1>(cr, ch, gm, lane);
                if (offs) fused_compute_chunk<B1, BF16, SC, 1, true>(cr, bl, NG, false, zo, acc);
                else fused_compute_chunk<B1, BF16, SC, 1, false>(cr, bl, NG, uint8_zp, zo, acc);
              }
            } else {
              FusedChunk<B2, SC, 1> cr;
              fused_load_chunk<B2, SC, 1>(cr, ch, gm, lane);
              if (offs) fused_compute_chunk<B2, BF16, SC, 1, true>(cr, bl, NG, false, zo, acc);
              else fused_compute_chunk<B2, BF16, SC, 1, false>(cr, bl, NG, uint8_zp, zo, acc);
            }
          }
          __syncwarp();
          ++stage;
          cc += nck;
        }
        if (len == nkc) {
          epilogue(t0 + tile);                 // the whole tile
        } else if (kc0 > 0) {
          // the tail of a tile an earlier warp started (only a run's first
          // piece can be one): park it for that warp
          float* dst = slot_s + (warp * 32 + lane) * SLOTF;
#pragma unroll
          for (int s2 = 0; s2 < 2; ++s2)
#pragma unroll
            for (int nn = 0; nn < 2; ++nn)
              if (nn < NG)
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[(s2 * NG + nn) * 4 + q] = acc[s2][nn][q];
        } else {
          own_tile = tile;                     // the head of a tile (only a run's last piece)
        }
        ci = pend;
      }
      __syncthreads();   // every warp is done with bop; the parked pieces are visible

      // ---- a tile split over warps: its first warp adds the later pieces in
      //      warp order (each later warp's run begins inside the tile) ----
      if (own_tile >= 0) {
        const int tile_end = (own_tile + 1) * nkc;
        for (int w2 = warp + 1; w2 < W; ++w2) {
          const int b0 = fused_warp_begin(w2, total, W);
          if (b0 >= tile_end) break;
          if (fused_warp_begin(w2 + 1, total, W) == b0) continue;   // an empty run
          const float* src = slot_s + (w2 * 32 + lane) * SLOTF;
#pragma unroll
          for (int s2 = 0; s2 < 2; ++s2)
#pragma unroll
            for (int nn = 0; nn < 2; ++nn)
              if (nn < NG)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[s2][nn][q] += src[(s2 * NG + nn) * 4 + q];
        }
        epilogue(t0 + own_tile);
      }
      __syncthreads();   // the block's h / y stores are issued; the slots are free

      // ---- completion: fc1 publishes the segment's h rows (release) ----
      if (ph == 0 && tid == 0)
        asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(done1 + seg), "r"(n) : "memory");
      u += n;
    }
  }
  cp_async_wait<0>();   // the producer's trailing (empty) groups

  // ---- every y row is written once all CTAs arrive; then each CTA adds the
  //      k slots in order for its equal share of the outputs.  The arrival
  //      counter only grows (this launch's target: gridDim * (epoch + 1)),
  //      so no CTA has to reset it: the last CTA to arrive clears the
  //      segment counters (no CTA reads them any more) and bumps the epoch
  //      for the next launch, and every CTA leaves right after its share ----
  __syncthreads();
  if (tid == 0) {
    const unsigned target = (unsigned)gridDim.x * (unsigned)(bc[6] + 1);
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(a.sync + 3) : "memory");
    if ((unsigned)old + 1u == target) {
      for (int i = 0; i < a.max_seg; ++i) done1[i] = 0;
      *reinterpret_cast<volatile int*>(a.sync) = bc[6] + 1;
    } else {
      fused_wait_geq(a.sync + 3, (int)target, a.wait);
    }
  }
  __syncthreads();
  {
    const int H4 = a.H / 4;
    const long long N = (long long)T * H4;
    const int i0 = (int)(N * blockIdx.x / gridDim.x), i1 = (int)(N * (blockIdx.x + 1) / gridDim.x);
    for (int idx = i0 + tid; idx < i1; idx += NT) {
      const int t = idx / H4, m = 4 * (idx % H4);
      float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < k; ++j) {
        const int r = t * k + j;
        const float wr = w_s[r];
        const uint4 uu = ld_cg_v4(a.ybuf + (size_t)r * a.H + m);
        s4.x = fmaf(wr, __uint_as_float(uu.x), s4.x);
        s4.y = fmaf(wr, __uint_as_float(uu.y), s4.y);
        s4.z = fmaf(wr, __uint_as_float(uu.z), s4.z);
        s4.w = fmaf(wr, __uint_as_float(uu.w), s4.w);
      }
      const size_t o = (size_t)t * a.H + m;
      if (BF16) store_d4<QMOE_BF16>(a.out, o, s4);
      else store_d4<QMOE_F16>(a.out, o, s4);
    }
  }

}

// Launch of one instantiated width pair (explicitly instantiated in
// qmoe_fused_w<b1><b2>.cu): cooperative, so every CTA is resident.
template <int B1, int B2>
cudaError_t launch_fused_pair(const FusedArgs& a, bool bf16, int sc, int grid, int warps, int smem, cudaStream_t s) {
  auto go = [&](auto kern) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(warps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
  };
  if (bf16) return sc == 64 ? go(fused_decode_kernel<B1, B2, true, 64>) : go(fused_decode_kernel<B1, B2, true, 128>);
  return sc == 64 ? go(fused_decode_kernel<B1, B2, false, 64>) : go(fused_decode_kernel<B1, B2, false, 128>);
}

// Host side (qmoe_fused.cu).
bool fused_widths_supported(int b1, int b2);
// Bytes per ring stage and super-chunks per stage of each projection for the
// shared memory left after `fixed_bytes`; false if a stage cannot hold one
// super-chunk.
bool fused_ring_shape(int budget, int fixed_bytes, int warps, int scb1, int scb2, int* sb, int* g1, int* g2);
cudaError_t launch_fused(const FusedArgs& a, int b1, int b2, bool bf16, int sc, int grid, int warps, int smem,
                         cudaStream_t s);

}  // namespace qmoe
