// Internal declarations shared by the QMoE CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/qmoe.h"

namespace qmoe {

// ----------------------------------------------------------------------------
// Device status word (bounded waits report here instead of hanging/trapping)
// ----------------------------------------------------------------------------
enum : int { DEV_OK = 0, DEV_TIMEOUT = 1 };

struct WaitCfg {
  int* status;            // device int, 0 = ok
  long long limit;        // iterations of a bounded wait before giving up
};

// Polls of the wait that drains a CTA's own in-flight copies after another
// wait ran out (large: those copies always complete).
constexpr long long kDrainWaitLimit = 1LL << 21;

// ----------------------------------------------------------------------------
// Work-list item: (expert, row_start in grouped order, rows, pad)
// ----------------------------------------------------------------------------
struct Item {
  int e, start, rows, pad;
};

// ----------------------------------------------------------------------------
// Decode (mma) prepacked layout of one projection.
//
// A "tile" is 16 output rows (fc2) or 16 gate rows + the matching 16 up rows
// (fc1, so the GLU fuses).  Along K the tile is cut into super-chunks of SC
// = max(64, B) values.  One super-chunk of one 16-row sub-tile holds
//   codes : 32 lanes x (SC*bits/32/16) words in mma-fragment order
//           (int3: a 2-bit plane then a 1-bit plane)
//   scales: [SC/B blocks][8][2] of D: (s[row g], s[row g+8])
//   zp    : [SC/B blocks][8] bytes: z[row g] | z[row g+8] << 4, padded to 16 B
// A super-chunk of the tile is [sub0 codes][sub1 codes][sub0 scales]
// [sub1 scales][sub0 zp][sub1 zp]; the tile is its super-chunks in K order;
// the expert is its tiles in row order.  Every section is 16-byte aligned.
// ----------------------------------------------------------------------------
struct DecodeLayout {
  int bits, B, SC, nkc, nsub, ntiles;
  int code_bytes;    // per sub-tile per super-chunk
  int scale_bytes;   // per sub-tile per super-chunk
  int zp_bytes;      // per sub-tile per super-chunk (0 unless uint8 zp)
  int scb;           // bytes of one super-chunk of a tile (all sub-tiles)
  size_t tile_bytes; // nkc * scb
  size_t expert_bytes;
};

DecodeLayout make_decode_layout(int bits, int B, int N_rows_per_sub, int K, int nsub,
                                int zp_mode, int dsize);

// ----------------------------------------------------------------------------
// Launchers (host side, defined in the .cu files)
// ----------------------------------------------------------------------------
struct RouteArgs {
  const float* logits;
  int T, E, k, normalize;
  int* ids;
  float* w;
  // grouping
  int* counts;
  int* offsets;
  int* perm;
  int* pos;
  Item* items[2];
  int* n_items;          // [2]
  int tb[2];             // rows per item of each class
  int threshold;         // experts with > threshold rows go to class 1
  int cap[2];            // capacity of each item list
  // Grouping spread over the routing CTAs (many routes): per routing CTA and
  // expert, its route count, then the expert's first position for that CTA
  // [ceil(T / 8), E]; per route its rank among its CTA's routes of its
  // expert [R].  Null: one CTA groups.
  int* cntg;
  int* rnk;
  // Unit counts of fc1's overlapped gather, one per class-1 item: cleared
  // here for the GEMM that follows (or null).
  int* gready;
  int gready_n;
};

// Routes per routing CTA (8 tokens of k routes) and whether a forward of T
// tokens takes the grouping spread over the routing CTAs.
__host__ __device__ inline bool route_spread_grouping(const RouteArgs& a, bool fused) {
  return !fused && a.cntg && a.rnk && (long long)a.T * a.k > 1024 && a.k <= 32;
}
// Tokens per routing CTA (8 warps): 8, or with the spread grouping up to 32
// while the CTA's routes stay <= 256 (8 chunks of 32, a warp each).
__host__ __device__ inline int route_tokens_per_cta(const RouteArgs& a, bool spread) {
  if (!spread) return 8;
  const int t = (256 / a.k) & ~7;
  return t > 32 ? 32 : (t < 8 ? 8 : t);
}

cudaError_t launch_route_group(const RouteArgs& a, bool fused, cudaStream_t s);

// Gated activation of fc1's output: SwiGLU (with its attributes) or GeGLU.
struct ActParams {
  int act;                  // QMOE_ACT_* (gated: SWIGLU, GEGLU_TANH)
  float alpha, beta, limit; // SwiGLU only
};

struct RepackArgs {
  const uint8_t* codes;     // canonical [E, N, K*bits/8]
  const void* scales;       // canonical [E, N, K/B], D
  const uint8_t* zp;        // canonical packed zp or null
  uint8_t* out;             // decode layout
  int E, N, K, I_or_0;      // I_or_0 = inter for fc1 (gate/up pairing), 0 for fc2
  int interleaved;          // fc1 canonical rows: 0 = [gate | up], 1 = (gate f, up f) pairs
  int dsize;
  DecodeLayout L;
};
cudaError_t launch_repack_decode(const RepackArgs& a, cudaStream_t s);

struct DecodeArgs {
  const uint8_t* wpk;       // decode layout
  DecodeLayout L;
  int K;                    // real K (<= nkc*SC)
  int N_out;                // output features of this fc (I for fc1, H for fc2)
  const Item* items;
  const int* n_items;
  int max_items;
  // B operand source: fc1 -> x rows by token (perm / k); fc2 -> rows of h
  const void* src;
  const int* perm;
  int k;
  int fc;                   // 1 or 2
  int ng;                   // token groups of 8 per item (1, 2 or 4)
  void* dst;                // fc1: h [R, I] D ; fc2: y [R, H] f32
  ActParams act;
  const float* bias;        // fc1: [E, I, 2] (gate, up) pairs ; fc2: [E, H] ; or null
  int zp_mode;
  float zp_offset;
  int bf16;
  WaitCfg wait;
  int pdl;                  // launch with programmatic dependent launch
  int inject_stall;         // test hook: arm stage 0's barrier, never issue its copy
  // fc2 only: when set, add w[route] * y into out_acc[token, m] (fp32
  // reductions) instead of writing y rows; used when the grouped GEMM also
  // contributes to the same forward.
  int atomic;
  float* out_acc;
  const float* w;
};
cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t s);

struct SimtArgs {
  const uint8_t* codes;     // canonical
  const void* scales;
  const uint8_t* zp;
  int bits, B, K, N_out, I_or_0;
  int zp_bytes_row;
  const Item* items;
  const int* n_items;
  int max_items;
  const void* src;
  const int* perm;
  int k, fc, dtype, zp_mode;
  ActParams act;
  const float* bias;        // fc1: [E, I, 2] (gate, up) pairs ; fc2: [E, H] ; or null
  int interleaved;          // fc1 canonical rows interleaved (gate f = row 2f, up f = row 2f+1)
  float zp_offset;
  void* dst;                // fc1: h [R, I] f32 ; fc2: y [R, H] f32
  int E;
};
cudaError_t launch_simt(const SimtArgs& a, cudaStream_t s);

struct FinalizeArgs {
  const float* y;           // [R, H] grouped order
  const float* w;           // [T*k]
  const int* pos;           // [T*k] grouped position of route r
  void* out;                // [T, H] D
  int T, H, k, dtype;
  int pdl;
};
cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t s);

// Dynamic shared memory of the grouping CTA (routing T tokens in it: T > 0)
// for R routes.
size_t group_smem_bytes(int E, int T, int R, bool spread);

}  // namespace qmoe

// ----------------------------------------------------------------------------
// Device helpers
// ----------------------------------------------------------------------------
#ifdef __CUDACC__
namespace qmoe {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> shared, completing on `bar` (complete_tx).  dst,
// src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// One poll of an mbarrier phase.  The suspend-time hint lets the hardware
// park the warp (up to ~1 us) until the phase completes instead of spinning,
// so waiting warps leave issue slots to the warps that compute.
constexpr uint32_t kSuspendHintNs = 1000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Non-blocking test of an mbarrier phase (no suspension): for the one thread
// whose loop paces a pipeline, where a parked poll would add latency.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: returns false (and records DEV_TIMEOUT) if the phase did not
// complete within `limit` polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  const WaitCfg& w) {
  for (long long i = 0; i < w.limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  atomicExch(w.status, DEV_TIMEOUT);
  return false;
}

// Lanes of the warp holding the same expert id as this lane (ids in
// [0, 2^nbits) or negative = none): one ballot per bit of the id, the same
// mask match.any.sync gives, without its cost.  Negative ids match only
// other negative ids.
__device__ __forceinline__ unsigned peers_of(int e, int nbits) {
  const unsigned valid = __ballot_sync(0xffffffffu, e >= 0);
  unsigned peers = e >= 0 ? valid : ~valid;
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (e >> b) & 1;
    const unsigned m = __ballot_sync(0xffffffffu, bit);
    peers &= bit ? m : ~m;
  }
  return peers;
}

// Bits of an expert id for E experts.
__host__ __device__ __forceinline__ int id_bits(int E) {
  int b = 0;
  while ((1 << b) < E) ++b;
  return b;
}

__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Packed 16-bit pair arithmetic, round-to-nearest-even, no contraction.
template <bool BF16>
__device__ __forceinline__ uint32_t sub2(uint32_t a, uint32_t b);
template <bool BF16>
__device__ __forceinline__ uint32_t mul2(uint32_t a, uint32_t b);

template <>
__device__ __forceinline__ uint32_t sub2<true>(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <>
__device__ __forceinline__ uint32_t sub2<false>(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <>
__device__ __forceinline__ uint32_t mul2<true>(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <>
__device__ __forceinline__ uint32_t mul2<false>(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Magic numbers that turn small codes into exact 16-bit floats with one OR.
//   v:    the pair (M, M) with ulp 1 at M (bf16 M = 128, f16 M = 1024):
//         M | c = M + c, then (M + c) - (M + z) = c - z for integer z;
//   half: the pair (M/2, M/2) with ulp 1/2 there (bf16 64, f16 512):
//         M/2 | (c << 1) = M/2 + c, and M/2 + z is exact for half-integer z.
template <bool BF16>
struct Magic;
template <>
struct Magic<true> {
  static constexpr uint32_t v = 0x43004300u;
  static constexpr uint32_t half = 0x42804280u;
  static constexpr float half_base = 64.f;
};
template <>
struct Magic<false> {
  static constexpr uint32_t v = 0x64006400u;
  static constexpr uint32_t half = 0x60006000u;
  static constexpr float half_base = 512.f;
};

// The pair (M/2 + z, M/2 + z) for a half-integer zero point z.
template <bool BF16>
__device__ __forceinline__ uint32_t half_magic_offset(float z) {
  const float v = Magic<BF16>::half_base + z;
  if (BF16) return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v)) * 0x00010001u;
  return (uint32_t)__half_as_ushort(__float2half_rn(v)) * 0x00010001u;
}

// 8-bit codes.  The pair of 8-bit codes sits in bits 0-7 and 16-23 of b (the
// bits above each are ignored); zq is the zero point of each as the kernels'
// subtrahend: fp16 (M + z, M + z) with M = 1024 (the fp16 significand holds
// M + c exactly); bf16 (z, z), because its 8-bit significand cannot hold
// 128 + c for c >= 128: there each code is split into nibbles, each made
// exact with M = 128, and rejoined as 16 hi + lo (exact below 256) before z
// is subtracted.  Either way the pair c - z is exact.
template <bool BF16>
__device__ __forceinline__ uint32_t fma2(uint32_t a, uint32_t b, uint32_t c);
template <>
__device__ __forceinline__ uint32_t fma2<true>(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
template <>
__device__ __forceinline__ uint32_t fma2<false>(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
template <bool BF16>
__device__ __forceinline__ uint32_t code8_minus_zp(uint32_t b, uint32_t zq) {
  if constexpr (!BF16) {
    return sub2<false>((b & 0x00FF00FFu) | Magic<false>::v, zq);
  } else {
    const uint32_t lo = sub2<true>((b & 0x000F000Fu) | Magic<true>::v, Magic<true>::v);
    const uint32_t hi = sub2<true>(((b >> 4) & 0x000F000Fu) | Magic<true>::v, Magic<true>::v);
    return sub2<true>(fma2<true>(hi, 0x41804180u /* (16, 16) */, lo), zq);
  }
}
// The subtrahend pair of code8_minus_zp for an integer zero point z in [0, 255].
template <bool BF16>
__device__ __forceinline__ uint32_t code8_zq(uint32_t z) {
  if constexpr (BF16) return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn((float)z)) * 0x00010001u;
  else return Magic<false>::v | (z * 0x00010001u);
}

// D = A(16x16, row) * B(16x8, col) + C, fp32 accumulate.
template <bool BF16>
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1);

template <>
__device__ __forceinline__ void mma16816<true>(float* c, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<false>(float* c, const uint32_t* a, uint32_t b0,
                                                uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Loads of one element of D as float.
template <int DT>
__device__ __forceinline__ float load_d(const void* p, size_t i);
template <>
__device__ __forceinline__ float load_d<QMOE_F32>(const void* p, size_t i) {
  return static_cast<const float*>(p)[i];
}
template <>
__device__ __forceinline__ float load_d<QMOE_F16>(const void* p, size_t i) {
  return __half2float(static_cast<const __half*>(p)[i]);
}
template <>
__device__ __forceinline__ float load_d<QMOE_BF16>(const void* p, size_t i) {
  return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

// Round-to-nearest-even into D, back to float.
template <int DT>
__device__ __forceinline__ float round_d(float v);
template <>
__device__ __forceinline__ float round_d<QMOE_F32>(float v) { return v; }
template <>
__device__ __forceinline__ float round_d<QMOE_F16>(float v) {
  return __half2float(__float2half_rn(v));
}
template <>
__device__ __forceinline__ float round_d<QMOE_BF16>(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

template <int DT>
__device__ __forceinline__ void store_d(void* p, size_t i, float v);
template <>
__device__ __forceinline__ void store_d<QMOE_F32>(void* p, size_t i, float v) {
  static_cast<float*>(p)[i] = v;
}
template <>
__device__ __forceinline__ void store_d<QMOE_F16>(void* p, size_t i, float v) {
  static_cast<__half*>(p)[i] = __float2half_rn(v);
}
template <>
__device__ __forceinline__ void store_d<QMOE_BF16>(void* p, size_t i, float v) {
  static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
}

// Four consecutive outputs (element i, i % 4 == 0) rounded into D with one
// store.
template <int DT>
__device__ __forceinline__ void store_d4(void* p, size_t i, float4 v) {
  if constexpr (DT == QMOE_F32) {
    *reinterpret_cast<float4*>(static_cast<float*>(p) + i) = v;
  } else if constexpr (DT == QMOE_F16) {
    const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(static_cast<__half*>(p) + i) = u;
  } else {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p) + i) = u;
  }
}

// Gated activations in fp32 (CUDA's expf / tanhf).
__device__ __forceinline__ float act_silu(float g) {
  return g >= 0.f ? g / (1.f + expf(-g)) : g * expf(g) / (1.f + expf(g));
}
__device__ __forceinline__ float act_gelu_tanh(float g) {
  return 0.5f * g * (1.f + tanhf(0.7978845608028654f * (g + 0.044715f * g * g * g)));
}
// SwiGLU with the qmoe.rs swiglu_value attributes: the gate bounded above by
// `limit`, the linear half clamped to [-limit, limit] (NaN kept), then
// g' * sigmoid(alpha * g') * (u' + beta).  alpha = 1, beta = 0, limit = +inf
// is plain silu(g) * u.
__device__ __forceinline__ float act_swiglu(float g, float u, float alpha, float beta, float limit) {
  g = fminf(g, limit);
  if (!isnan(u)) u = fminf(fmaxf(u, -limit), limit);
  const float z = alpha * g;
  const float sig = z >= 0.f ? 1.f / (1.f + expf(-z)) : expf(z) / (1.f + expf(z));
  return g * sig * (u + beta);
}
__device__ __forceinline__ float glu(const ActParams& p, float g, float u) {
  return p.act == QMOE_ACT_SWIGLU ? act_swiglu(g, u, p.alpha, p.beta, p.limit) : act_gelu_tanh(g) * u;
}
// Non-gated activation of one fc1 output [qmoe.rs qmoe_activate]: relu,
// tanh-GELU, silu (v * stable sigmoid(v)) or identity.
__device__ __forceinline__ float act_single(const ActParams& p, float v) {
  switch (p.act) {
    case QMOE_ACT_RELU: return fmaxf(v, 0.f);
    case QMOE_ACT_GELU_TANH: return act_gelu_tanh(v);
    case QMOE_ACT_SILU: return v * (v >= 0.f ? 1.f / (1.f + expf(-v)) : expf(v) / (1.f + expf(v)));
    default: return v;
  }
}
__host__ __device__ __forceinline__ bool act_gated(int act) {
  return act == QMOE_ACT_SWIGLU || act == QMOE_ACT_GEGLU_TANH;
}

}  // namespace qmoe
#endif
