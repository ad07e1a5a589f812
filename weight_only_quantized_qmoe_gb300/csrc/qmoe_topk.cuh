// Warp-level top-k routing of QMoE tokens, shared by the single-launch
// forward and the separate routing kernels.
//
// Definition followed: onnx-runtime-ep-cuda src/kernels/qmoe.rs (CUDA_SRC,
// total_order_key / route_value_is_better / qmoe_route): experts are ranked
// by a total-order key of the fp32 logit, ties to the lower expert index; the
// weight of a chosen expert is exp(l - max) over the sum of exp(l - max) of
// all E experts, or of the k chosen when renormalising.
//
// GB300 form (ours): one warp ranks a token.  Lane l holds the logits of
// experts l, l + 32, ... (NPL of them) as (key, index) pairs and sorts them
// once, best first; a rank is then one warp-wide redux.sync max of the lanes'
// heads and one redux.sync min of the indices at that key (the tie rule),
// and the lane that owned the winner drops its head.  TOK tokens run
// interleaved so their dependency chains overlap.
#pragma once
#include <climits>

#include "qmoe_internal.cuh"

namespace qmoe {

__device__ __forceinline__ int topk_redux_max(int v) {
  int r;
  asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}
__device__ __forceinline__ int topk_redux_min(int v) {
  int r;
  asm volatile("redux.sync.min.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

// Signed integer whose order is the total order of the fp32 values.
__device__ __forceinline__ int topk_order_key(float v) {
  const int b = __float_as_int(v);
  return b ^ ((b >> 31) & 0x7fffffff);
}

// (key, index) a ranks before b: larger key, or equal key and lower index.
__device__ __forceinline__ bool topk_before(int ka, int ia, int kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

template <int NPL>
__device__ __forceinline__ void topk_sort(int (&key)[NPL], int (&idx)[NPL]) {
  // odd-even transposition: NPL rounds of neighbour compare-exchanges
#pragma unroll
  for (int round = 0; round < NPL; ++round) {
#pragma unroll
    for (int i = round & 1; i + 1 < NPL; i += 2) {
      if (topk_before(key[i + 1], idx[i + 1], key[i], idx[i])) {
        const int tk = key[i], ti = idx[i];
        key[i] = key[i + 1];
        idx[i] = idx[i + 1];
        key[i + 1] = tk;
        idx[i + 1] = ti;
      }
    }
  }
}

// Tokens t0 .. t0 + TOK - 1 (those < T) of the logits lg[T, E] (shared or
// global memory): ids[t * k + j] = the expert of rank j, w[t * k + j] its
// weight.  Called by all 32 lanes of a warp; E <= 32 * NPL, k <= 32.
template <int NPL, int TOK>
__device__ __forceinline__ void topk_route_tokens(const float* lg_all, int t0, int T, int E, int k, int normalize,
                                                  int* ids, float* w) {
  const int lane = threadIdx.x & 31;
  int key[TOK][NPL], idx[TOK][NPL];
  int mine[TOK], top[TOK];
#pragma unroll
  for (int u = 0; u < TOK; ++u) {
    mine[u] = 0;
    top[u] = 0;
    const float* lg = lg_all + (size_t)min(t0 + u, T - 1) * E;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      // experts past E rank after every real one (lowest key, index >= E)
      key[u][i] = e < E ? topk_order_key(lg[e]) : INT_MIN;
      idx[u][i] = e;
    }
    topk_sort<NPL>(key[u], idx[u]);
  }
  for (int slot = 0; slot < k; ++slot) {
    int m[TOK];
#pragma unroll
    for (int u = 0; u < TOK; ++u) m[u] = topk_redux_max(key[u][0]);
#pragma unroll
    for (int u = 0; u < TOK; ++u) {
      const int sel = topk_redux_min(key[u][0] == m[u] ? idx[u][0] : INT_MAX);
      if (lane == slot) mine[u] = sel;
      if (slot == 0) top[u] = sel;
      const bool pop = (sel & 31) == lane;   // expert e sits in lane e % 32
#pragma unroll
      for (int i = 0; i + 1 < NPL; ++i) {
        key[u][i] = pop ? key[u][i + 1] : key[u][i];
        idx[u][i] = pop ? idx[u][i + 1] : idx[u][i];
      }
      if (pop) {
        key[u][NPL - 1] = INT_MIN;
        idx[u][NPL - 1] = INT_MAX;
      }
    }
  }
#pragma unroll
  for (int u = 0; u < TOK; ++u) {
    const int t = t0 + u;
    if (t >= T) break;
    const float* lg = lg_all + (size_t)t * E;
    const float mx = lg[top[u]];   // the top-ranked logit is the maximum
    const float p = lane < k ? expf(lg[mine[u]] - mx) : 0.f;
    float den = p;
    if (normalize) {
      // butterfly over the k lanes holding the chosen experts' terms
      for (int o = 1; o < k; o <<= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    } else {
      den = 0.f;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) den += expf(lg[e] - mx);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    }
    if (lane < k) {
      ids[t * k + lane] = mine[u];
      w[t * k + lane] = p / den;
    }
  }
}

}  // namespace qmoe
