// Routing (top-k + softmax weights), expert grouping, tile work-lists and the
// slot-ordered combine of the QMoE layer forward.
//
// Routing follows onnx-runtime-ep-cuda src/kernels/qmoe.rs (CUDA_SRC,
// total_order_key / route_value_is_better / qmoe_route): experts are ranked
// by a total-order key of the fp32 logit, ties to the lower index; the
// weight of a selected expert is exp(l - max_all) divided by the sum over all
// E experts, or over the k chosen when renormalising.  Here one warp ranks a
// token (qmoe_topk.cuh for E <= 256; k warp-wide shuffle arg-max rounds
// above) instead of one thread per token.
//
// Grouping replaces that page's count / 1-thread prefix / atomic-cursor
// assignment with one CTA that builds a *stable* permutation (routes of an
// expert in ascending route order), so the result is deterministic.  The
// work-lists follow metrale gemm_quant_moe.rs moe_build_tile_worklist
// (experts ascending, then m-tile); each item carries its row range.
#include <climits>

#include "qmoe_internal.cuh"
#include "qmoe_topk.cuh"

namespace qmoe {

__device__ __forceinline__ int total_order_key(float v) {
  int b = __float_as_int(v);
  return b ^ ((b >> 31) & 0x7fffffff);
}

// One warp ranks the E logits of one token and writes ids[0..k) and
// w[0..k).  NPL = logits held per lane (E <= 32 * NPL); used for E > 256,
// where sorting each lane's logits would not pay.
template <int NPL>
__device__ void route_token(const float* __restrict__ lg, int E, int k, int normalize,
                            int* __restrict__ ids, float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  int key[NPL];
  uint32_t taken = 0;  // bit i: logit lane + 32 i is selected or absent
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float v = lg[e];
      key[i] = total_order_key(v);
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

  float sum_sel = 0.f;
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
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const int ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ok > bk || (ok == bk && oi < bi)) {
        bk = ok;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == 0) ids[slot] = bi;
    sum_sel += expf(lg[bi] - mx);
  }
  __syncwarp();
  const float denom = normalize ? sum_sel : sum_all;
  for (int slot = lane; slot < k; slot += 32) w[slot] = expf(lg[ids[slot]] - mx) / denom;
}

// Tokens [t0, t0 + TOK) of the forward (those < T) by one warp.
template <int NPL, int TOK>
__device__ __forceinline__ void route_warp(const float* lg, int t0, const RouteArgs& a) {
  if constexpr (NPL <= 8) {
    if (a.k <= 32) {   // a lane per rank
      topk_route_tokens<NPL, TOK>(lg, t0, a.T, a.E, a.k, a.normalize, a.ids, a.w);
      return;
    }
  }
#pragma unroll
  for (int u = 0; u < TOK; ++u)
    if (t0 + u < a.T)
      route_token<NPL>(lg + (size_t)(t0 + u) * a.E, a.E, a.k, a.normalize, a.ids + (size_t)(t0 + u) * a.k,
                       a.w + (size_t)(t0 + u) * a.k);
}

// TPB tokens per CTA (route_tokens_per_cta), two at a time per warp.  With
// the spread grouping the CTA then counts its TPB * k <= 256 routes per
// expert (a warp per chunk of 32 routes, ballot-built peer masks) into
// cntg[blockIdx.x], and stores each route's rank among the CTA's routes of
// its expert (stable) in rnk.  Dynamic shared memory: [8][E] ints with the
// spread grouping.
template <int NPL>
__global__ void __launch_bounds__(256) route_kernel(const RouteArgs a, int spread) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int TPB = route_tokens_per_cta(a, spread != 0);
  for (int t = blockIdx.x * TPB + 2 * warp; t < min(a.T, (blockIdx.x + 1) * TPB); t += 16)
    route_warp<NPL, 2>(a.logits, t, a);
  if (spread) {
    extern __shared__ int cc[];   // [8][E]
    const int E = a.E, R = a.T * a.k;
    for (int i = tid; i < 8 * E; i += 256) cc[i] = 0;
    __syncthreads();              // also: every ids write of the CTA is visible
    const int rb0 = blockIdx.x * TPB * a.k, rb1 = min(R, rb0 + TPB * a.k);
    const int nch = (rb1 - rb0 + 31) / 32;   // <= 8 (k <= 32)
    const unsigned lt = (1u << lane) - 1u;
    int e = -1, rank = 0;
    if (warp < nch) {
      const int r = rb0 + warp * 32 + lane;
      e = r < rb1 ? a.ids[r] : -1;
      const unsigned peers = peers_of(e, id_bits(E));
      rank = __popc(peers & lt);
      if (e >= 0 && rank == 0) cc[warp * E + e] = __popc(peers);
    }
    __syncthreads();
    for (int x = tid; x < E; x += 256) {
      int run = 0;
      for (int w = 0; w < nch; ++w) {
        const int c = cc[w * E + x];
        cc[w * E + x] = run;
        run += c;
      }
      a.cntg[(size_t)blockIdx.x * E + x] = run;
    }
    __syncthreads();
    if (e >= 0) a.rnk[rb0 + warp * 32 + lane] = cc[warp * E + e] + rank;
  }
  pdl_launch_dependents();
}

// Spread grouping, last step: each route's position = its expert's first
// position for its routing CTA + its rank there; the permutation and its
// inverse.
__global__ void __launch_bounds__(256) scatter_kernel(const RouteArgs a) {
  pdl_wait();
  const int R = a.T * a.k;
  const int r = blockIdx.x * 256 + threadIdx.x;
  if (r < R) {
    const int e = a.ids[r];
    const int p = a.cntg[(size_t)(r / (route_tokens_per_cta(a, true) * a.k)) * a.E + e] + a.rnk[r];
    a.perm[p] = r;
    a.pos[r] = p;
  }
  pdl_launch_dependents();
}

// Exclusive scan of v over the 1024 threads of the block; returns the
// exclusive prefix, *total gets the sum.  ws: 32 ints of shared memory.
__device__ int block_exclusive_scan(int v, int* ws, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) ws[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = ws[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    ws[lane] = s;
  }
  __syncthreads();
  const int excl = incl - v + (warp > 0 ? ws[warp - 1] : 0);
  *total = ws[31];
  __syncthreads();
  return excl;
}

// The single-CTA routing stages the logits when they take at most 64 KB.
__host__ __device__ inline bool group_stages_logits(int T, int E) { return (int64_t)T * E <= 16384; }
// The grouping CTA builds the permutation of R > 1024 routes in shared
// memory when cnt, off, ws and the R ints take at most 200 KB.
__host__ __device__ inline bool group_perm_in_smem(int R, int E) {
  return R > 1024 && (int64_t)(33 * E + 32 + R) * 4 <= 200 * 1024;
}

// Work-lists: class 0 (decode kernel) for experts with 1..threshold rows,
// class 1 (grouped GEMM) above; each cut into items of tb[cls] rows.  Thread
// e < E holds expert e's row count and row offset; all threads call it.
__device__ void build_worklists(const RouteArgs& a, int count, int excl, int* ws) {
  const int tid = threadIdx.x;
  for (int cls = 0; cls < 2; ++cls) {
    const int tb = a.tb[cls];
    int nb = 0;
    if (tid < a.E && count > 0 && ((count > a.threshold) == (cls == 1))) nb = (count + tb - 1) / tb;
    int ntot;
    const int ib = block_exclusive_scan(nb, ws, &ntot);
    for (int i = 0; i < nb; ++i) {
      if (ib + i < a.cap[cls]) {
        Item it;
        it.e = tid;
        it.start = excl + i * tb;
        it.rows = min(tb, count - i * tb);
        it.pad = 0;
        a.items[cls][ib + i] = it;
      }
    }
    if (tid == 0) a.n_items[cls] = min(ntot, a.cap[cls]);
  }
}

// One CTA of 1024 threads: optional routing of all tokens (small T), then
// counts, offsets, the stable permutation, its inverse and both work-lists.
// Shared memory: cnt[32][E] (per-warp, per-expert counts, later bases),
// off[E], scan scratch.
template <int NPL>
__global__ void __launch_bounds__(1024) group_kernel(const RouteArgs a, int do_route) {
  extern __shared__ int smem[];
  const int E = a.E;
  const bool spread = !do_route && route_spread_grouping(a, false);
  int* cnt = smem;                                               // [32][E] (spread: [P][E], P * E <= 1024)
  int* off = smem + (spread ? max(32 * E, 1024) : 32 * E);       // [E]
  int* ws = off + E;                                             // [32]
  float* lg_s = reinterpret_cast<float*>(ws + 32);               // [T, E] when staged
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = a.T * a.k;
  const int nb = id_bits(E);
  if (a.gready) {
    // after the previous forward's GEMMs (stream order; launched here after
    // the routing CTAs' completion when they run first)
    if (!do_route) pdl_wait();
    for (int i = tid; i < a.gready_n; i += blockDim.x) a.gready[i] = 0;
  }

  if (spread) {
    // ---- counts per routing CTA are in cntg: thread (part, e) walks expert
    //      e's column over a contiguous range of routing CTAs, twice ----
    pdl_wait();
    int* psum = cnt;
    const int TPB = route_tokens_per_cta(a, true);
    const int nblk = (a.T + TPB - 1) / TPB;
    const int P = E >= 1024 ? 1 : 1024 / E;
    const int e = tid % E, part = tid / E;
    const bool mine = part < P;
    const int b0 = mine ? (int)((long long)part * nblk / P) : 0;
    const int b1 = mine ? (int)((long long)(part + 1) * nblk / P) : 0;
    int s = 0;
#pragma unroll 8
    for (int b = b0; b < b1; ++b) s += a.cntg[(size_t)b * E + e];
    if (mine) psum[part * E + e] = s;
    __syncthreads();
    int count = 0;
    if (tid < E) {
      for (int q = 0; q < P; ++q) {
        const int v = psum[q * E + tid];
        psum[q * E + tid] = count;
        count += v;
      }
    }
    int total;
    const int excl = block_exclusive_scan(count, ws, &total);
    if (tid < E) {
      off[tid] = excl;
      a.counts[tid] = count;
      a.offsets[tid] = excl;
    }
    if (tid == 0) a.offsets[E] = total;
    __syncthreads();
    if (mine) {
      int run = off[e] + psum[part * E + e];
#pragma unroll 8
      for (int b = b0; b < b1; ++b) {
        const int c = a.cntg[(size_t)b * E + e];
        a.cntg[(size_t)b * E + e] = run;
        run += c;
      }
    }
    build_worklists(a, count, excl, ws);
    pdl_launch_dependents();
    return;
  }

  if (do_route) {
    // the logits in shared memory when they fit (one coalesced pass), then
    // two tokens per warp
    const float* lg = a.logits;
    if (group_stages_logits(a.T, E)) {
      for (int i = tid; i < a.T * E; i += blockDim.x) lg_s[i] = a.logits[i];
      __syncthreads();
      lg = lg_s;
    }
    for (int t = 2 * warp; t < a.T; t += 64) route_warp<NPL, 2>(lg, t, a);
  } else {
    pdl_wait();
  }
  for (int i = tid; i < 32 * E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();

  if (R <= 32 * 32) {
    // ---- up to 32 chunks of 32 routes, a warp each, all at once ----
    const unsigned lt = (1u << lane) - 1u;
    const int r = warp * 32 + lane;
    const int e = r < R ? a.ids[r] : -1;
    const unsigned peers = peers_of(e, nb);
    const int rank = __popc(peers & lt);
    if (e >= 0 && rank == 0) cnt[warp * E + e] = __popc(peers);
    __syncthreads();
    int count = 0;
    if (tid < E) {
      const int nch = (R + 31) / 32;
      for (int w = 0; w < nch; ++w) {
        const int c = cnt[w * E + tid];
        cnt[w * E + tid] = count;
        count += c;
      }
    }
    int total;
    const int excl = block_exclusive_scan(count, ws, &total);
    if (tid < E) {
      off[tid] = excl;
      a.counts[tid] = count;
      a.offsets[tid] = excl;
    }
    if (tid == 0) a.offsets[E] = total;
    __syncthreads();
    if (e >= 0) {
      const int p = off[e] + cnt[warp * E + e] + rank;
      a.perm[p] = r;
      a.pos[r] = p;
    }
    build_worklists(a, count, excl, ws);
    pdl_launch_dependents();
    return;
  }

  // Pass 1: each warp counts its contiguous segment of routes per expert.
  // Loads are issued kU 32-route groups at a time so their latencies overlap.
  constexpr int kU = 8;
  const int seg = (((R + 31) / 32) + 31) & ~31;
  const int beg = warp * seg, end = min(R, beg + seg);
  for (int base = beg; base < end; base += 32 * kU) {
    int ev[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int r = base + 32 * u + lane;
      ev[u] = r < end ? a.ids[r] : -1;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = ev[u];
      const unsigned peers = peers_of(e, nb);
      if (e >= 0 && lane == __ffs(peers) - 1) cnt[warp * E + e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();

  // Column scan: cnt[w][e] <- routes of e in segments before w.
  int count = 0;
  if (tid < E) {
    for (int w = 0; w < 32; ++w) {
      const int c = cnt[w * E + tid];
      cnt[w * E + tid] = count;
      count += c;
    }
  }
  int total;
  const int excl = block_exclusive_scan(count, ws, &total);
  if (tid < E) {
    off[tid] = excl;
    a.counts[tid] = count;
    a.offsets[tid] = excl;
  }
  if (tid == 0) a.offsets[E] = total;
  __syncthreads();
  for (int i = tid; i < 32 * E; i += blockDim.x) cnt[i] += off[i % E];
  __syncthreads();

  // Pass 2: stable placement, walking each segment in route order.  The
  // permutation is scattered by expert: it is built in shared memory when it
  // fits (after cnt, off and ws) and written out in one coalesced pass.
  int* perm_s = group_perm_in_smem(R, E) ? ws + 32 : nullptr;
  const unsigned lt = (1u << lane) - 1u;
  for (int base = beg; base < end; base += 32 * kU) {
    int ev[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int r = base + 32 * u + lane;
      ev[u] = r < end ? a.ids[r] : -1;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int r = base + 32 * u + lane;
      const int e = ev[u];
      const unsigned peers = peers_of(e, nb);
      if (e >= 0) {
        const int p = cnt[warp * E + e] + __popc(peers & lt);
        if (perm_s) perm_s[p] = r;
        else a.perm[p] = r;
        a.pos[r] = p;
      }
      __syncwarp();
      if (e >= 0 && lane == __ffs(peers) - 1) cnt[warp * E + e] += __popc(peers);
      __syncwarp();
    }
  }

  if (perm_s) {
    __syncthreads();
    for (int i = tid; i < R; i += blockDim.x) a.perm[i] = perm_s[i];
  }
  build_worklists(a, count, excl, ws);
  pdl_launch_dependents();
}

size_t group_smem_bytes(int E, int T, int R, bool spread) {
  if (spread) return (size_t)((32 * E > 1024 ? 32 * E : 1024) + E + 32) * sizeof(int);
  size_t extra = 0;
  if (T > 0 && group_stages_logits(T, E)) extra = (size_t)T * E * sizeof(float);
  if (group_perm_in_smem(R, E) && (size_t)R * sizeof(int) > extra) extra = (size_t)R * sizeof(int);
  return (size_t)(33 * E + 32) * sizeof(int) + extra;
}

template <int NPL>
static cudaError_t launch_rg(const RouteArgs& a, bool fused, cudaStream_t s) {
  const bool spread = route_spread_grouping(a, fused);
  const size_t smem = group_smem_bytes(a.E, fused ? a.T : 0, a.T * a.k, spread);
  cudaError_t err =
      cudaFuncSetAttribute(group_kernel<NPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  if (fused) {
    group_kernel<NPL><<<1, 1024, smem, s>>>(a, 1);
    return cudaGetLastError();
  }
  const int tpb = route_tokens_per_cta(a, spread);
  route_kernel<NPL><<<(a.T + tpb - 1) / tpb, 256, spread ? 8 * a.E * sizeof(int) : 0, s>>>(a, spread ? 1 : 0);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1024);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, group_kernel<NPL>, a, 0);
  if (err != cudaSuccess || !spread) return err;
  cfg.gridDim = dim3((a.T * a.k + 255) / 256);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, scatter_kernel, a);
}

cudaError_t launch_route_group(const RouteArgs& a, bool fused, cudaStream_t s) {
  if (a.E <= 32) return launch_rg<1>(a, fused, s);
  if (a.E <= 64) return launch_rg<2>(a, fused, s);
  if (a.E <= 128) return launch_rg<4>(a, fused, s);
  if (a.E <= 256) return launch_rg<8>(a, fused, s);
  if (a.E <= 512) return launch_rg<16>(a, fused, s);
  return launch_rg<32>(a, fused, s);
}

// ----------------------------------------------------------------------------
// Combine: out[t, m] = R_D( sum_j w[t*k+j] * y[pos[t*k+j], m] ), j ascending
// (qmoe.rs qmoe_combine_impl; fp32 accumulate, round to nearest even).
// ----------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(256) finalize_kernel(const FinalizeArgs a) {
  pdl_wait();
  const int H4 = a.H / 4;
  const size_t n = (size_t)a.T * H4;
  const float4* y4 = reinterpret_cast<const float4*>(a.y);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / H4), m4 = (int)(i % H4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // slots in groups of 8: every load of a group is issued before its adds
    // (the adds stay in slot order)
    for (int j0 = 0; j0 < a.k; j0 += 8) {
      const int nj = min(8, a.k - j0);
      float wr[8];
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (u < nj) {
          const int r = t * a.k + j0 + u;
          wr[u] = a.w[r];
          v[u] = y4[(size_t)a.pos[r] * H4 + m4];
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (u < nj) {
          acc.x = fmaf(wr[u], v[u].x, acc.x);
          acc.y = fmaf(wr[u], v[u].y, acc.y);
          acc.z = fmaf(wr[u], v[u].z, acc.z);
          acc.w = fmaf(wr[u], v[u].w, acc.w);
        }
      }
    }
    const size_t o = (size_t)t * a.H + (size_t)m4 * 4;
    store_d<DT>(a.out, o + 0, acc.x);
    store_d<DT>(a.out, o + 1, acc.y);
    store_d<DT>(a.out, o + 2, acc.z);
    store_d<DT>(a.out, o + 3, acc.w);
  }
}

cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t s) {
  const size_t n = (size_t)a.T * (a.H / 4);
  int grid = (int)((n + 255) / 256);
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
  cfg.numAttrs = a.pdl ? 1 : 0;
  switch (a.dtype) {
    case QMOE_F32: return cudaLaunchKernelEx(&cfg, finalize_kernel<QMOE_F32>, a);
    case QMOE_F16: return cudaLaunchKernelEx(&cfg, finalize_kernel<QMOE_F16>, a);
    default: return cudaLaunchKernelEx(&cfg, finalize_kernel<QMOE_BF16>, a);
  }
}

}  // namespace qmoe
