// C ABI of the QMoE layer (include/qmoe.h): validation, device memory
// ownership, prepack and the forward's launch sequence on one stream.
//
// Launch sequence of qmoe_forward (all on the caller's stream, no host sync,
// no allocation once reserved -> capturable into a CUDA graph):
//   route + group + work-lists    (1 CTA for small T; route grid + 1 CTA else)
//   fc1 (+ fused GLU)             decode mma kernel   | SIMT kernel for f32
//   fc2                           decode mma kernel   | SIMT kernel for f32
//   combine                       slot-ordered weighted sum, round into D
// Consecutive kernels use programmatic dependent launch.
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <string>

#include "qmoe_internal.cuh"
#include "qmoe_prefill.cuh"
#include "qmoe_fused.cuh"

using namespace qmoe;

namespace {

struct Proj {
  uint8_t* codes = nullptr;
  void* scales = nullptr;
  uint8_t* zp = nullptr;
  uint8_t* dec = nullptr;
  uint8_t* gq = nullptr;
  size_t codes_bytes = 0, scales_bytes = 0, zp_bytes = 0, dec_bytes = 0, gq_bytes = 0;
  int N = 0, K = 0, bits = 0, zp_row = 0;
  DecodeLayout L{};
  GemmLayout GL{};
  bool ready = false;
};

const char* kStatusNames[] = {"QMOE_OK",          "QMOE_ERR_INVALID_ARG", "QMOE_ERR_UNSUPPORTED",
                              "QMOE_ERR_CUDA",    "QMOE_ERR_OOM",         "QMOE_ERR_STATE",
                              "QMOE_ERR_TIMEOUT"};

// Polls of a bounded device-side wait (each poll parks the warp for up to
// ~1 us): about two seconds before a wait gives up.
constexpr long long kDefaultWaitLimit = 1LL << 21;

}  // namespace

struct qmoe_layer {
  int H, I, E, k, B, zp_mode, act, dtype, dsize;
  int bits[2];
  // SwiGLU attributes (qmoe.rs swiglu_value defaults: alpha 1, beta 0, no limit)
  float sw_alpha = 1.f, sw_beta = 0.f, sw_limit = INFINITY;
  int fc1_interleaved = 0;                 // fc1 canonical rows: [gate | up] or (gate, up) pairs
  int fc1_separate = 0;                    // gate rows from fc1, up rows from a separate fc3
  int act_created = 0;                     // the activation given to qmoe_create (act may differ: silu + fc3)
  bool fc1_half[2] = {false, false};       // separate: gate / up halves copied in
  float* bias[2] = {nullptr, nullptr};     // fc1: [E, I, 2] (gate, up) pairs ; fc2: [E, H]
  int normalize = 1;
  float zp_offset = NAN;
  bool offset_set = false;
  int gemm_min_rows = 0;
  int fused = 2;                           // single launch: 0 off, 1 whenever it applies, 2 auto
  int deterministic = QMOE_COMBINE_AUTO;   // tensor-core path: slot-ordered combine or fp32 reductions
  int last_path = QMOE_PATH_NONE;
  int device = -1;
  long long wait_limit = kDefaultWaitLimit;
  int inject_stall = 0;
  Proj proj[2];

  // workspace for up to cap_T tokens
  int64_t cap_T = 0;
  int* ids = nullptr;
  float* w = nullptr;
  int* counts = nullptr;
  int* offsets = nullptr;
  int* perm = nullptr;
  int* pos = nullptr;
  int* cntg = nullptr;         // spread grouping: route count / first position per (routing CTA, expert)
  int* rnk = nullptr;          // spread grouping: rank of each route within its routing CTA and expert
  int* gready = nullptr;       // fc1's overlapped gather: finished units per class-1 item
  int* n_items = nullptr;
  Item* items[2] = {nullptr, nullptr};
  int cap_items[2] = {0, 0};
  void* hbuf = nullptr;
  float* ybuf = nullptr;
  int* status = nullptr;
  void* x_stage = nullptr;
  float* logits_stage = nullptr;
  void* out_stage = nullptr;
  uint8_t* xt = nullptr;       // x of GEMM-class items, tiled token layout (fc1 B operand)
  uint8_t* ht = nullptr;       // h of GEMM-class items, tiled token layout (fc2 B operand)
  float* out_acc = nullptr;    // fp32 [T, H] combine accumulator (mixed forwards)
  int* sync = nullptr;         // counters of the single-launch decode forward (zero before the first launch)
  size_t sync_n = 0;           // ints in sync
  bool tiles_ok = false;
  int num_sms = 0;

  int64_t last_T = 0;
  int last_tb[2] = {0, 0};
  cudaEvent_t trace[QMOE_TRACE_NUM_EVENTS] = {};
  bool trace_on = false;
  std::string err;
};

namespace {

// Status word of qmoe_forward_noalloc's static array in the current context
// (nullptr if that entry point has not run there); defined with the array.
cudaError_t noalloc_status_word(void** out);

qmoe_status fail(qmoe_layer* l, qmoe_status st, const std::string& msg) {
  if (l) l->err = msg;
  return st;
}

qmoe_status cuda_fail(qmoe_layer* l, cudaError_t e, const char* what) {
  cudaGetLastError();  // clear a sticky launch error if any
  const qmoe_status st = e == cudaErrorMemoryAllocation ? QMOE_ERR_OOM : QMOE_ERR_CUDA;
  return fail(l, st, std::string(what) + ": " + cudaGetErrorString(e));
}

#define QMOE_CUDA(layer, call, what)                 \
  do {                                               \
    cudaError_t e_ = (call);                         \
    if (e_ != cudaSuccess) return cuda_fail(layer, e_, what); \
  } while (0)

bool exact_in(double v, int dtype) {
  // Is v exactly representable (finite, normal or zero) in dtype?
  if (v == 0.0) return true;
  if (!std::isfinite(v)) return false;
  const int p = dtype == QMOE_F32 ? 24 : dtype == QMOE_F16 ? 11 : 8;
  const int emin = dtype == QMOE_F16 ? -14 : -126;
  const int emax = dtype == QMOE_F16 ? 15 : 127;
  int e;
  const double m = std::frexp(v, &e);  // v = m * 2^e, 0.5 <= |m| < 1
  if (e - 1 < emin || e - 1 > emax) return false;
  const double scaled = std::ldexp(m, p);
  return scaled == std::floor(scaled);
}

template <typename T>
cudaError_t dalloc(T** p, size_t bytes) {
  *p = nullptr;
  if (bytes == 0) bytes = 16;
  return cudaMalloc(reinterpret_cast<void**>(p), bytes);
}

ActParams act_params(const qmoe_layer* l) {
  ActParams p;
  p.act = l->act;
  p.alpha = l->sw_alpha;
  p.beta = l->sw_beta;
  p.limit = l->sw_limit;
  return p;
}

// fc1 bias [E, 2I] in the canonical row order -> (gate, up) pairs [E, I, 2].
__global__ void pair_bias_kernel(const float* __restrict__ src, float* __restrict__ dst, int E, int I,
                                 int interleaved) {
  const size_t n = (size_t)E * I;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t e = i / I, f = i % I;
    const float* row = src + e * 2 * I;
    dst[2 * i] = interleaved ? row[2 * f] : row[f];
    dst[2 * i + 1] = interleaved ? row[2 * f + 1] : row[I + f];
  }
}

cudaError_t launch_pair_bias(const float* src, float* dst, int E, int I, int interleaved, cudaStream_t s) {
  const size_t n = (size_t)E * I;
  const int grid = (int)std::min<size_t>((n + 255) / 256, 4096);
  pair_bias_kernel<<<grid, 256, 0, s>>>(src, dst, E, I, interleaved);
  return cudaGetLastError();
}

// Separate fc1 / fc3 bias [E, I] -> one half of the (gate, up) pairs; NULL
// source zeroes the half.
__global__ void half_bias_kernel(const float* __restrict__ src, float* __restrict__ dst, size_t n, int half) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[2 * i + half] = src ? src[i] : 0.f;
}

cudaError_t launch_half_bias(const float* src, float* dst, size_t n, int half, cudaStream_t s) {
  const int grid = (int)std::min<size_t>((n + 255) / 256, 4096);
  half_bias_kernel<<<grid, 256, 0, s>>>(src, dst, n, half);
  return cudaGetLastError();
}

void free_workspace(qmoe_layer* l) {
  void* bufs[] = {l->ids, l->w, l->counts, l->offsets, l->perm, l->pos, l->n_items, l->items[0],
                  l->items[1], l->hbuf, l->ybuf, l->status, l->x_stage, l->logits_stage,
                  l->out_stage, l->xt, l->ht, l->out_acc, l->sync, l->cntg, l->rnk, l->gready};
  for (void* b : bufs)
    if (b) cudaFree(b);
  l->ids = nullptr;
  l->w = nullptr;
  l->counts = l->offsets = l->perm = l->pos = l->n_items = nullptr;
  l->items[0] = l->items[1] = nullptr;
  l->hbuf = nullptr;
  l->ybuf = nullptr;
  l->status = nullptr;
  l->x_stage = nullptr;
  l->logits_stage = nullptr;
  l->out_stage = nullptr;
  l->xt = nullptr;
  l->ht = nullptr;
  l->out_acc = nullptr;
  l->sync = nullptr;
  l->cntg = l->rnk = l->gready = nullptr;
  l->tiles_ok = false;
  l->cap_T = 0;
}

// Rows per work item of each class for a forward of T tokens.
void item_heights(const qmoe_layer* l, int64_t T, int* tb0, int* tb1) {
  if (l->dtype == QMOE_F32) {
    *tb0 = 4;  // SIMT kernel
  } else {
    const int64_t R = T * l->k;
    const int64_t active = R < l->E ? R : l->E;
    const double per = active > 0 ? (double)R / (double)active : 1.0;
    int ng = per <= 8.0 ? 1 : per <= 12.0 ? 2 : 4;
    // The staged rows (ng * 8 tokens x K, 16-bit) must fit in shared memory
    // next to the weight ring: cap ng by the longer K of the two projections.
    const int kmax = l->H > l->I ? l->H : l->I;
    const int ktiles = (kmax + 127) / 128 * 8;
    while (ng > 1 && ng * ktiles * 256 > 160 * 1024) ng /= 2;
    *tb0 = 8 * ng;
  }
  *tb1 = 128;
}

int64_t items_cap(const qmoe_layer* l, int which, int64_t T, int tb) {
  const int64_t R = T * l->k;
  const int64_t active = R < l->E ? R : l->E;
  return active + R / (tb > 0 ? tb : 1) + 1;
}

qmoe_status ensure_workspace(qmoe_layer* l, int64_t T) {
  if (T <= l->cap_T) return QMOE_OK;
  free_workspace(l);
  const int64_t R = T * l->k;
  const size_t ds = (size_t)l->dsize;
  QMOE_CUDA(l, dalloc(&l->ids, R * sizeof(int)), "allocate workspace");
  QMOE_CUDA(l, dalloc(&l->w, R * sizeof(float)), "allocate workspace");
  QMOE_CUDA(l, dalloc(&l->counts, l->E * sizeof(int)), "allocate workspace");
  QMOE_CUDA(l, dalloc(&l->offsets, (l->E + 1) * sizeof(int)), "allocate workspace");
  QMOE_CUDA(l, dalloc(&l->perm, R * sizeof(int)), "allocate workspace");
  QMOE_CUDA(l, dalloc(&l->pos, R * sizeof(int)), "allocate workspace");
  // spread grouping: per routing CTA (8 tokens) and expert, per route
  QMOE_CUDA(l, dalloc(&l->cntg, (size_t)((T + 7) / 8) * l->E * sizeof(int)), "allocate workspace");
  QMOE_CUDA(l, dalloc(&l->rnk, R * sizeof(int)), "allocate workspace");
  QMOE_CUDA(l, dalloc(&l->n_items, 2 * sizeof(int)), "allocate workspace");
  for (int c = 0; c < 2; ++c) {
    const int64_t cap = items_cap(l, c, T, 4);
    if (cap > INT_MAX / 2) return fail(l, QMOE_ERR_INVALID_ARG, "token count too large");
    l->cap_items[c] = (int)cap;
    QMOE_CUDA(l, dalloc(&l->items[c], cap * sizeof(Item)), "allocate workspace");
  }
  QMOE_CUDA(l, dalloc(&l->gready, (size_t)l->cap_items[1] * sizeof(int)), "allocate workspace");
  QMOE_CUDA(l, dalloc(&l->hbuf, (size_t)R * l->I * ds), "allocate workspace");
  QMOE_CUDA(l, dalloc(&l->ybuf, (size_t)R * l->H * sizeof(float)), "allocate workspace");
  QMOE_CUDA(l, dalloc(&l->status, sizeof(int)), "allocate workspace");
  QMOE_CUDA(l, cudaMemset(l->status, 0, sizeof(int)), "clear status");
  QMOE_CUDA(l, dalloc(&l->x_stage, (size_t)T * l->H * ds), "allocate workspace");
  QMOE_CUDA(l, dalloc(&l->logits_stage, (size_t)T * l->E * sizeof(float)), "allocate workspace");
  QMOE_CUDA(l, dalloc(&l->out_stage, (size_t)T * l->H * ds), "allocate workspace");
  if (l->dtype != QMOE_F32) {
    // GEMM-class items hold at most 128 rows each: one 128-row block per item.
    const size_t blocks = (size_t)items_cap(l, 1, T, 128);
    QMOE_CUDA(l, dalloc(&l->xt, blocks * (size_t)((l->H + 63) / 64) * kTokTileBytes), "allocate workspace");
    QMOE_CUDA(l, dalloc(&l->ht, blocks * (size_t)((l->I + 63) / 64) * kTokTileBytes), "allocate workspace");
    QMOE_CUDA(l, dalloc(&l->out_acc, (size_t)T * l->H * sizeof(float)), "allocate workspace");
    QMOE_CUDA(l, cudaMemset(l->out_acc, 0, (size_t)T * l->H * sizeof(float)), "clear accumulator");
    l->tiles_ok = true;
  }
  {
    // counters of the single launch: header, one per segment (group of <= 16
    // routed rows of an expert; at most min(R, E) + R / 16 + 1)
    const size_t segs = (size_t)(R < l->E ? R : l->E) + R / kFusedRowsPerGroup + 1;
    const size_t n = (size_t)kSyncHeader + segs;
    QMOE_CUDA(l, dalloc(&l->sync, n * sizeof(int)), "allocate workspace");
    l->sync_n = n;
    QMOE_CUDA(l, cudaMemset(l->sync, 0, n * sizeof(int)), "clear counters");
  }
  if (l->num_sms == 0) {
    int dev = 0;
    QMOE_CUDA(l, cudaGetDevice(&dev), "cudaGetDevice");
    QMOE_CUDA(l, cudaDeviceGetAttribute(&l->num_sms, cudaDevAttrMultiProcessorCount, dev), "query SMs");
  }
  l->cap_T = T;
  return QMOE_OK;
}

bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) != cudaSuccess) return false;
  return st != cudaStreamCaptureStatusNone;
}

void trace(qmoe_layer* l, int i, cudaStream_t s) {
  // Under stream capture the record becomes an event-record node of the graph.
  if (l->trace_on && l->trace[i])
    cudaEventRecordWithFlags(l->trace[i], s, capturing(s) ? cudaEventRecordExternal : cudaEventRecordDefault);
}

// ----------------------------------------------------------------------------
// Single-launch decode forward (qmoe_fused.cu): small token counts, 16-bit
// activations, code widths {2, 3, 4}.
// ----------------------------------------------------------------------------
// Shared memory of a CTA: two 8-warp CTAs per SM when the plan fits (each
// CTA's barriers are then covered by the other's work), else one 16-warp CTA.
constexpr int kFusedSmemTwoPerSm = 113 * 1024;
constexpr int kFusedSmemOnePerSm = 227 * 1024;
// Weights up to this size are prefetched into the L2 during routing.
constexpr size_t kFusedPrefetchMaxBytes = 64ull << 20;
// Smallest ring stage worth two CTAs per SM (16 warps x 3 stages in flight).
constexpr int kFusedMinStageTwoPerSm = 1024;

struct FusedShape {
  int smem, sb, g1, g2, ng_max, warps, ctas_per_sm;
};

// Segments (groups of <= 16 routed rows of one expert) a forward of T tokens
// can have at most.
int fused_max_segments(const qmoe_layer* l, int64_t T) {
  const int64_t R = T * l->k;
  return (int)((R < l->E ? R : l->E) + R / kFusedRowsPerGroup + 1);
}

// Tokens up to which the automatic combine choice adds the slots in order.
constexpr int64_t kCombineAutoMaxTokens = 64;

// Routes up to which the automatic choice takes the single launch (measured:
// it wins at 8 tokens x top-2, the separate kernels at 256 routes).
constexpr int64_t kFusedAutoMaxRoutes = 64;

bool fused_applies(const qmoe_layer* l, int64_t T, FusedShape* fs) {
  if (!l->fused || l->dtype == QMOE_F32 || !l->sync) return false;
  if (l->fused == 2 && T * l->k > kFusedAutoMaxRoutes) return false;
  if (T > kFusedMaxTokens || l->E > kFusedMaxExperts || l->k > kFusedMaxK) return false;
  if (T * l->k > kFusedMaxRoutes || l->E % 4) return false;
  if (!fused_widths_supported(l->bits[0], l->bits[1])) return false;
  const int sc = l->proj[0].L.SC;
  const int nkc = l->proj[0].L.nkc > l->proj[1].L.nkc ? l->proj[0].L.nkc : l->proj[1].L.nkc;
  const int R = (int)(T * l->k);
  // an expert's group of rows holds at most min(16, T) tokens
  fs->ng_max = T > 8 ? 2 : 1;
  const int scb1 = l->proj[0].L.scb, scb2 = l->proj[1].L.scb;
  // one 16-warp CTA per SM (measured faster than two 8-warp CTAs: the B
  // staging is not held twice, so the rings are deeper)
  for (int warps : {16}) {
    const int budget = warps == 8 ? kFusedSmemTwoPerSm : kFusedSmemOnePerSm;
    const int fixed = fused_plan(R, l->E, nkc * sc, fs->ng_max, 0, warps).total;
    if (fixed >= budget) continue;
    if (!fused_ring_shape(budget, fixed, warps, scb1, scb2, &fs->sb, &fs->g1, &fs->g2)) continue;
    if (warps == 8 && fs->sb < kFusedMinStageTwoPerSm) continue;
    fs->smem = fused_plan(R, l->E, nkc * sc, fs->ng_max, fs->sb, warps).total;
    if (fs->smem > budget) continue;
    // the routing and grouping scratch sits in the ring area before the rings start
    if (R > 32 * warps || fused_prologue((int)T, l->E, R).total > warps * kFusedStages * fs->sb) continue;
    fs->warps = warps;
    fs->ctas_per_sm = warps == 8 ? 2 : 1;
    return true;
  }
  return false;
}

qmoe_status forward_fused(qmoe_layer* l, const void* x, const float* logits, void* out, int64_t T,
                          const FusedShape& fs, cudaStream_t s) {
  FusedArgs a{};
  a.logits = logits;
  a.x = x;
  a.out = out;
  a.T = (int)T;
  a.E = l->E;
  a.k = l->k;
  a.normalize = l->normalize;
  a.H = l->H;
  a.I = l->I;
  a.gated = act_gated(l->act) ? 1 : 0;
  for (int f = 0; f < 2; ++f) {
    const Proj& p = l->proj[f];
    FusedProj& q = a.p[f];
    q.wpk = p.dec;
    q.L = p.L;
    q.K = p.K;
    q.ntiles = p.L.ntiles;
    q.g = f == 0 ? fs.g1 : fs.g2;
    q.bias = l->bias[f];
  }
  a.act = act_params(l);
  a.zp_mode = l->zp_mode;
  a.zp_offset = l->zp_offset;
  a.ids = l->ids;
  a.w = l->w;
  a.counts = l->counts;
  a.offsets = l->offsets;
  a.perm = l->perm;
  a.items0 = l->items[0];
  a.n_items = l->n_items;
  a.hbuf = l->hbuf;
  a.ybuf = l->ybuf;
  a.sync = l->sync;
  a.max_seg = fused_max_segments(l, l->cap_T);
  a.ng_max = fs.ng_max;
  a.sb = fs.sb;
  a.wait = WaitCfg{l->status, l->wait_limit};
  a.inject_stall = l->inject_stall;
  // weights that fit the L2 (129 MB) with room to spare are prefetched while
  // the CTAs route (decode layouts are multiples of 16 bytes per expert)
  a.prefetch_l2 = (size_t)l->E * (l->proj[0].L.expert_bytes + l->proj[1].L.expert_bytes) <= kFusedPrefetchMaxBytes;
  l->last_T = T;
  l->last_path = QMOE_PATH_FUSED;
  l->last_tb[0] = kFusedRowsPerGroup;
  l->last_tb[1] = 128;
  trace(l, QMOE_TRACE_BEGIN, s);
  QMOE_CUDA(l, launch_fused(a, l->bits[0], l->bits[1], l->dtype == QMOE_BF16, l->proj[0].L.SC,
                            l->num_sms * fs.ctas_per_sm, fs.warps, fs.smem, s),
            "launch the single-launch decode forward");
  for (int i = QMOE_TRACE_ROUTED; i <= QMOE_TRACE_END; ++i) trace(l, i, s);
  return QMOE_OK;
}

}  // namespace

extern "C" {

qmoe_status qmoe_create(int hidden, int inter, int experts, int top_k, int bits_fc1, int bits_fc2,
                        int block_size, int zp_mode, int activation, int dtype, qmoe_layer** out) {
  if (!out) return QMOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (hidden <= 0 || inter <= 0 || experts <= 0 || top_k <= 0) return QMOE_ERR_INVALID_ARG;
  if (experts > 1024) return QMOE_ERR_UNSUPPORTED;
  if (top_k > experts) return QMOE_ERR_INVALID_ARG;
  for (int b : {bits_fc1, bits_fc2})
    if (b != 1 && b != 2 && b != 3 && b != 4 && b != 8) return QMOE_ERR_UNSUPPORTED;
  if (block_size != 32 && block_size != 64 && block_size != 128) return QMOE_ERR_UNSUPPORTED;
  if (hidden % block_size || inter % block_size) return QMOE_ERR_INVALID_ARG;
  if (zp_mode < QMOE_ZP_SYMMETRIC || zp_mode > QMOE_ZP_OFFSET) return QMOE_ERR_INVALID_ARG;
  if (activation < QMOE_ACT_SWIGLU || activation > QMOE_ACT_IDENTITY) return QMOE_ERR_INVALID_ARG;
  if (dtype < QMOE_F32 || dtype > QMOE_BF16) return QMOE_ERR_INVALID_ARG;
  if ((long long)hidden * inter > (1LL << 31)) return QMOE_ERR_UNSUPPORTED;
  qmoe_layer* l = new qmoe_layer();
  l->H = hidden;
  l->I = inter;
  l->E = experts;
  l->k = top_k;
  l->bits[0] = bits_fc1;
  l->bits[1] = bits_fc2;
  l->B = block_size;
  l->zp_mode = zp_mode;
  l->act = activation;
  l->act_created = activation;
  l->dtype = dtype;
  l->dsize = dtype == QMOE_F32 ? 4 : 2;
  *out = l;
  return QMOE_OK;
}

qmoe_status qmoe_set_routing(qmoe_layer* l, int normalize) {
  if (!l) return QMOE_ERR_INVALID_ARG;
  l->normalize = normalize ? 1 : 0;
  return QMOE_OK;
}

qmoe_status qmoe_set_zero_point_offset(qmoe_layer* l, float offset) {
  if (!l) return QMOE_ERR_INVALID_ARG;
  if (l->zp_mode != QMOE_ZP_OFFSET)
    return fail(l, QMOE_ERR_STATE, "zero_point_offset needs zp_mode == QMOE_ZP_OFFSET");
  if (!std::isfinite(offset)) return fail(l, QMOE_ERR_INVALID_ARG, "zero_point_offset must be finite");
  // Supported centres: multiples of 1/2 inside the code range.  Then every
  // (code - offset) is exact in D and the kernels form it with one packed
  // subtraction from a half-unit magic number.
  const int maxcode = (1 << (l->bits[0] < l->bits[1] ? l->bits[0] : l->bits[1])) - 1;
  if (std::floor(2.0 * offset) != 2.0 * offset || offset < 0.0f || offset > (float)maxcode)
    return fail(l, QMOE_ERR_UNSUPPORTED,
                "zero_point_offset must be a multiple of 0.5 within the code range; "
                "requantize with a half-integer centre");
  for (int f = 0; f < 2; ++f)
    for (int c = 0; c < (1 << l->bits[f]); ++c)
      if (!exact_in((double)c - (double)offset, l->dtype) || !exact_in((double)offset, l->dtype))
        return fail(l, QMOE_ERR_UNSUPPORTED,
                    "zero_point_offset: (code - offset) is not exact in the activation type; "
                    "requantize with a coarser fractional centre");
  l->zp_offset = offset;
  l->offset_set = true;
  return QMOE_OK;
}

qmoe_status qmoe_set_swiglu_params(qmoe_layer* l, float alpha, float beta, float limit) {
  if (!l) return QMOE_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || alpha == 0.f || !std::isfinite(beta) || std::isnan(limit) || !(limit > 0.f))
    return fail(l, QMOE_ERR_INVALID_ARG, "swiglu: alpha finite and nonzero, beta finite, limit > 0 (or +inf)");
  l->sw_alpha = alpha;
  l->sw_beta = beta;
  l->sw_limit = limit;
  return QMOE_OK;
}

qmoe_status qmoe_set_fc1_layout(qmoe_layer* l, int layout) {
  if (!l || layout < QMOE_FC1_CONCAT || layout > QMOE_FC1_SEPARATE_FC3) return QMOE_ERR_INVALID_ARG;
  // silu beside a separate fc3 is the gated form [qmoe.rs uses_separate_gate,
  // qmoe_activate: gate = fc1, linear = fc3, through swiglu_value]
  const bool silu_fc3 = l->act_created == QMOE_ACT_SILU && layout == QMOE_FC1_SEPARATE_FC3;
  if (layout != QMOE_FC1_CONCAT && !act_gated(l->act_created) && !silu_fc3)
    return fail(l, QMOE_ERR_INVALID_ARG, "fc1 row layouts apply to gated activations only");
  if (l->proj[0].ready || l->bias[0] || l->fc1_half[0] || l->fc1_half[1])
    return fail(l, QMOE_ERR_STATE,
                "set the fc1 layout before qmoe_prepack(fc=1/3) and qmoe_set_bias(fc=1/3)");
  // Separate projections are assembled into the concatenated order.
  l->fc1_interleaved = layout == QMOE_FC1_INTERLEAVED ? 1 : 0;
  l->fc1_separate = layout == QMOE_FC1_SEPARATE_FC3 ? 1 : 0;
  l->act = silu_fc3 ? QMOE_ACT_SWIGLU : l->act_created;
  return QMOE_OK;
}

qmoe_status qmoe_set_bias(qmoe_layer* l, int fc, const float* bias, void* stream) {
  if (!l) return QMOE_ERR_INVALID_ARG;
  if (fc != 1 && fc != 2 && fc != 3) return fail(l, QMOE_ERR_INVALID_ARG, "fc must be 1, 2 or 3");
  if (fc == 3 && !l->fc1_separate)
    return fail(l, QMOE_ERR_STATE, "fc=3 needs qmoe_set_fc1_layout(QMOE_FC1_SEPARATE_FC3)");
  if (l->fc1_separate && fc != 2) {
    // one half of the (gate, up) pairs: fc1 = gate, fc3 = up
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float*& dst = l->bias[0];
    const size_t n = (size_t)l->E * l->I;
    if (!dst) {
      if (!bias) return QMOE_OK;
      QMOE_CUDA(l, dalloc(&dst, 2 * n * sizeof(float)), "allocate bias");
      QMOE_CUDA(l, cudaMemsetAsync(dst, 0, 2 * n * sizeof(float), s), "clear bias");
    }
    QMOE_CUDA(l, launch_half_bias(bias, dst, n, fc == 1 ? 0 : 1, s), "re-lay fc1/fc3 bias");
    return QMOE_OK;
  }
  float*& dst = l->bias[fc - 1];
  if (!bias) {
    if (dst) {
      QMOE_CUDA(l, cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "synchronise");
      cudaFree(dst);
    }
    dst = nullptr;
    return QMOE_OK;
  }
  const bool gated = act_gated(l->act);
  const size_t n = (size_t)l->E * (fc == 1 ? (gated ? 2 * l->I : l->I) : l->H);
  if (!dst) QMOE_CUDA(l, dalloc(&dst, n * sizeof(float)), "allocate bias");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (fc == 2 || !gated)   // fc2, or a non-gated fc1: rows as given
    QMOE_CUDA(l, cudaMemcpyAsync(dst, bias, n * sizeof(float), cudaMemcpyDeviceToDevice, s), "copy bias");
  else
    QMOE_CUDA(l, launch_pair_bias(bias, dst, l->E, l->I, l->fc1_interleaved, s), "re-lay fc1 bias");
  return QMOE_OK;
}

qmoe_status qmoe_set_gemm_min_rows(qmoe_layer* l, int min_rows) {
  if (!l || min_rows < 0) return QMOE_ERR_INVALID_ARG;
  l->gemm_min_rows = min_rows;
  return QMOE_OK;
}

qmoe_status qmoe_set_fused_decode(qmoe_layer* l, int mode) {
  if (!l || mode < 0 || mode > 2) return QMOE_ERR_INVALID_ARG;
  l->fused = mode;
  return QMOE_OK;
}

int qmoe_last_forward_path(const qmoe_layer* l) { return l ? l->last_path : QMOE_PATH_NONE; }

qmoe_status qmoe_set_deterministic(qmoe_layer* l, int mode) {
  if (!l) return QMOE_ERR_INVALID_ARG;
  if (mode != QMOE_COMBINE_REDUCE && mode != QMOE_COMBINE_ORDERED && mode != QMOE_COMBINE_AUTO)
    return fail(l, QMOE_ERR_INVALID_ARG, "combine mode must be 0, 1 or 2");
  l->deterministic = mode;
  return QMOE_OK;
}

qmoe_status qmoe_set_wait_limit(qmoe_layer* l, int64_t iterations) {
  if (!l || iterations < 0) return QMOE_ERR_INVALID_ARG;
  l->wait_limit = iterations == 0 ? kDefaultWaitLimit : iterations;
  return QMOE_OK;
}

qmoe_status qmoe_debug_inject_stall(qmoe_layer* l, int enable) {
  if (!l) return QMOE_ERR_INVALID_ARG;
  l->inject_stall = enable ? 1 : 0;
  return QMOE_OK;
}

qmoe_status qmoe_reserve(qmoe_layer* l, int64_t max_tokens) {
  if (!l || max_tokens < 0) return QMOE_ERR_INVALID_ARG;
  if ((max_tokens * l->k) > INT_MAX / 8) return fail(l, QMOE_ERR_INVALID_ARG, "max_tokens too large");
  if (max_tokens == 0) return QMOE_OK;
  return ensure_workspace(l, max_tokens);
}

qmoe_status qmoe_prepack(qmoe_layer* l, int fc, const uint8_t* codes, const void* scales,
                         const uint8_t* zero_points, void* stream) {
  if (!l) return QMOE_ERR_INVALID_ARG;
  if (fc != 1 && fc != 2 && fc != 3) return fail(l, QMOE_ERR_INVALID_ARG, "fc must be 1, 2 or 3");
  if (fc == 3 && !l->fc1_separate)
    return fail(l, QMOE_ERR_STATE, "fc=3 needs qmoe_set_fc1_layout(QMOE_FC1_SEPARATE_FC3)");
  // With separate projections, fc1 (gate) and fc3 (up) each fill half of
  // fc1's rows, assembled here in the concatenated order.
  const int half = l->fc1_separate && fc != 2 ? (fc == 1 ? 0 : 1) : -1;
  if (fc == 3) fc = 1;
  if (!codes || !scales) return fail(l, QMOE_ERR_INVALID_ARG, "codes and scales are required");
  if ((zero_points != nullptr) != (l->zp_mode == QMOE_ZP_UINT8))
    return fail(l, QMOE_ERR_INVALID_ARG, "zero_points must be given iff zp_mode == QMOE_ZP_UINT8");
  if (l->zp_mode == QMOE_ZP_OFFSET && !l->offset_set)
    return fail(l, QMOE_ERR_STATE, "call qmoe_set_zero_point_offset before qmoe_prepack");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Proj& p = l->proj[fc - 1];
  const bool gated = act_gated(l->act);
  // fc1 rows: gate and up (gated activations) or one row per feature; the
  // GEMM and decode layouts treat a non-gated fc1 like fc2 (plain rows)
  const bool pairs = fc == 1 && gated;
  p.bits = l->bits[fc - 1];
  p.N = fc == 1 ? (gated ? 2 * l->I : l->I) : l->H;
  p.K = fc == 1 ? l->H : l->I;
  const size_t E = (size_t)l->E;
  const size_t codes_bytes = E * p.N * ((size_t)p.K * p.bits / 8);
  const size_t scales_bytes = E * p.N * (size_t)(p.K / l->B) * l->dsize;
  p.zp_row = (p.K / l->B * p.bits + 7) / 8;
  const size_t zp_bytes = zero_points ? E * p.N * (size_t)p.zp_row : 0;
  int dev = -1;
  QMOE_CUDA(l, cudaGetDevice(&dev), "cudaGetDevice");
  if (l->device >= 0 && l->device != dev)
    return fail(l, QMOE_ERR_STATE, "prepack on a different device than the layer's");
  l->device = dev;
  if (p.codes_bytes != codes_bytes) {
    if (p.codes) cudaFree(p.codes);
    QMOE_CUDA(l, dalloc(&p.codes, codes_bytes), "allocate codes");
    p.codes_bytes = codes_bytes;
  }
  if (p.scales_bytes != scales_bytes) {
    if (p.scales) cudaFree(p.scales);
    QMOE_CUDA(l, dalloc(&p.scales, scales_bytes), "allocate scales");
    p.scales_bytes = scales_bytes;
  }
  if (p.zp_bytes != zp_bytes) {
    if (p.zp) cudaFree(p.zp);
    p.zp = nullptr;
    if (zp_bytes) QMOE_CUDA(l, dalloc(&p.zp, zp_bytes), "allocate zero points");
    p.zp_bytes = zp_bytes;
  }
  if (half < 0) {
    QMOE_CUDA(l, cudaMemcpyAsync(p.codes, codes, codes_bytes, cudaMemcpyDeviceToDevice, s), "copy codes");
    QMOE_CUDA(l, cudaMemcpyAsync(p.scales, scales, scales_bytes, cudaMemcpyDeviceToDevice, s), "copy scales");
    if (zp_bytes)
      QMOE_CUDA(l, cudaMemcpyAsync(p.zp, zero_points, zp_bytes, cudaMemcpyDeviceToDevice, s), "copy zp");
  } else {
    // per expert: the caller's I rows -> rows [half*I, half*I + I) of the 2I
    auto copy_half = [&](void* dst, const void* src, size_t total_bytes) {
      const size_t blk = total_bytes / (2 * E);   // bytes of I rows
      return cudaMemcpy2DAsync(static_cast<uint8_t*>(dst) + half * blk, 2 * blk, src, blk, blk, E,
                               cudaMemcpyDeviceToDevice, s);
    };
    QMOE_CUDA(l, copy_half(p.codes, codes, codes_bytes), "copy codes");
    QMOE_CUDA(l, copy_half(p.scales, scales, scales_bytes), "copy scales");
    if (zp_bytes) QMOE_CUDA(l, copy_half(p.zp, zero_points, zp_bytes), "copy zp");
    l->fc1_half[half] = true;
    if (!(l->fc1_half[0] && l->fc1_half[1])) {
      p.ready = false;   // the layouts are built once both halves are in
      return QMOE_OK;
    }
  }
  if (l->dtype != QMOE_F32) {
    p.L = make_decode_layout(p.bits, l->B, fc == 1 ? l->I : l->H, p.K, pairs ? 2 : 1, l->zp_mode,
                             l->dsize);
    const size_t dec_bytes = p.L.expert_bytes * E;
    if (p.dec_bytes != dec_bytes) {
      if (p.dec) cudaFree(p.dec);
      QMOE_CUDA(l, dalloc(&p.dec, dec_bytes), "allocate decode layout");
      p.dec_bytes = dec_bytes;
    }
    RepackArgs ra{};
    ra.codes = p.codes;
    ra.scales = p.scales;
    ra.zp = p.zp;
    ra.out = p.dec;
    ra.E = l->E;
    ra.N = p.N;
    ra.K = p.K;
    ra.I_or_0 = pairs ? l->I : 0;
    ra.interleaved = l->fc1_interleaved;
    ra.dsize = l->dsize;
    ra.L = p.L;
    QMOE_CUDA(l, launch_repack_decode(ra, s), "repack weights");
    p.GL = make_gemm_layout(p.bits, l->B, pairs ? 1 : 2, p.N, p.K, l->I, l->zp_mode);
    const size_t gq_bytes = p.GL.expert_bytes * E;
    if (p.gq_bytes != gq_bytes) {
      if (p.gq) cudaFree(p.gq);
      QMOE_CUDA(l, dalloc(&p.gq, gq_bytes), "allocate GEMM layout");
      p.gq_bytes = gq_bytes;
    }
    GemmRepackArgs ga{};
    ga.codes = p.codes;
    ga.scales = p.scales;
    ga.zp = p.zp;
    ga.out = p.gq;
    ga.E = l->E;
    ga.N = p.N;
    ga.K = p.K;
    ga.I = l->I;
    ga.fc = pairs ? 1 : 2;
    ga.interleaved = l->fc1_interleaved;
    ga.L = p.GL;
    QMOE_CUDA(l, launch_repack_gemm(ga, s), "repack weights (GEMM layout)");
  }
  p.ready = true;
  return QMOE_OK;
}

qmoe_status qmoe_forward(qmoe_layer* l, const void* x, const float* logits, void* out,
                         int64_t T, void* stream) {
  if (!l) return QMOE_ERR_INVALID_ARG;
  if (T < 0) return fail(l, QMOE_ERR_INVALID_ARG, "num_tokens < 0");
  if (T == 0) return QMOE_OK;
  if (!x || !logits || !out) return fail(l, QMOE_ERR_INVALID_ARG, "null x / logits / out");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(l, QMOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
  if (!l->proj[0].ready || !l->proj[1].ready)
    return fail(l, QMOE_ERR_STATE, "prepack fc1 and fc2 before qmoe_forward");
  if (T * l->k > INT_MAX / 8) return fail(l, QMOE_ERR_INVALID_ARG, "num_tokens too large");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T > l->cap_T) {
    if (capturing(s))
      return fail(l, QMOE_ERR_STATE, "num_tokens exceeds the reservation during graph capture");
    const qmoe_status st = ensure_workspace(l, T);
    if (st != QMOE_OK) return st;
  }
  FusedShape fs{};
  if (fused_applies(l, T, &fs)) return forward_fused(l, x, logits, out, T, fs, s);
  int tb0, tb1;
  item_heights(l, T, &tb0, &tb1);
  l->last_T = T;
  l->last_path = QMOE_PATH_SEPARATE;
  l->last_tb[0] = tb0;
  l->last_tb[1] = tb1;
  const WaitCfg wait{l->status, l->wait_limit};
  // An expert can receive at most T rows: only when T exceeds the threshold
  // can the grouped-GEMM class be non-empty.
  const bool gemm = l->dtype != QMOE_F32 && l->tiles_ok && T > l->gemm_min_rows;
  const int threshold = gemm ? l->gemm_min_rows : INT_MAX;
  // slot-ordered combine: asked for, or automatic at decode sizes (measured
  // +2-3 % there against +4.3 % at the prefill workload)
  const bool ordered = l->deterministic == QMOE_COMBINE_ORDERED ||
                       (l->deterministic == QMOE_COMBINE_AUTO && T <= kCombineAutoMaxTokens);

  trace(l, QMOE_TRACE_BEGIN, s);
  RouteArgs ra{};
  ra.logits = logits;
  ra.T = (int)T;
  ra.E = l->E;
  ra.k = l->k;
  ra.normalize = l->normalize;
  ra.ids = l->ids;
  ra.w = l->w;
  ra.counts = l->counts;
  ra.offsets = l->offsets;
  ra.perm = l->perm;
  ra.pos = l->pos;
  ra.cntg = l->cntg;
  ra.rnk = l->rnk;
  ra.items[0] = l->items[0];
  ra.items[1] = l->items[1];
  ra.n_items = l->n_items;
  ra.tb[0] = tb0;
  ra.tb[1] = tb1;
  ra.threshold = threshold;
  ra.cap[0] = (int)items_cap(l, 0, T, tb0);
  ra.cap[1] = (int)items_cap(l, 1, T, tb1);
  if (gemm) {
    // class-0 experts have at most `threshold` rows each
    const int64_t per = ((int64_t)threshold + tb0 - 1) / tb0;
    if ((int64_t)l->E * per < ra.cap[0]) ra.cap[0] = (int)((int64_t)l->E * per);
  }
  // fc1's grouped GEMM writes its token tiles itself, overlapped with its
  // MMAs, at prefill shapes (T > 64); decode shapes gather first (measured:
  // the overlap costs their fc1 more than the gather kernel takes)
  const bool gemm_gathers = gemm && T > 64;
  ra.gready = gemm_gathers ? l->gready : nullptr;
  ra.gready_n = ra.cap[1];
  QMOE_CUDA(l, launch_route_group(ra, T <= 64, s), "launch routing");
  if (gemm && !gemm_gathers)
    QMOE_CUDA(l, launch_gather_tiles(x, l->perm, l->k, l->H, l->items[1], l->n_items + 1, ra.cap[1], l->xt, s),
              "launch gather");
  trace(l, QMOE_TRACE_ROUTED, s);

  for (int f = 0; f < 2; ++f) {
    const Proj& p = l->proj[f];
    if (l->dtype == QMOE_F32) {
      SimtArgs sa{};
      sa.codes = p.codes;
      sa.scales = p.scales;
      sa.zp = p.zp;
      sa.bits = p.bits;
      sa.B = l->B;
      sa.K = p.K;
      sa.N_out = f == 0 ? l->I : l->H;
      sa.I_or_0 = f == 0 ? l->I : 0;
      sa.zp_bytes_row = p.zp_row;
      sa.items = l->items[0];
      sa.n_items = l->n_items;
      sa.max_items = ra.cap[0];
      sa.src = f == 0 ? x : l->hbuf;
      sa.perm = l->perm;
      sa.k = l->k;
      sa.fc = f + 1;
      sa.dtype = l->dtype;
      sa.act = act_params(l);
      sa.bias = l->bias[f];
      sa.interleaved = l->fc1_interleaved;
      sa.zp_mode = l->zp_mode;
      sa.zp_offset = l->zp_offset;
      sa.dst = f == 0 ? l->hbuf : (void*)l->ybuf;
      sa.E = l->E;
      QMOE_CUDA(l, launch_simt(sa, s), "launch SIMT projection");
    } else {
      DecodeArgs da{};
      da.wpk = p.dec;
      da.L = p.L;
      da.K = p.K;
      da.N_out = f == 0 ? l->I : l->H;
      da.items = l->items[0];
      da.n_items = l->n_items;
      da.max_items = ra.cap[0];
      da.src = f == 0 ? x : l->hbuf;
      da.perm = l->perm;
      da.k = l->k;
      da.fc = f + 1;
      da.ng = tb0 / 8;
      da.dst = f == 0 ? l->hbuf : (void*)l->ybuf;
      da.act = act_params(l);
      da.bias = l->bias[f];
      da.zp_mode = l->zp_mode;
      da.zp_offset = l->zp_offset;
      da.bf16 = l->dtype == QMOE_BF16;
      da.wait = wait;
      da.pdl = 1;
      da.inject_stall = l->inject_stall;
      da.atomic = gemm && f == 1 && !ordered;
      da.out_acc = l->out_acc;
      da.w = l->w;
      QMOE_CUDA(l, launch_decode_mma(da, s), "launch decode projection");
      if (gemm) {
        GemmArgs ga{};
        ga.wq = p.gq;
        ga.L = p.GL;
        ga.items = l->items[1];
        ga.n_items = l->n_items + 1;
        ga.max_items = ra.cap[1];
        const int64_t max_tiles = (int64_t)ra.cap[1] * p.GL.ntiles;
        ga.grid = (int)(max_tiles < l->num_sms ? max_tiles : l->num_sms);
        // an expert receives at most T rows: with T <= 64 every item fits
        // the decode ring shape
        ga.dec = T <= 64 ? 1 : 0;
        ga.fc = f + 1;
        ga.act = act_params(l);
        ga.bias = l->bias[f];
        ga.zp_mode = l->zp_mode;
        ga.bf16 = l->dtype == QMOE_BF16;
        ga.zp_offset = l->zp_offset;
        ga.btiles = f == 0 ? l->xt : l->ht;
        if (f == 0) {
          ga.gx = gemm_gathers ? x : nullptr;
          ga.gH = l->H;
          ga.gready = l->gready;
          // fc2 reduces into the accumulator (finalize reads it, no clearing there)
          ga.zacc = ordered ? nullptr : l->out_acc;
          ga.zacc_n4 = (size_t)T * l->H / 4;
        }
        ga.htiles = l->ht;
        ga.h_ksteps = (l->I + 63) / 64;
        ga.out_acc = l->out_acc;
        ga.ybuf = f == 1 && ordered ? l->ybuf : nullptr;
        ga.perm = l->perm;
        ga.w = l->w;
        ga.k = l->k;
        ga.N_out = f == 0 ? l->I : l->H;
        ga.wait = wait;
        ga.inject_stall = l->inject_stall;
        QMOE_CUDA(l, launch_gemm(ga, s), "launch grouped GEMM");
      }
    }
    trace(l, f == 0 ? QMOE_TRACE_FC1 : QMOE_TRACE_FC2, s);
  }

  if (gemm && !ordered) {
    QMOE_CUDA(l, launch_finalize_acc(l->out_acc, out, (size_t)T * l->H, l->dtype, s), "launch combine");
  } else {
    FinalizeArgs fa{};
    fa.y = l->ybuf;
    fa.w = l->w;
    fa.pos = l->pos;
    fa.out = out;
    fa.T = (int)T;
    fa.H = l->H;
    fa.k = l->k;
    fa.dtype = l->dtype;
    fa.pdl = 1;
    QMOE_CUDA(l, launch_finalize(fa, s), "launch combine");
  }
  trace(l, QMOE_TRACE_END, s);
  return QMOE_OK;
}

qmoe_status qmoe_forward_host(qmoe_layer* l, const void* x_host, const float* logits_host,
                              void* out_host, int64_t T, void* stream) {
  if (!l) return QMOE_ERR_INVALID_ARG;
  if (T < 0) return fail(l, QMOE_ERR_INVALID_ARG, "num_tokens < 0");
  if (T == 0) return QMOE_OK;
  if (!x_host || !logits_host || !out_host) return fail(l, QMOE_ERR_INVALID_ARG, "null host buffer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T > l->cap_T) {
    const qmoe_status st = ensure_workspace(l, T);
    if (st != QMOE_OK) return st;
  }
  const size_t xb = (size_t)T * l->H * l->dsize;
  QMOE_CUDA(l, cudaMemcpyAsync(l->x_stage, x_host, xb, cudaMemcpyHostToDevice, s), "copy x");
  QMOE_CUDA(l, cudaMemcpyAsync(l->logits_stage, logits_host, (size_t)T * l->E * sizeof(float),
                               cudaMemcpyHostToDevice, s),
            "copy logits");
  const qmoe_status st = qmoe_forward(l, l->x_stage, l->logits_stage, l->out_stage, T, stream);
  if (st != QMOE_OK) return st;
  QMOE_CUDA(l, cudaMemcpyAsync(out_host, l->out_stage, xb, cudaMemcpyDeviceToHost, s), "copy out");
  QMOE_CUDA(l, cudaStreamSynchronize(s), "synchronise");
  return QMOE_OK;
}

qmoe_status qmoe_get_routing(qmoe_layer* l, int32_t* ids, float* weights, int32_t* perm,
                             int32_t* offsets, void* stream) {
  if (!l) return QMOE_ERR_INVALID_ARG;
  if (l->last_T == 0) return fail(l, QMOE_ERR_STATE, "no forward has run");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t R = (size_t)l->last_T * l->k;
  if (ids) QMOE_CUDA(l, cudaMemcpyAsync(ids, l->ids, R * 4, cudaMemcpyDeviceToDevice, s), "copy ids");
  if (weights) QMOE_CUDA(l, cudaMemcpyAsync(weights, l->w, R * 4, cudaMemcpyDeviceToDevice, s), "copy w");
  if (perm) QMOE_CUDA(l, cudaMemcpyAsync(perm, l->perm, R * 4, cudaMemcpyDeviceToDevice, s), "copy perm");
  if (offsets)
    QMOE_CUDA(l, cudaMemcpyAsync(offsets, l->offsets, (l->E + 1) * 4, cudaMemcpyDeviceToDevice, s),
              "copy offsets");
  return QMOE_OK;
}

int64_t qmoe_worklist_capacity(const qmoe_layer* l, int which, int64_t T) {
  if (!l || (which != 0 && which != 1) || T < 0) return -1;
  int tb0, tb1;
  item_heights(l, T, &tb0, &tb1);
  return items_cap(l, which, T, which == 0 ? tb0 : tb1);
}

qmoe_status qmoe_get_worklist(qmoe_layer* l, int which, int32_t* items, int32_t* count,
                              int64_t capacity, int* m_tile_host, void* stream) {
  if (!l || (which != 0 && which != 1)) return QMOE_ERR_INVALID_ARG;
  if (l->last_T == 0) return fail(l, QMOE_ERR_STATE, "no forward has run");
  const int64_t need = items_cap(l, which, l->last_T, l->last_tb[which]);
  if (capacity < need) return fail(l, QMOE_ERR_INVALID_ARG, "work-list capacity too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (items)
    QMOE_CUDA(l, cudaMemcpyAsync(items, l->items[which], need * sizeof(Item), cudaMemcpyDeviceToDevice, s),
              "copy items");
  if (count)
    QMOE_CUDA(l, cudaMemcpyAsync(count, l->n_items + which, sizeof(int), cudaMemcpyDeviceToDevice, s),
              "copy count");
  if (m_tile_host) *m_tile_host = l->last_tb[which];
  return QMOE_OK;
}

qmoe_status qmoe_set_trace_events(qmoe_layer* l, void* const* events, int n) {
  if (!l) return QMOE_ERR_INVALID_ARG;
  if (!events) {
    l->trace_on = false;
    return QMOE_OK;
  }
  if (n != QMOE_TRACE_NUM_EVENTS) return fail(l, QMOE_ERR_INVALID_ARG, "need QMOE_TRACE_NUM_EVENTS events");
  for (int i = 0; i < n; ++i) l->trace[i] = static_cast<cudaEvent_t>(events[i]);
  l->trace_on = true;
  return QMOE_OK;
}

qmoe_status qmoe_poll_device_status(qmoe_layer* l) {
  if (!l) return QMOE_ERR_INVALID_ARG;
  // The layer's own status word and, once qmoe_forward_noalloc has run in
  // this context, the one at the start of its static array.
  int* words[2] = {l->status, nullptr};
  void* na = nullptr;
  QMOE_CUDA(l, noalloc_status_word(&na), "look up the static scratch array");
  words[1] = static_cast<int*>(na);
  if (!words[0] && !words[1]) return QMOE_OK;
  QMOE_CUDA(l, cudaDeviceSynchronize(), "synchronise");
  int h = 0;
  for (int* w : words) {
    if (!w) continue;
    int v = 0;
    QMOE_CUDA(l, cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost), "read status");
    if (v != 0) QMOE_CUDA(l, cudaMemset(w, 0, sizeof(int)), "clear status");
    if (v == DEV_TIMEOUT) h = DEV_TIMEOUT;
    // after a wait of the layer ran out, its single-launch counters start over
    if (v != 0 && w == l->status && l->sync)
      QMOE_CUDA(l, cudaMemset(l->sync, 0, l->sync_n * sizeof(int)), "clear counters");
  }
  if (h == DEV_TIMEOUT) return fail(l, QMOE_ERR_TIMEOUT, "a bounded device-side wait ran out");
  return QMOE_OK;
}

const char* qmoe_last_error(const qmoe_layer* l) {
  if (!l) return "null layer";
  return l->err.c_str();
}

const char* qmoe_status_string(qmoe_status st) {
  if ((int)st < 0 || (int)st > 6) return "QMOE_ERR_UNKNOWN";
  return kStatusNames[st];
}

void qmoe_destroy(qmoe_layer* l) {
  if (!l) return;
  if (l->device >= 0 || l->cap_T > 0) cudaDeviceSynchronize();
  free_workspace(l);
  for (float* b : l->bias)
    if (b) cudaFree(b);
  for (Proj& p : l->proj) {
    if (p.codes) cudaFree(p.codes);
    if (p.scales) cudaFree(p.scales);
    if (p.zp) cudaFree(p.zp);
    if (p.dec) cudaFree(p.dec);
    if (p.gq) cudaFree(p.gq);
  }
  delete l;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Forward without allocation: the workspace lives in one static device array.
//
// For callers that may not allocate device memory when they run the layer
// (allocation-free graph capture, a framework allocator that owns the whole
// device, fixed memory plans).  See qmoe_forward_noalloc in qmoe.h.
// ----------------------------------------------------------------------------
namespace {

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[QMOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};
CUcontext g_noalloc_ctx[kMaxDevices] = {};

// The calling thread's current CUDA context, through the runtime's driver
// entry-point lookup (the library does not link the driver library itself,
// so it still loads on a machine without a GPU driver); nullptr if unknown.
CUcontext current_context() {
  using GetCurrent = CUresult (*)(CUcontext*);
  static GetCurrent fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<GetCurrent>(p);
  }();
  CUcontext ctx = nullptr;
  if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// (with that device current) once per device and CUDA context and cached; a
// new context (after cudaDeviceReset, say) may place the array elsewhere.
// `lookup` = false only reads the cache (nullptr if never looked up here).
cudaError_t noalloc_scratch(void** out, bool lookup = true) {
  *out = nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev] || g_noalloc_ctx[dev] != ctx) {
    if (!lookup) return cudaSuccess;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx[dev] = ctx;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

struct NoAllocPlan {
  size_t ids, w, counts, offsets, perm, pos, n_items, items0, items1, hbuf, ybuf, status, total;
};

size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

namespace {
// The status word is the array's first int (offset 0 in every plan).
cudaError_t noalloc_status_word(void** out) { return noalloc_scratch(out, false); }
}  // namespace

namespace {

NoAllocPlan noalloc_plan(const qmoe_layer* l, int64_t T, int cap0) {
  const size_t R = (size_t)T * l->k;
  NoAllocPlan p;
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o = up256(o + bytes); return at; };
  // The status word sits at offset 0 whatever the token count, so a timeout
  // stays readable (qmoe_poll_device_status) until it is polled.
  p.status = take(sizeof(int));
  p.ids = take(R * sizeof(int));
  p.w = take(R * sizeof(float));
  p.counts = take((size_t)l->E * sizeof(int));
  p.offsets = take(((size_t)l->E + 1) * sizeof(int));
  p.perm = take(R * sizeof(int));
  p.pos = take(R * sizeof(int));
  p.n_items = take(2 * sizeof(int));
  p.items0 = take((size_t)cap0 * sizeof(Item));
  p.items1 = take(sizeof(Item));
  p.hbuf = take(R * l->I * (size_t)l->dsize);
  p.ybuf = take(R * l->H * sizeof(float));
  p.total = o;
  return p;
}

}  // namespace

extern "C" qmoe_status qmoe_forward_noalloc(qmoe_layer* l, const void* x, const float* logits,
                                            void* out, int64_t T, void* stream) {
  if (!l) return QMOE_ERR_INVALID_ARG;
  if (T < 0) return fail(l, QMOE_ERR_INVALID_ARG, "num_tokens < 0");
  if (T == 0) return QMOE_OK;
  if (!x || !logits || !out) return fail(l, QMOE_ERR_INVALID_ARG, "null x / logits / out");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(l, QMOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
  if (!l->proj[0].ready || !l->proj[1].ready)
    return fail(l, QMOE_ERR_STATE, "prepack fc1 and fc2 before qmoe_forward_noalloc");
  if (T * l->k > INT_MAX / 8) return fail(l, QMOE_ERR_INVALID_ARG, "num_tokens too large");
  int tb0, tb1;
  item_heights(l, T, &tb0, &tb1);
  const int64_t cap0 = items_cap(l, 0, T, tb0);
  const NoAllocPlan plan = noalloc_plan(l, T, (int)cap0);
  if (plan.total > (size_t)QMOE_NOALLOC_SCRATCH_BYTES)
    return fail(l, QMOE_ERR_UNSUPPORTED,
                "qmoe_forward_noalloc: " + std::to_string(T) + " tokens need " +
                    std::to_string(plan.total) + " bytes of scratch, more than the " +
                    std::to_string((size_t)QMOE_NOALLOC_SCRATCH_BYTES) +
                    "-byte static array; use qmoe_forward");
  void* base = nullptr;
  QMOE_CUDA(l, noalloc_scratch(&base), "look up the static scratch array");
  unsigned char* sb = static_cast<unsigned char*>(base);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The status word is zero when the library loads and is cleared only by
  // qmoe_poll_device_status (a timeout stays visible until it is polled).
  int* status = reinterpret_cast<int*>(sb + plan.status);
  int* ids = reinterpret_cast<int*>(sb + plan.ids);
  float* w = reinterpret_cast<float*>(sb + plan.w);
  int* perm = reinterpret_cast<int*>(sb + plan.perm);
  int* pos = reinterpret_cast<int*>(sb + plan.pos);
  int* n_items = reinterpret_cast<int*>(sb + plan.n_items);
  Item* items0 = reinterpret_cast<Item*>(sb + plan.items0);
  void* hbuf = sb + plan.hbuf;
  float* ybuf = reinterpret_cast<float*>(sb + plan.ybuf);

  RouteArgs ra{};
  ra.logits = logits;
  ra.T = (int)T;
  ra.E = l->E;
  ra.k = l->k;
  ra.normalize = l->normalize;
  ra.ids = ids;
  ra.w = w;
  ra.counts = reinterpret_cast<int*>(sb + plan.counts);
  ra.offsets = reinterpret_cast<int*>(sb + plan.offsets);
  ra.perm = perm;
  ra.pos = pos;
  ra.items[0] = items0;
  ra.items[1] = reinterpret_cast<Item*>(sb + plan.items1);
  ra.n_items = n_items;
  ra.tb[0] = tb0;
  ra.tb[1] = tb1;
  ra.threshold = INT_MAX;  // decode kernels only
  ra.cap[0] = (int)cap0;
  ra.cap[1] = 1;
  QMOE_CUDA(l, launch_route_group(ra, T <= 64, s), "launch routing");

  const WaitCfg wait{status, l->wait_limit};
  for (int f = 0; f < 2; ++f) {
    const Proj& p = l->proj[f];
    if (l->dtype == QMOE_F32) {
      SimtArgs sa{};
      sa.codes = p.codes;
      sa.scales = p.scales;
      sa.zp = p.zp;
      sa.bits = p.bits;
      sa.B = l->B;
      sa.K = p.K;
      sa.N_out = f == 0 ? l->I : l->H;
      sa.I_or_0 = f == 0 ? l->I : 0;
      sa.zp_bytes_row = p.zp_row;
      sa.items = items0;
      sa.n_items = n_items;
      sa.max_items = (int)cap0;
      sa.src = f == 0 ? x : hbuf;
      sa.perm = perm;
      sa.k = l->k;
      sa.fc = f + 1;
      sa.dtype = l->dtype;
      sa.act = act_params(l);
      sa.bias = l->bias[f];
      sa.interleaved = l->fc1_interleaved;
      sa.zp_mode = l->zp_mode;
      sa.zp_offset = l->zp_offset;
      sa.dst = f == 0 ? hbuf : (void*)ybuf;
      sa.E = l->E;
      QMOE_CUDA(l, launch_simt(sa, s), "launch SIMT projection");
    } else {
      DecodeArgs da{};
      da.wpk = p.dec;
      da.L = p.L;
      da.K = p.K;
      da.N_out = f == 0 ? l->I : l->H;
      da.items = items0;
      da.n_items = n_items;
      da.max_items = (int)cap0;
      da.src = f == 0 ? x : hbuf;
      da.perm = perm;
      da.k = l->k;
      da.fc = f + 1;
      da.ng = tb0 / 8;
      da.dst = f == 0 ? hbuf : (void*)ybuf;
      da.act = act_params(l);
      da.bias = l->bias[f];
      da.zp_mode = l->zp_mode;
      da.zp_offset = l->zp_offset;
      da.bf16 = l->dtype == QMOE_BF16;
      da.wait = wait;
      da.pdl = 1;
      da.inject_stall = l->inject_stall;
      QMOE_CUDA(l, launch_decode_mma(da, s), "launch decode projection");
    }
  }
  FinalizeArgs fa{};
  fa.y = ybuf;
  fa.w = w;
  fa.pos = pos;
  fa.out = out;
  fa.T = (int)T;
  fa.H = l->H;
  fa.k = l->k;
  fa.dtype = l->dtype;
  fa.pdl = 1;
  QMOE_CUDA(l, launch_finalize(fa, s), "launch combine");
  return QMOE_OK;
}
