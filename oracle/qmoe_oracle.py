"""CPU oracle of the QMoE layer forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module.  The CUDA library never calls it, and it shares no
code with the CUDA path: it reads the canonical (boundary) tensors directly.

It is a plain, slow, obviously-correct restatement of what the layer computes,
in float64, written from these pages:

* onnx-runtime-ep-cuda ``src/kernels/qmoe.rs`` (CUDA_SRC): ``total_order_key``
  / ``route_value_is_better`` and ``qmoe_route`` (selection order, softmax
  weights, renormalisation); ``decode_affine_weight`` (LSB-first packing,
  ``(q - zp) * scale``, symmetric centre ``1 << (bits-1)``, packed zero
  points); ``swiglu_value`` and the tanh-GELU of ``qmoe_activate``;
  ``qmoe_combine_impl`` (slot-ordered weighted combine, round to nearest
  even into the output type).
* onnxruntime PR "[CUDA] QMoE: fused int2 mixed-input GEMM + GeGLU activation
  + fractional zero-point": ``zero_point_offset`` (``(code - offset) *
  scale``) and the GeGLU gate (``down(gelu_tanh(gate) * up)``).
* onnxruntime PR "[CUDA] Add fast INT3 QMoE kernels ...": review item "Round
  dequantized weights before accumulation" -- each dequantised weight is
  rounded to the activation type before it is multiplied.
* metrale ``gemm_quant_moe.rs``, ``moe_build_tile_worklist``: the tile
  work-list order (experts ascending, then m-tile, then n-tile).

Readings where the pages leave a step open:
selection is on the fp32 logits (equal to selection on the exact softmax,
which is strictly increasing); fc1 rows are concatenated ``[gate | up]``;
scales are stored in the activation type D; biases are fp32 (qmoe.rs);
the SwiGLU attributes do not apply to GeGLU; intermediates (fc1 output,
activation, fc2 output) stay unrounded in float64; the int3 stream is one
LSB-first bit stream per row.

Every function here is pinned by ``tests/test_oracle.py`` against something
other than itself (brute force, hand cases from the pages, library routines,
invariants).
"""
from __future__ import annotations

import numpy as np

# Formats: (significand bits incl. the implicit one, minimum normal exponent,
# maximum exponent).
_FORMATS = {
    "f32": (24, -126, 127),
    "f16": (11, -14, 15),
    "bf16": (8, -126, 127),
}


# ----------------------------------------------------------------------------
# Rounding into the activation type
# ----------------------------------------------------------------------------
def round_to_dtype(x, dtype: str) -> np.ndarray:
    """Round float64 values to the nearest value of ``dtype`` (ties to even),
    returned as float64.  Covers subnormals and overflow to infinity.

    Used for the dequantised weights (PR "fast INT3" review: round the
    dequantised weight to T) and the layer output (``qmoe_store`` uses
    ``__float2half_rn`` / ``__float2bfloat16_rn``).
    """
    p, emin, emax = _FORMATS[dtype]
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                 # x = m * 2**e, 0.5 <= |m| < 1
    unbiased = e - 1                   # x = 1.f * 2**unbiased
    keep = p - np.maximum(emin - unbiased, 0)   # significand bits kept
    r = np.ldexp(np.rint(np.ldexp(m, keep)), e - keep)
    max_finite = (2.0 - 2.0 ** (1 - p)) * 2.0 ** emax
    r = np.where(np.abs(r) > max_finite, np.copysign(np.inf, x), r)
    return np.where(np.isfinite(x), r, x)


# ----------------------------------------------------------------------------
# a-1: routing
# ----------------------------------------------------------------------------
def total_order_key(logits_f32) -> np.ndarray:
    """Signed 32-bit key that orders fp32 values totally (-0.0 < +0.0):
    the sign-magnitude bit pattern with the magnitude bits flipped for
    negative values (qmoe.rs ``total_order_key``)."""
    bits = np.asarray(logits_f32, dtype=np.float32).view(np.int32).astype(np.int64)
    neg = bits < 0
    key = np.where(neg, bits ^ 0x7FFFFFFF, bits)
    return key.astype(np.int32)


def select_experts(logits_f32, k: int) -> np.ndarray:
    """Top-k experts per token, in rank order (slot j = rank j).  Larger key
    first; equal keys go to the lower expert index (qmoe.rs
    ``route_value_is_better`` and the k passes of ``qmoe_route``)."""
    logits_f32 = np.asarray(logits_f32, dtype=np.float32)
    T, E = logits_f32.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    key = total_order_key(logits_f32).astype(np.int64)
    idx = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((idx, -key), axis=1)
    return order[:, :k].astype(np.int32)


def routing_weights(logits_f32, ids, normalize: bool) -> np.ndarray:
    """Softmax routing weights of the selected experts (qmoe.rs ``qmoe_route``
    without ``router_weights``): ``p_e = exp(l_e - max_all)``; divided by the
    sum over all E experts, or over the k selected ones when ``normalize``."""
    l = np.asarray(logits_f32, dtype=np.float32).astype(np.float64)
    m = l.max(axis=1, keepdims=True)
    p = np.exp(l - m)
    p_sel = np.take_along_axis(p, np.asarray(ids, dtype=np.int64), axis=1)
    denom = p_sel.sum(axis=1, keepdims=True) if normalize else p.sum(axis=1, keepdims=True)
    return p_sel / denom


# ----------------------------------------------------------------------------
# a-2 / a-3: grouping and tile work-list
# ----------------------------------------------------------------------------
def group_routes(ids, E: int):
    """Expert grouping of the routes r = t*k + j.

    Returns ``counts[E]``, exclusive ``offsets[E+1]``, the stable permutation
    ``perm`` (the routes of expert e, in ascending r, occupy
    ``perm[offsets[e]:offsets[e+1]]``) and its inverse ``pos``.
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    perm = np.empty(flat.size, dtype=np.int64)
    cursor = offsets[:-1].copy()
    for r, e in enumerate(flat):          # ascending r: stable
        perm[cursor[e]] = r
        cursor[e] += 1
    pos = np.empty_like(perm)
    pos[perm] = np.arange(perm.size)
    return counts, offsets, perm, pos


def build_worklist(offsets, m_tile: int, n_tiles: int = 1, expert_filter=None):
    """Tile work-list (metrale ``moe_build_tile_worklist``): one item per
    (expert, m-tile, n-tile) of each expert that has rows, experts ascending,
    then m-tile, then n-tile.  Items are ``(e, row_start, rows, n_tile)``
    with ``row_start`` an index into the grouped (permuted) route order.
    ``expert_filter(e, count)`` restricts the list to a class of experts."""
    items = []
    E = len(offsets) - 1
    for e in range(E):
        c = int(offsets[e + 1] - offsets[e])
        if c == 0 or (expert_filter is not None and not expert_filter(e, c)):
            continue
        for m in range((c + m_tile - 1) // m_tile):
            start = int(offsets[e]) + m * m_tile
            rows = min(m_tile, c - m * m_tile)
            for n in range(n_tiles):
                items.append((e, start, rows, n))
    return items


# ----------------------------------------------------------------------------
# a-0 / a-4: dequantisation
# ----------------------------------------------------------------------------
def unpack_fields(packed, bits: int, count: int) -> np.ndarray:
    """Read ``count`` fields of ``bits`` bits from LSB-first bit streams
    (last axis = bytes): field d = bits [d*bits, d*bits + bits) of the row
    (qmoe.rs ``decode_affine_weight``: byte d/pack, shift (d%pack)*bits)."""
    packed = np.asarray(packed, dtype=np.uint8)
    bitarr = np.unpackbits(packed, axis=-1, bitorder="little")
    bitarr = bitarr[..., : count * bits].reshape(packed.shape[:-1] + (count, bits))
    weights = (1 << np.arange(bits)).astype(np.int64)
    return (bitarr.astype(np.int64) * weights).sum(axis=-1)


def zero_points(zp_mode: str, bits: int, n_rows: int, n_blocks: int,
                zp_packed=None, zp_offset: float = float("nan")) -> np.ndarray:
    """Per-(row, block) zero point as float64.

    * ``sym``:    the symmetric centre 2**(bits-1) (qmoe.rs).
    * ``uint8``:  the block's field of the packed zero-point row (qmoe.rs).
    * ``offset``: one fractional centre for every weight (PR "fused int2 ...",
      ``zero_point_offset``).
    """
    if zp_mode == "sym":
        return np.full((n_rows, n_blocks), float(1 << (bits - 1)))
    if zp_mode == "uint8":
        return unpack_fields(zp_packed, bits, n_blocks).astype(np.float64)
    if zp_mode == "offset":
        return np.full((n_rows, n_blocks), float(zp_offset))
    raise ValueError(zp_mode)


def dequantize(codes_packed, scales, bits: int, B: int, K: int, dtype: str,
               zp_mode: str, zp_packed=None, zp_offset: float = float("nan")) -> np.ndarray:
    """Dense weights of one expert, ``W[n, d] = R_D((q[n,d] - z[n, d//B]) *
    s[n, d//B])``: the affine decode of qmoe.rs ``decode_affine_weight`` with
    the zero point of :func:`zero_points`, then rounded to the activation type
    (PR "fast INT3" review).  ``(q - z) * s`` is exact in float64."""
    q = unpack_fields(codes_packed, bits, K).astype(np.float64)      # [N, K]
    n_rows = q.shape[0]
    s = np.asarray(scales, dtype=np.float64)                          # [N, K/B]
    z = zero_points(zp_mode, bits, n_rows, K // B, zp_packed, zp_offset)
    blk = np.arange(K) // B
    return round_to_dtype((q - z[:, blk]) * s[:, blk], dtype)


# ----------------------------------------------------------------------------
# a-6: gated activation
# ----------------------------------------------------------------------------
def silu(g):
    """``g * sigmoid(g)``: ``swiglu_value`` with alpha = 1, beta = 0 and no
    limit (the qmoe.rs attribute defaults)."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def gelu_tanh(g):
    """tanh-form GELU of ``qmoe_activate`` (activation 1):
    ``0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)))``."""
    g = np.asarray(g, dtype=np.float64)
    return 0.5 * g * (1.0 + np.tanh(0.7978845608028654 * (g + 0.044715 * g * g * g)))


def swiglu(g, u, alpha: float = 1.0, beta: float = 0.0, limit: float = float("inf")):
    """qmoe.rs ``swiglu_value``: the gate is bounded above by ``limit``, the
    linear half clamped to [-limit, limit]; then
    ``g' * sigmoid(alpha * g') * (u' + beta)``.  With the attribute defaults
    (alpha 1, beta 0, no limit) this is ``silu(g) * u``."""
    g = np.minimum(np.asarray(g, dtype=np.float64), limit)
    u = np.clip(np.asarray(u, dtype=np.float64), -limit, limit)
    return g / (1.0 + np.exp(-alpha * g)) * (u + beta)


GATED = ("swiglu", "geglu")


def act_single(a, act: str):
    """Non-gated activation of fc1's output (qmoe.rs ``qmoe_activate``,
    activation 0 / 1 / 2 without fc3 / 4): relu, tanh-GELU (evaluated in
    double there too), silu v * sigmoid(v), identity."""
    a = np.asarray(a, dtype=np.float64)
    if act == "relu":
        return np.maximum(a, 0.0)
    if act == "gelu":
        return gelu_tanh(a)
    if act == "silu":
        return silu(a)
    if act == "identity":
        return a
    raise ValueError(act)


def split_gate_up(a, inter: int, layout: str = "concat"):
    """Gate and up halves of fc1's output (qmoe.rs ``qmoe_activate``):
    swiglu_fusion == 2 concatenates them (gate = a[:, :I], up = a[:, I:]),
    swiglu_fusion == 1 interleaves them (gate = a[:, 2f], up = a[:, 2f+1])."""
    if layout == "interleaved":
        return a[:, 0:2 * inter:2], a[:, 1:2 * inter:2]
    return a[:, :inter], a[:, inter:2 * inter]


def glu(a, inter: int, act: str, layout: str = "concat", alpha: float = 1.0, beta: float = 0.0,
        limit: float = float("inf")):
    """Gated activation of fc1's output: SwiGLU with the qmoe.rs attributes,
    or GeGLU (tanh-GELU gate times up; PR "fused int2 ..."; the SwiGLU
    attributes do not apply to it)."""
    gate, up = split_gate_up(a, inter, layout)
    if act == "swiglu":
        return swiglu(gate, up, alpha, beta, limit)
    return gelu_tanh(gate) * up


# ----------------------------------------------------------------------------
# The whole layer
# ----------------------------------------------------------------------------
def to_f64(t) -> np.ndarray:
    """Exact float64 copy of a CPU torch tensor / numpy array (f32/f16/bf16)."""
    if hasattr(t, "double"):
        return t.double().numpy()
    return np.asarray(t, dtype=np.float64)


def expert_weights(inputs: dict, fc: int, e: int) -> np.ndarray:
    """Dense dequantised weights of expert e for fc1 ([2I, H]; [I, H] for a
    non-gated activation or of gate rows beside a separate fc3), fc2 ([H, I])
    or fc3 ([I, H] up rows; fc1's code width, zero points and block size)."""
    cfg = inputs["cfg"]
    bits, K = (cfg.bits2, cfg.I) if fc == 2 else (cfg.bits1, cfg.H)
    pre = f"fc{fc}_"
    zp = inputs[pre + "zp"]
    return dequantize(
        np.asarray(inputs[pre + "codes"][e]), to_f64(inputs[pre + "scales"][e]), bits,
        cfg.B, K, cfg.dtype, cfg.zp_mode,
        None if zp is None else np.asarray(zp[e]), cfg.zp_offset)


def projection_bias(inputs: dict, fc: int, e: int):
    """fp32 bias row of expert e added to the projection output (qmoe.rs
    ``qmoe_linear_impl``: ``output = value + bias[expert * out + feature]``),
    or 0 without biases."""
    b = inputs.get(f"fc{fc}_bias")
    return 0.0 if b is None else to_f64(b[e])


def routing(inputs: dict):
    """Selection, weights, grouping for all tokens."""
    cfg = inputs["cfg"]
    logits = np.asarray(inputs["logits"], dtype=np.float32)
    ids = select_experts(logits, cfg.k)
    w = routing_weights(logits, ids, cfg.normalize)
    counts, offsets, perm, pos = group_routes(ids, cfg.E)
    return {"ids": ids, "weights": w, "counts": counts, "offsets": offsets,
            "perm": perm, "pos": pos}


def forward(inputs: dict, tokens=None, round_h: bool = False, return_parts: bool = False):
    """The QMoE layer forward on float64 data.

    ``out[t, m] = R_D( sum_j w[t, j] * y[t*k + j, m] )`` (slot order j) with
    ``y[r] = W2_e @ act_glu(W1_e @ x[t] + b1_e) + b2_e`` for route r = t*k + j
    of expert e = ids[t, j] (biases zero unless given).  ``tokens`` restricts the output to a subset of token rows
    (routing is still computed for all tokens).  ``round_h`` rounds the
    activation to D before fc2 (only to measure that gap; off by default).
    """
    cfg = inputs["cfg"]
    x = to_f64(inputs["x"])
    rt = routing(inputs)
    ids, w = rt["ids"], rt["weights"]
    tokens = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    need = {}
    for t in tokens:
        for j in range(cfg.k):
            need.setdefault(int(ids[t, j]), []).append((int(t), j))
    y = {}
    for e in sorted(need):
        rows = need[e]
        xe = x[[t for t, _ in rows]]                       # [M_e, H]
        a = xe @ expert_weights(inputs, 1, e).T + projection_bias(inputs, 1, e)   # [M_e, 2I] (I non-gated)
        layout = cfg.fc1_layout
        if layout == "separate":
            # qmoe.rs qmoe_activate with fc3: gate = fc1's output, linear = fc3's
            a3 = xe @ expert_weights(inputs, 3, e).T + projection_bias(inputs, 3, e)   # [M_e, I]
            a, layout = np.concatenate([a, a3], axis=1), "concat"
        if cfg.act in GATED:
            h = glu(a, cfg.I, cfg.act, layout, cfg.swiglu_alpha, cfg.swiglu_beta, cfg.swiglu_limit)
        elif cfg.act == "silu" and cfg.fc1_layout == "separate":
            # qmoe.rs uses_separate_gate: silu beside fc3 takes the gated
            # branch of qmoe_activate (swiglu_value of gate = fc1, linear = fc3)
            h = glu(a, cfg.I, "swiglu", layout, cfg.swiglu_alpha, cfg.swiglu_beta, cfg.swiglu_limit)
        else:
            h = act_single(a, cfg.act)
        if round_h:
            h = round_to_dtype(h, cfg.dtype)
        ye = h @ expert_weights(inputs, 2, e).T + projection_bias(inputs, 2, e)  # [M_e, H]
        for (t, j), row in zip(rows, ye):
            y[(t, j)] = row
    out = np.zeros((len(tokens), cfg.H))
    for i, t in enumerate(tokens):
        acc = np.zeros(cfg.H)
        for j in range(cfg.k):
            acc = acc + w[t, j] * y[(int(t), j)]
        out[i] = acc
    out = round_to_dtype(out, cfg.dtype)
    if return_parts:
        return out, rt
    return out


def tolerance(dtype: str, ref_max: float) -> float:
    """Output tolerance: 2e-3*max|ref| + 1e-3 for f32/f16 and
    8e-3*max|ref| + 4e-3 for bf16."""
    if dtype == "bf16":
        return 8e-3 * ref_max + 4e-3
    return 2e-3 * ref_max + 1e-3
