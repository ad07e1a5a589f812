"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Routing (selected experts, permutation, offsets, work-lists) must match
bit-exactly; outputs within max|err| <= 2e-3*max|ref| + 1e-3 (f32/f16) or
8e-3*max|ref| + 4e-3 (bf16)."""
import numpy as np
import pytest
import torch

from oracle import qmoe_oracle as O
from qmoe_inputs import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qm():
    from weight_only_quantized_qmoe_gb300 import build
    build.build()
    import weight_only_quantized_qmoe_gb300 as q
    return q


# The projection paths: the single launch (default; it serves 16-bit
# activations, <= 64 tokens and code widths {2, 3, 4}, the separate kernels
# otherwise), and with it switched off the tensor-core grouped GEMM for every
# expert or the mma.sync decode kernel (threshold above any expert's rows).
PATHS = {"fused": (1, 0), "gemm": (0, 0), "decode": (0, 10 ** 6)}


def separate_path(min_rows):
    """The separate kernels with experts above `min_rows` rows on the GEMM."""
    return (0, min_rows)


def run_layer(qm, inp, reserve=None, path="fused"):
    cfg = inp["cfg"]
    layer = qm.QMoELayer.from_config(cfg)
    fused, min_rows = PATHS.get(path, path)
    layer.set_fused_decode(fused)
    layer.set_gemm_min_rows(min_rows)
    if reserve:
        layer.reserve(reserve)
    x, logits = qm.load_inputs(layer, inp)
    out = layer.forward(x, logits)
    torch.cuda.synchronize()
    assert layer.poll() == 0
    return layer, out


def check_routing(layer, inp, path="fused"):
    from weight_only_quantized_qmoe_gb300 import binding
    cfg = inp["cfg"]
    ids, w, perm, offs = layer.routing(cfg.T)
    torch.cuda.synchronize()
    rt = O.routing(inp)
    np.testing.assert_array_equal(ids.cpu().numpy().reshape(cfg.T, cfg.k), rt["ids"])
    np.testing.assert_array_equal(perm.cpu().numpy(), rt["perm"])
    np.testing.assert_array_equal(offs.cpu().numpy(), rt["offsets"])
    np.testing.assert_allclose(w.cpu().numpy().reshape(cfg.T, cfg.k), rt["weights"],
                               rtol=2e-6, atol=1e-7)
    min_rows = PATHS.get(path, path)[1]
    if layer.last_path() == binding.QMOE_PATH_FUSED:
        # the single launch: every expert's rows in groups of m_tile, no GEMM class
        thr = 10 ** 9
    else:
        # experts with more than `min_rows` rows go to the grouped GEMM
        # (class 1) once T can exceed it; the rest to the decode kernel (class 0)
        thr = min_rows if (cfg.dtype != "f32" and cfg.T > min_rows) else None
    for which in (0, 1):
        items, m_tile = layer.worklist(which, cfg.T)
        if thr is None:
            flt = (lambda e, c: which == 0)
        else:
            flt = (lambda e, c, w_=which: (c > thr) == (w_ == 1))
        ref = O.build_worklist(rt["offsets"], m_tile, expert_filter=flt)
        got = [tuple(int(v) for v in row[:3]) for row in items.numpy()]
        assert got == [(e, s, r) for e, s, r, _ in ref], f"work-list {which}"
    return rt


def check_out(out, ref, dtype, tokens=None):
    got = out.float().cpu().numpy().astype(np.float64)
    if tokens is not None:
        got = got[tokens]
    err = np.abs(got - ref).max()
    tol = O.tolerance(dtype, np.abs(ref).max())
    assert err <= tol, f"max|err| {err:.3e} > tol {tol:.3e} (max|ref| {np.abs(ref).max():.3e})"
    return err, tol


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("name", ["tiny", "decode_int2", "decode_many_expert_int4", "mixed_int3_int4"])
def test_config_parity(qm, name, path):
    inp = make_inputs(CONFIGS[name])
    layer, out = run_layer(qm, inp, path=path)
    check_routing(layer, inp, path=path)
    check_out(out, O.forward(inp), inp["cfg"].dtype)


def stratified_tokens(rt, k, m_tile, seed=11):
    """Tokens whose routes reach every (expert, m_tile-row tile) of the grouped
    order: one random route per tile plus each expert's last (ragged) row.
    Returns the sorted tokens and the set of all (expert, tile) pairs."""
    rng = np.random.default_rng(seed)
    offsets, perm = rt["offsets"], rt["perm"]
    tokens, tiles = set(), set()
    for e in range(len(offsets) - 1):
        c = int(offsets[e + 1] - offsets[e])
        for t0 in range(0, c, m_tile):
            tiles.add((e, t0 // m_tile))
            tokens.add(int(perm[offsets[e] + t0 + rng.integers(min(m_tile, c - t0))]) // k)
        if c:
            tokens.add(int(perm[offsets[e + 1] - 1]) // k)
    return np.array(sorted(tokens)), tiles


def test_prefill_config_every_tile(qm):
    # Full-size prefill (T = 4096, 32768 routes, K = 4096): the oracle runs on
    # a token set whose routes land in every (expert, 128-row m-tile) of the
    # grouped GEMM, each expert's ragged last tile included.
    cfg = CONFIGS["prefill_int4"]
    inp = make_inputs(cfg)
    layer, out = run_layer(qm, inp)
    rt = check_routing(layer, inp)
    tokens, tiles = stratified_tokens(rt, cfg.k, 128)
    covered = set()
    for t in tokens:
        for j in range(cfg.k):
            r = t * cfg.k + j
            e = int(rt["ids"][t, j])
            covered.add((e, (int(rt["pos"][r]) - int(rt["offsets"][e])) // 128))
    assert covered == tiles and len(tiles) == sum(-(-int(c) // 128) for c in rt["counts"])
    ref = O.forward(inp, tokens=tokens)
    check_out(out, ref, cfg.dtype, tokens)


# ---------------------------------------------------------------------------
# Edge cases and the variant matrix (small shapes, full oracle comparison)
# ---------------------------------------------------------------------------
BASE = CONFIGS["tiny"].with_(H=256, I=128, E=8, k=2, dtype="bf16", B=32)

VARIANTS = {
    "T1": dict(T=1),
    "ragged_T37": dict(T=37),
    "k_equals_E": dict(E=4, k=4, T=9),
    "k1_no_renorm": dict(k=1, normalize=False, T=20),
    "int2_f16_offset_geglu": dict(bits1=2, bits2=2, zp_mode="offset", zp_offset=1.5, dtype="f16",
                                  act="geglu", B=128, T=6),
    "int2_K_much_larger_than_64": dict(bits1=2, bits2=2, H=1024, I=512, B=64, T=5),
    "int3_sym_B32": dict(bits1=3, bits2=3, B=32, T=11),
    "int3_uint8_B64": dict(bits1=3, bits2=4, zp_mode="uint8", zp_lo=0, zp_hi=7, B=64, T=7),
    "int4_uint8_f16_B128": dict(zp_mode="uint8", zp_lo=5, zp_hi=11, dtype="f16", B=128, T=13),
    "int2_uint8_B32": dict(bits1=2, bits2=2, zp_mode="uint8", zp_lo=0, zp_hi=3, B=32, T=10),
    "mixed_4_2_geglu_bf16": dict(bits1=4, bits2=2, act="geglu", T=16),
    "K_not_multiple_of_64": dict(H=96, I=96, B=32, T=6),
    "f32_int3_offset": dict(dtype="f32", bits1=3, bits2=2, zp_mode="offset", zp_offset=2.5, T=5),
    "f32_uint8": dict(dtype="f32", zp_mode="uint8", zp_lo=3, zp_hi=12, T=9),
    "many_tokens_one_group": dict(T=300, E=4, k=2),
    "wide_E_256": dict(E=256, k=6, T=40),
}


# qmoe.rs swiglu_fusion 1 (interleaved gate/up), the separate fc3 up
# projection, SwiGLU alpha / beta / limit (the limit clamps many gates and up
# values at these sizes) and fp32 biases, on both projection paths and the
# fp32 SIMT path.
FEATURE_VARIANTS = {
    "interleaved_bias_swiglu_params": dict(fc1_layout="interleaved", bias=True, swiglu_alpha=1.702,
                                           swiglu_beta=1.0, swiglu_limit=0.3, T=13),
    "bias_geglu_int2_offset_f16": dict(act="geglu", bias=True, bits1=2, bits2=2, zp_mode="offset",
                                       zp_offset=1.5, dtype="f16", B=128, T=9),
    "interleaved_uint8_T150": dict(fc1_layout="interleaved", zp_mode="uint8", zp_lo=5, zp_hi=11,
                                   E=4, T=150),
    "f32_interleaved_bias_params": dict(dtype="f32", fc1_layout="interleaved", bias=True,
                                        swiglu_alpha=1.702, swiglu_beta=1.0, swiglu_limit=0.3, T=7),
    # a long fc2 reduction (K = 1024) with biases
    "bias_long_fc2_k": dict(bias=True, I=1024, E=4, T=6),
    # qmoe.rs unfused SwiGLU: gate rows in fc1, up rows in a separate fc3
    "separate_fc3_bias_swiglu_params": dict(fc1_layout="separate", bias=True, swiglu_alpha=1.702,
                                            swiglu_beta=1.0, swiglu_limit=0.3, T=13),
    "separate_fc3_geglu_int2_offset_f16": dict(fc1_layout="separate", act="geglu", bias=True, bits1=2,
                                               bits2=2, zp_mode="offset", zp_offset=1.5, dtype="f16",
                                               B=128, T=9),
    "separate_fc3_uint8_T150": dict(fc1_layout="separate", zp_mode="uint8", zp_lo=5, zp_hi=11, E=4, T=150),
    "f32_separate_fc3_bias": dict(dtype="f32", fc1_layout="separate", bias=True, T=7),
    # qmoe.rs uses_separate_gate: silu beside fc3 is the gated form
    "silu_fc3_params": dict(act="silu", fc1_layout="separate", swiglu_limit=0.5, bias=True, T=11),
    # non-gated activations (qmoe.rs qmoe_activate): fc1 has I rows, h = act(fc1 output)
    "relu_bias": dict(act="relu", bias=True, T=13),
    "gelu_uint8_f16_B64": dict(act="gelu", zp_mode="uint8", zp_lo=5, zp_hi=11, dtype="f16", B=64, T=9),
    "silu_int2_offset_B128": dict(act="silu", bits1=2, bits2=2, zp_mode="offset", zp_offset=1.5, B=128,
                                  T=20),
    "identity_int8_f16": dict(act="identity", bits1=8, bits2=8, dtype="f16", T=12, scale_lo=0.0005,
                              scale_hi=0.002),
    "relu_T150_prefill_ring": dict(act="relu", bias=True, E=4, T=150),
    "f32_silu_bias": dict(dtype="f32", act="silu", bias=True, T=7),
}


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("name", list(FEATURE_VARIANTS))
def test_feature_parity(qm, name, path):
    cfg = BASE.with_(**FEATURE_VARIANTS[name])
    inp = make_inputs(cfg)
    layer, out = run_layer(qm, inp, path=path)
    check_routing(layer, inp, path=path)
    check_out(out, O.forward(inp), cfg.dtype)


# Every (fc1, fc2) code width in {2,3,4}^2 at every block size, on both
# projection paths; the zero-point mode and activation dtype rotate through
# the matrix so each appears with every width and block size.
def _width_cases():
    cases = []
    zps = ["sym", "uint8", "offset"]
    for b1 in (2, 3, 4):
        for b2 in (2, 3, 4):
            for blk in (32, 64, 128):
                i = len(cases)
                zp = zps[(b1 + b2 + blk // 32) % 3]
                kw = dict(bits1=b1, bits2=b2, B=blk, zp_mode=zp, dtype=("bf16", "f16")[i % 2], T=12)
                if zp == "uint8":
                    kw.update(zp_lo=0, zp_hi=(1 << min(b1, b2)) - 1)
                if zp == "offset":
                    kw.update(zp_offset=1.5)
                cases.append((f"w{b1}{b2}_B{blk}_{zp}", kw))
    return cases


WIDTH_CASES = dict(_width_cases())
# 8-bit codes (fp16 magic path; bf16 nibble-split path) with every zero-point
# mode, mixed with narrower widths, and on the fp32 SIMT path; scales sized so
# that fp16 outputs stay in range with codes up to +-255 from the centre.
# 1-bit codes likewise.
WIDTH_CASES.update({
    "w88_B32_sym_f16": dict(bits1=8, bits2=8, B=32, dtype="f16", T=12, scale_lo=0.0005, scale_hi=0.002),
    "w88_B128_sym_bf16": dict(bits1=8, bits2=8, B=128, dtype="bf16", T=12, scale_lo=0.0005, scale_hi=0.002),
    "w84_B64_uint8_bf16": dict(bits1=8, bits2=4, B=64, zp_mode="uint8", zp_lo=0, zp_hi=15, dtype="bf16",
                               T=12, scale_lo=0.0005, scale_hi=0.002),
    "w88_B32_uint8_far_bf16": dict(bits1=8, bits2=8, B=32, zp_mode="uint8", zp_lo=20, zp_hi=240,
                                   dtype="bf16", T=12, scale_lo=0.0005, scale_hi=0.002),
    "w28_B64_offset_half_f16": dict(bits1=2, bits2=8, B=64, zp_mode="offset", zp_offset=1.5, dtype="f16",
                                    T=12, scale_lo=0.01, scale_hi=0.03),
    "w48_B32_offset_int_bf16": dict(bits1=4, bits2=8, B=32, zp_mode="offset", zp_offset=3.0,
                                    dtype="bf16", T=12, scale_lo=0.002, scale_hi=0.006),
    # 1-bit codes (centre 1)
    "w11_B32_sym_bf16": dict(bits1=1, bits2=1, B=32, dtype="bf16", T=12, scale_lo=0.05, scale_hi=0.2),
    "w12_B64_offset_f16": dict(bits1=1, bits2=2, B=64, zp_mode="offset", zp_offset=0.5, dtype="f16", T=12,
                               scale_lo=0.05, scale_hi=0.2),
    "w41_B128_uint8_bf16": dict(bits1=4, bits2=1, B=128, zp_mode="uint8", zp_lo=0, zp_hi=1, dtype="bf16",
                                T=12, scale_lo=0.005, scale_hi=0.02),
    "w18_B32_sym_f16": dict(bits1=1, bits2=8, B=32, dtype="f16", T=12, scale_lo=0.05, scale_hi=0.1),
    "w11_B64_sym_f32": dict(bits1=1, bits2=1, B=64, dtype="f32", T=9, scale_lo=0.05, scale_hi=0.2),
    "w88_B64_uint8_f32": dict(bits1=8, bits2=8, B=64, zp_mode="uint8", zp_lo=90, zp_hi=170, dtype="f32",
                              T=9, scale_lo=0.0005, scale_hi=0.002),
})


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("name", list(WIDTH_CASES))
def test_width_matrix_parity(qm, name, path):
    cfg = BASE.with_(**WIDTH_CASES[name])
    inp = make_inputs(cfg)
    layer, out = run_layer(qm, inp, path=path)
    check_routing(layer, inp, path=path)
    check_out(out, O.forward(inp), cfg.dtype)


# The block-size-32 ("two scales per 64-deep step") int2 and mixed int2/int4
# decode of the "fast INT3" PR's tests: widths (2,2), (2,4), (4,2), 1, 4 and
# 64 token rows, top-10 routing, on both projection paths.
@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("T", [1, 4, 64])
@pytest.mark.parametrize("widths", [(2, 2), (2, 4), (4, 2)])
def test_block32_int2_decode_parity(qm, widths, T, path):
    cfg = BASE.with_(bits1=widths[0], bits2=widths[1], B=32, E=64, k=10, T=T, H=256, I=256,
                     scale_lo=0.02, scale_hi=0.08)
    inp = make_inputs(cfg)
    layer, out = run_layer(qm, inp, path=path)
    check_routing(layer, inp, path=path)
    check_out(out, O.forward(inp), cfg.dtype)


@pytest.mark.parametrize("name", list(VARIANTS))
def test_variant_parity(qm, name):
    cfg = BASE.with_(**VARIANTS[name])
    inp = make_inputs(cfg)
    layer, out = run_layer(qm, inp)
    check_routing(layer, inp)
    check_out(out, O.forward(inp), cfg.dtype)


# More than 1024 routes with k <= 32 past the single-CTA sizes (T > 64): the
# grouping is spread over the routing CTAs (per-CTA counts and stable ranks,
# one prefix CTA, a scatter kernel).
SPREAD = {
    "R1032_just_past": dict(T=129, E=8, k=8),
    "E3_many_ranges": dict(T=400, E=3, k=3),
    "E1024_k32": dict(T=72, E=1024, k=32, H=64, I=64),
    "ragged_last_cta_T1001": dict(T=1001, E=64, k=8),
}


@pytest.mark.parametrize("name", sorted(SPREAD))
def test_spread_grouping_parity(qm, name):
    cfg = BASE.with_(**SPREAD[name])
    inp = make_inputs(cfg)
    layer, out = run_layer(qm, inp, path="gemm")
    check_routing(layer, inp, path="gemm")
    check_out(out, O.forward(inp), cfg.dtype)


def test_all_tokens_on_one_expert_and_empty_experts(qm):
    cfg = BASE.with_(T=40, k=2, E=8)
    inp = make_inputs(cfg)
    logits = inp["logits"].clone()
    logits[:, 3] += 50.0          # every token picks expert 3 first
    logits[:, 5] += 40.0          # ... and expert 5 second; the others stay empty
    inp["logits"] = logits
    layer, out = run_layer(qm, inp)
    rt = check_routing(layer, inp)
    assert rt["counts"][3] == 40 and rt["counts"][5] == 40 and rt["counts"].sum() == 80
    check_out(out, O.forward(inp), cfg.dtype)


def test_tied_logits_lowest_index_wins(qm):
    cfg = BASE.with_(T=16, E=8, k=3)
    inp = make_inputs(cfg)
    lg = np.zeros((16, 8), np.float32)
    lg[:, ::2] = -0.0            # -0.0 ranks below +0.0
    lg[3] = 1.0
    inp["logits"] = torch.from_numpy(lg)
    layer, out = run_layer(qm, inp)
    rt = check_routing(layer, inp)
    assert list(rt["ids"][0]) == [1, 3, 5]
    check_out(out, O.forward(inp), cfg.dtype)


def test_zero_tokens_and_growth(qm):
    cfg = BASE.with_(T=6)
    inp = make_inputs(cfg)
    layer = qm.QMoELayer.from_config(cfg)
    layer.reserve(2)
    x, logits = qm.load_inputs(layer, inp)
    empty = torch.empty((0, cfg.H), dtype=x.dtype, device="cuda")
    layer.forward(empty, logits[:0])                 # no work, no error
    out = layer.forward(x, logits)                   # grows past the reservation
    torch.cuda.synchronize()
    check_out(out, O.forward(inp), cfg.dtype)


@pytest.mark.parametrize("path", sorted(PATHS))
def test_graph_capture_replay_matches_eager(qm, path):
    cfg = CONFIGS["decode_int2"]
    inp = make_inputs(cfg)
    layer = qm.QMoELayer.from_config(cfg)
    layer.set_fused_decode(PATHS[path][0])
    layer.set_gemm_min_rows(PATHS[path][1])
    layer.reserve(cfg.T)
    x, logits = qm.load_inputs(layer, inp)
    eager = layer.forward(x, logits).clone()
    out = torch.empty_like(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(x, logits, out, stream=s)      # warm on the capture stream
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.forward(x, logits, out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    if path != "gemm":
        assert torch.equal(out, eager)               # slot-ordered combine: bitwise deterministic
    else:
        # fp32 reductions into the combine accumulator: the order of the k
        # slot additions may differ run to run (a last-bit difference at most
        # after rounding to D).
        torch.testing.assert_close(out.float(), eager.float(), rtol=1e-2, atol=1e-2)
    check_out(out, O.forward(inp), cfg.dtype)


def test_capture_beyond_reservation_is_refused(qm):
    cfg = BASE.with_(T=8)
    inp = make_inputs(cfg)
    layer = qm.QMoELayer.from_config(cfg)
    layer.reserve(4)
    x, logits = qm.load_inputs(layer, inp)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with pytest.raises(qm.QMoEError) as ei:
        with torch.cuda.graph(g, stream=s):
            layer.forward(x, logits, stream=s)
    assert ei.value.status == qm.QMOE_ERR_STATE


@pytest.mark.parametrize("path", sorted(PATHS))
def test_forward_host_matches_device(qm, path):
    cfg = CONFIGS["decode_many_expert_int4"]
    inp = make_inputs(cfg)
    layer = qm.QMoELayer.from_config(cfg)
    layer.set_fused_decode(PATHS[path][0])
    layer.set_gemm_min_rows(PATHS[path][1])
    layer.reserve(cfg.T)
    x, logits = qm.load_inputs(layer, inp)
    dev = layer.forward(x, logits)
    xh = inp["x"].pin_memory()
    lh = inp["logits"].pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    layer.forward_host(xh, lh, oh)
    torch.cuda.synchronize()
    if path != "gemm":
        assert torch.equal(oh, dev.cpu())            # slot-ordered combine: bitwise deterministic
    else:
        # fp32 reductions into the combine accumulator: slot order may differ
        torch.testing.assert_close(oh.float(), dev.cpu().float(), rtol=1e-2, atol=1e-2)
    check_out(oh, O.forward(inp), cfg.dtype)


@pytest.mark.parametrize("path", sorted(PATHS))
def test_bounded_wait_reports_timeout_and_context_survives(qm, path):
    # Host-injected failure: the first copy stage of every decode warp (or of
    # every grouped-GEMM CTA) is armed but never issued, so the bounded waits
    # on it run out; in the single launch every fc2 item waits on a flag that
    # nothing sets.  The kernel records QMOE_ERR_TIMEOUT, drains its real
    # copies and returns; the context stays usable and the next forward is
    # correct.
    cfg = BASE.with_(T=4)
    inp = make_inputs(cfg)
    layer = qm.QMoELayer.from_config(cfg)
    layer.set_fused_decode(PATHS[path][0])
    layer.set_gemm_min_rows(PATHS[path][1])
    x, logits = qm.load_inputs(layer, inp)
    layer.set_wait_limit(2000)
    layer.inject_stall(True)
    layer.forward(x, logits)
    torch.cuda.synchronize()
    assert layer.poll() == qm.QMOE_ERR_TIMEOUT
    layer.inject_stall(False)
    layer.set_wait_limit(0)                          # back to the default
    out = layer.forward(x, logits)
    torch.cuda.synchronize()
    assert layer.poll() == 0
    check_out(out, O.forward(inp), cfg.dtype)


def test_trace_events_bracket_stages(qm):
    cfg = CONFIGS["decode_int2"]
    inp = make_inputs(cfg)
    layer = qm.QMoELayer.from_config(cfg)
    x, logits = qm.load_inputs(layer, inp)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(qm.QMOE_TRACE_NUM_EVENTS)]
    layer.set_trace_events(ev)
    layer.forward(x, logits)
    torch.cuda.synchronize()
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(len(ev) - 1)]
    assert all(t >= 0 for t in times)
    layer.set_trace_events(None)


def test_automatic_combine_is_ordered_at_decode_sizes(qm):
    # The default combine mode (QMOE_COMBINE_AUTO) adds the slots in order for
    # forwards of <= 64 tokens on the tensor-core path too: two forwards agree
    # bit for bit; an unknown mode is refused.
    cfg = BASE.with_(T=48, E=16, k=4)
    inp = make_inputs(cfg)
    layer = qm.QMoELayer.from_config(cfg)
    layer.set_fused_decode(0)
    x, logits = qm.load_inputs(layer, inp)
    out1 = layer.forward(x, logits).clone()
    out2 = layer.forward(x, logits)
    torch.cuda.synchronize()
    assert layer.poll() == 0
    assert torch.equal(out1, out2)
    check_out(out1, O.forward(inp), cfg.dtype)
    with pytest.raises(qm.QMoEError):
        layer.set_deterministic(3)


@pytest.mark.parametrize("min_rows", [0, 24])
def test_deterministic_gemm_combine(qm, min_rows):
    # qmoe_set_deterministic: the fc2 GEMM writes y rows and the k slots are
    # added in order [qmoe.rs qmoe_combine_impl] instead of fp32 reductions;
    # with min_rows = 24 the forward mixes decode-class and GEMM-class experts.
    cfg = BASE.with_(T=200, E=16, k=2, zipf_bias=1.5)
    inp = make_inputs(cfg)
    layer = qm.QMoELayer.from_config(cfg)
    layer.set_fused_decode(0)
    layer.set_gemm_min_rows(min_rows)
    layer.set_deterministic(1)
    x, logits = qm.load_inputs(layer, inp)
    out1 = layer.forward(x, logits).clone()
    out2 = layer.forward(x, logits)
    torch.cuda.synchronize()
    assert layer.poll() == 0
    assert torch.equal(out1, out2)
    check_routing(layer, inp, path=separate_path(min_rows))
    check_out(out1, O.forward(inp), cfg.dtype)
