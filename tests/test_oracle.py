"""Pins for the CPU oracle, each against something other than the oracle itself:
values the pages print, library routines, brute force on tiny inputs,
invariants, and planted mistakes that a pin must catch."""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import qmoe_oracle as O
from qmoe_inputs import CONFIGS, make_inputs, pack_fields

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.split() for l in f if l.strip() and not l.startswith("#")]


# ---------------------------------------------------------------------------
# Rounding into D
# ---------------------------------------------------------------------------
def test_round_f16_matches_numpy_cast():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(200000) * np.exp2(rng.integers(-30, 17, 200000))
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(O.round_to_dtype(x, "f16"), ref)


def test_round_f32_matches_numpy_cast():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(200000) * np.exp2(rng.integers(-140, 100, 200000))
    ref = x.astype(np.float32).astype(np.float64)
    np.testing.assert_array_equal(O.round_to_dtype(x, "f32"), ref)


def test_round_bf16_matches_torch_cast_of_f32():
    # torch rounds f32 -> bf16 to nearest even; for f32 inputs that is a
    # single rounding, so it pins the bf16 path.
    rng = np.random.default_rng(2)
    x32 = (rng.standard_normal(200000) * np.exp2(rng.integers(-130, 60, 200000))).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(O.round_to_dtype(x32.astype(np.float64), "bf16"), ref)


def test_round_ties_to_even():
    # bf16 keeps 8 significant bits: 1 + 2^-8 is a tie between 1 and 1 + 2^-7.
    assert O.round_to_dtype(1 + 2.0 ** -8, "bf16") == 1.0
    assert O.round_to_dtype(1 + 3 * 2.0 ** -8, "bf16") == 1 + 2 * 2.0 ** -7
    assert O.round_to_dtype(1 + 2.0 ** -11, "f16") == 1.0
    assert O.round_to_dtype(-(1 + 3 * 2.0 ** -11), "f16") == -(1 + 2.0 ** -9)
    assert O.round_to_dtype(65520.0, "f16") == np.inf       # overflow tie -> inf
    assert O.round_to_dtype(2.0 ** -25, "f16") == 0.0        # half of min subnormal
    assert O.round_to_dtype(3 * 2.0 ** -26, "f16") == 2.0 ** -24


# ---------------------------------------------------------------------------
# Routing
# ---------------------------------------------------------------------------
def _brute_select(row, k):
    # Sort by value descending; +0.0 ranks above -0.0; ties to lower index.
    items = sorted(range(len(row)),
                   key=lambda e: (-float(row[e]), math.copysign(1.0, float(row[e])) < 0, e))
    return items[:k]


def test_selection_brute_force_with_ties_and_zeros():
    rng = np.random.default_rng(3)
    for trial in range(300):
        E = int(rng.integers(1, 12))
        k = int(rng.integers(1, E + 1))
        T = 5
        vals = np.array([0.0, -0.0, 1.0, -1.0, 0.5, 2.5, -3.0, 1e-30, -1e-30], np.float32)
        logits = rng.choice(vals, size=(T, E)).astype(np.float32)
        ids = O.select_experts(logits, k)
        for t in range(T):
            assert list(ids[t]) == _brute_select(logits[t], k), (logits[t], k)


def test_selection_k_equals_E_is_full_key_order():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((7, 9)).astype(np.float32)
    ids = O.select_experts(logits, 9)
    for t in range(7):
        assert sorted(ids[t]) == list(range(9))
        assert list(ids[t]) == list(np.argsort(-logits[t].astype(np.float64), kind="stable"))


def test_weights_renormalised_sum_to_one_and_softmax():
    rng = np.random.default_rng(5)
    logits = (rng.standard_normal((64, 32)) * 3).astype(np.float32)
    ids = O.select_experts(logits, 4)
    w = O.routing_weights(logits, ids, True)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    sm = scipy.special.softmax(logits.astype(np.float64), axis=1)
    w_all = O.routing_weights(logits, ids, False)
    np.testing.assert_allclose(w_all, np.take_along_axis(sm, ids.astype(np.int64), 1), rtol=1e-14)
    sel = np.take_along_axis(sm, ids.astype(np.int64), 1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-14)
    w1 = O.routing_weights(logits, O.select_experts(logits, 1), True)
    np.testing.assert_array_equal(w1, 1.0)


def test_group_matches_stable_argsort():
    rng = np.random.default_rng(6)
    for E, R in [(4, 8), (128, 256), (64, 32768), (8, 1), (3, 0)]:
        ids = rng.integers(0, E, size=R)
        counts, offsets, perm, pos = O.group_routes(ids, E)
        np.testing.assert_array_equal(counts, np.bincount(ids, minlength=E))
        assert offsets[0] == 0 and offsets[-1] == R
        np.testing.assert_array_equal(np.diff(offsets), counts)
        np.testing.assert_array_equal(perm, np.argsort(ids, kind="stable"))
        np.testing.assert_array_equal(np.sort(perm), np.arange(R))
        np.testing.assert_array_equal(perm[pos], np.arange(R))
        assert np.all(np.diff(ids[perm]) >= 0) if R else True


def test_worklist_order_and_count():
    offsets = np.array([0, 300, 300, 301, 557])
    items = O.build_worklist(offsets, 128, 3)
    counts = np.diff(offsets)
    assert len(items) == sum(-(-c // 128) * 3 for c in counts)
    # brute-force enumeration
    ref = []
    for e in range(4):
        for m in range(-(-counts[e] // 128)):
            for n in range(3):
                ref.append((e, int(offsets[e]) + 128 * m, int(min(128, counts[e] - 128 * m)), n))
    assert items == ref


# ---------------------------------------------------------------------------
# Unpacking / dequantisation
# ---------------------------------------------------------------------------
def test_unpack_hand_cases():
    for bits, hexbytes, *codes in _rows("packed_bytes.txt"):
        bits = int(bits)
        raw = np.frombuffer(bytes.fromhex(hexbytes), np.uint8)
        got = O.unpack_fields(raw, bits, len(codes))
        assert list(got) == [int(c) for c in codes]


def test_unpack_int3_straddles_bytes():
    codes = [1, 2, 3, 4, 5, 6, 7, 0, 5, 3, 6, 7, 1, 0, 2, 4]
    stream = sum(c << (3 * i) for i, c in enumerate(codes))
    raw = np.frombuffer(stream.to_bytes(6, "little"), np.uint8)
    assert list(O.unpack_fields(raw, 3, 16)) == codes


def test_pack_unpack_roundtrip():
    rng = np.random.default_rng(7)
    for bits in (1, 2, 3, 4, 8):
        vals = rng.integers(0, 1 << bits, size=(5, 96))
        np.testing.assert_array_equal(O.unpack_fields(pack_fields(vals, bits), bits, 96), vals)


def test_dequant_fractional_offset_golden():
    for bits, off, code, mult in _rows("zero_point_offset_int2.txt"):
        bits, off, code, mult = int(bits), float(off), int(code), float(mult)
        s = 0.03125
        row = pack_fields(np.array([[code] * 32]), bits)
        W = O.dequantize(row, np.array([[s]]), bits, 32, 32, "f32", "offset", zp_offset=off)
        np.testing.assert_array_equal(W, mult * s)


def test_dequant_symmetric_golden():
    for bits, code, mult in _rows("symmetric_centre.txt"):
        bits, code, mult = int(bits), int(code), float(mult)
        s = 0.0078125
        row = pack_fields(np.array([[code] * 32]), bits)
        W = O.dequantize(row, np.array([[s]]), bits, 32, 32, "bf16", "sym")
        np.testing.assert_array_equal(W, mult * s)


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8])
def test_zero_point_modes_agree_at_the_centre(bits):
    rng = np.random.default_rng(8 + bits)
    N, K, B = 6, 128, 32
    codes = rng.integers(0, 256, size=(N, K * bits // 8), dtype=np.uint8)
    scales = torch.from_numpy(rng.uniform(0.005, 0.02, (N, K // B)).astype(np.float32)).to(torch.bfloat16).double().numpy()
    centre = 1 << (bits - 1)
    zp = pack_fields(np.full((N, K // B), centre), bits)
    a = O.dequantize(codes, scales, bits, B, K, "bf16", "sym")
    b = O.dequantize(codes, scales, bits, B, K, "bf16", "uint8", zp_packed=zp)
    c = O.dequantize(codes, scales, bits, B, K, "bf16", "offset", zp_offset=float(centre))
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, c)


def test_dequant_block_indexing_and_rounding():
    # Per-block scale/zero point: weight d uses block d // B; the product is
    # rounded once into D.
    rng = np.random.default_rng(9)
    N, K, B, bits = 3, 128, 32, 4
    q = rng.integers(0, 16, size=(N, K))
    z = rng.integers(6, 10, size=(N, K // B))
    s32 = rng.uniform(0.005, 0.02, (N, K // B)).astype(np.float32)
    s = torch.from_numpy(s32).to(torch.bfloat16).double().numpy()
    W = O.dequantize(pack_fields(q, bits), s, bits, B, K, "bf16", "uint8", zp_packed=pack_fields(z, bits))
    for n in range(N):
        for d in range(K):
            exact = (q[n, d] - z[n, d // B]) * s[n, d // B]
            ref = float(torch.tensor(exact, dtype=torch.float32).to(torch.bfloat16))
            assert W[n, d] == ref


def test_swiglu_attributes_match_a_torch_restatement():
    # g' sigmoid(alpha g') == silu(alpha g') / alpha, computed by torch
    g = torch.linspace(-9, 9, 181, dtype=torch.float64)[:, None]
    u = torch.linspace(-5, 5, 41, dtype=torch.float64)[None, :]
    for alpha, beta, limit in [(1.0, 0.0, float("inf")), (1.702, 1.0, 7.0), (0.5, -0.25, 1.5), (3.0, 2.0, 0.1)]:
        gb = torch.clamp(g, max=limit)
        ref = torch.nn.functional.silu(alpha * gb) / alpha * (torch.clamp(u, -limit, limit) + beta)
        np.testing.assert_allclose(O.swiglu(g.numpy(), u.numpy(), alpha, beta, limit), ref.numpy(),
                                   rtol=1e-13, atol=1e-300)
    # attribute defaults: plain silu(g) * u
    np.testing.assert_allclose(O.swiglu(g.numpy(), u.numpy()),
                               (torch.nn.functional.silu(g) * u).numpy(), rtol=1e-15, atol=1e-300)


def test_interleaved_layout_is_a_row_permutation_of_concat():
    # Interleaved rows (2f = gate f, 2f+1 = up f) moved to [gate | up] give the
    # same layer.
    cfg = CONFIGS["tiny"].with_(fc1_layout="interleaved", bias=True, H=64, I=32, E=3, k=2)
    inp = make_inputs(cfg)
    order = np.concatenate([np.arange(0, 64, 2), np.arange(1, 64, 2)])
    cat = dict(inp)
    cat["cfg"] = cfg.with_(fc1_layout="concat")
    for key in ("fc1_codes", "fc1_scales", "fc1_bias"):
        cat[key] = inp[key][:, order]
    np.testing.assert_array_equal(O.forward(inp), O.forward(cat))


def test_non_gated_activations_match_torch():
    # qmoe.rs qmoe_activate: relu, tanh-GELU, silu, identity
    v = np.linspace(-8, 8, 161)
    tv = torch.from_numpy(v)
    np.testing.assert_allclose(O.act_single(v, "relu"), torch.relu(tv).numpy(), rtol=0, atol=0)
    np.testing.assert_allclose(O.act_single(v, "gelu"),
                               torch.nn.functional.gelu(tv, approximate="tanh").numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(O.act_single(v, "silu"), torch.nn.functional.silu(tv).numpy(), rtol=1e-13,
                               atol=1e-15)
    np.testing.assert_array_equal(O.act_single(v, "identity"), v)


def test_activations_match_torch():
    g = torch.linspace(-12, 12, 2001, dtype=torch.float64)
    np.testing.assert_allclose(O.silu(g.numpy()), torch.nn.functional.silu(g).numpy(), rtol=1e-15, atol=1e-300)
    np.testing.assert_allclose(O.gelu_tanh(g.numpy()),
                               torch.nn.functional.gelu(g, approximate="tanh").numpy(),
                               rtol=1e-12, atol=1e-15)   # 1 + tanh(z) cancels for z << 0


# ---------------------------------------------------------------------------
# Whole layer against an independent brute force
# ---------------------------------------------------------------------------
def _bf_round(v, dtype):
    if dtype == "f32":
        return float(np.float32(v))
    if dtype == "f16":
        return float(np.float16(v))
    return float(torch.tensor(v, dtype=torch.float64).to(torch.float32).to(torch.bfloat16))


def _brute_layer(inp):
    """Independent restatement: Python integers for the bit streams, sorted()
    for the selection, math.exp for the softmax, explicit loops for the dots."""
    cfg = inp["cfg"]
    x = inp["x"].double().tolist()
    logits = inp["logits"].tolist()

    def weight(fc, e, n, d):
        bits, K = (cfg.bits2, cfg.I) if fc == 2 else (cfg.bits1, cfg.H)
        pre = f"fc{fc}_"
        if fc == 1 and cfg.fc1_layout == "separate" and n >= cfg.I:
            pre, n = "fc3_", n - cfg.I     # the up rows live in fc3
        row = bytes(inp[pre + "codes"][e, n].numpy())
        q = (int.from_bytes(row, "little") >> (d * bits)) & ((1 << bits) - 1)
        blk = d // cfg.B
        if cfg.zp_mode == "sym":
            z = float(1 << (bits - 1))
        elif cfg.zp_mode == "offset":
            z = cfg.zp_offset
        else:
            zrow = bytes(inp[pre + "zp"][e, n].numpy())
            z = float((int.from_bytes(zrow, "little") >> (blk * bits)) & ((1 << bits) - 1))
        s = float(inp[pre + "scales"][e, n, blk].double())
        return _bf_round((q - z) * s, cfg.dtype)

    W1 = {}
    W2 = {}
    out = []
    for t in range(cfg.T):
        sel = _brute_select(np.float32(logits[t]), cfg.k)
        m = max(logits[t])
        p = [math.exp(l - m) for l in logits[t]]
        den = sum(p[e] for e in sel) if cfg.normalize else sum(p)
        acc = [0.0] * cfg.H
        for e in sel:
            if e not in W1:
                n1 = 2 * cfg.I if (cfg.act in ("swiglu", "geglu") or cfg.fc1_layout == "separate") else cfg.I
                W1[e] = [[weight(1, e, n, d) for d in range(cfg.H)] for n in range(n1)]
                W2[e] = [[weight(2, e, n, d) for d in range(cfg.I)] for n in range(cfg.H)]
            b1 = inp["fc1_bias"][e].tolist() if inp.get("fc1_bias") is not None else [0.0] * (2 * cfg.I)
            if cfg.fc1_layout == "separate":
                b3 = inp["fc3_bias"][e].tolist() if inp.get("fc3_bias") is not None else [0.0] * cfg.I
                b1 = (b1 if inp.get("fc1_bias") is not None else [0.0] * cfg.I) + b3
            b2 = inp["fc2_bias"][e].tolist() if inp.get("fc2_bias") is not None else [0.0] * cfg.H
            gated = cfg.act in ("swiglu", "geglu")
            n1 = 2 * cfg.I if (gated or cfg.fc1_layout == "separate") else cfg.I
            a = [sum(W1[e][n][d] * x[t][d] for d in range(cfg.H)) + b1[n] for n in range(n1)]
            h = []
            for n in range(cfg.I):
                if not gated and cfg.fc1_layout != "separate":
                    v = a[n]
                    h.append({"relu": max(v, 0.0), "identity": v, "silu": v / (1 + math.exp(-v)),
                              "gelu": 0.5 * v * (1 + math.tanh(math.sqrt(2 / math.pi) * (v + 0.044715 * v ** 3)))
                              }[cfg.act])
                    continue
                if cfg.fc1_layout == "interleaved":
                    g, u = a[2 * n], a[2 * n + 1]
                else:
                    g, u = a[n], a[cfg.I + n]
                if cfg.act in ("swiglu", "silu"):   # silu here only beside fc3 (gated)
                    L = cfg.swiglu_limit
                    g = min(g, L)
                    u = max(-L, min(L, u))
                    h.append(g / (1 + math.exp(-cfg.swiglu_alpha * g)) * (u + cfg.swiglu_beta))
                else:
                    h.append(0.5 * g * (1 + math.tanh(math.sqrt(2 / math.pi) * (g + 0.044715 * g ** 3))) * u)
            for mm in range(cfg.H):
                acc[mm] += p[e] / den * (sum(W2[e][mm][n] * h[n] for n in range(cfg.I)) + b2[mm])
        out.append([_bf_round(v, cfg.dtype) for v in acc])
    return np.array(out)


SMALL_VARIANTS = {
    "tiny": dict(),
    "geglu_offset_int2_f16": dict(act="geglu", bits1=2, bits2=2, zp_mode="offset", zp_offset=1.5,
                                  dtype="f16", H=64, I=64, B=64, scale_lo=0.01, scale_hi=0.05),
    "uint8_int4_bf16": dict(zp_mode="uint8", zp_lo=6, zp_hi=9, dtype="bf16", H=64, I=64, E=6, k=3),
    "int3_int4_unnorm": dict(bits1=3, bits2=4, normalize=False, dtype="bf16", H=64, I=64, E=5, k=2),
    "int3_uint8_int2": dict(bits1=3, bits2=2, zp_mode="uint8", zp_lo=0, zp_hi=3, dtype="bf16",
                            H=64, I=64, E=3, k=3),
    # qmoe.rs swiglu_fusion == 1 (interleaved gate/up), SwiGLU alpha / beta /
    # limit (the limit clamps a good share of the gates here), fp32 biases
    "interleaved_bias_swiglu_params": dict(fc1_layout="interleaved", bias=True, swiglu_alpha=1.702,
                                           swiglu_beta=1.0, swiglu_limit=0.3, dtype="bf16",
                                           H=64, I=64, E=4, k=2),
    "bias_geglu_f16": dict(act="geglu", bias=True, bits1=2, bits2=2, zp_mode="offset", zp_offset=1.5,
                           dtype="f16", H=64, I=64, B=64, scale_lo=0.01, scale_hi=0.05),
    # 8-bit codes with byte zero points away from the centre
    "int8_uint8_f16": dict(bits1=8, bits2=8, zp_mode="uint8", zp_lo=100, zp_hi=150, dtype="f16",
                           H=64, I=64, scale_lo=0.0005, scale_hi=0.002),
    # 1-bit codes (centre 1) with 1-bit zero points
    "int1_uint8_bf16": dict(bits1=1, bits2=1, zp_mode="uint8", zp_lo=0, zp_hi=1, dtype="bf16",
                            H=64, I=64, scale_lo=0.05, scale_hi=0.2),
    # non-gated activations: fc1 has I rows, h = act(fc1 output)
    "relu_bias_f16": dict(act="relu", bias=True, dtype="f16", H=64, I=64),
    "gelu_int3": dict(act="gelu", bits1=3, bits2=4, dtype="bf16", H=64, I=64, E=3, k=2),
    "silu_uint8": dict(act="silu", zp_mode="uint8", zp_lo=6, zp_hi=9, dtype="f32", H=64, I=64),
    "identity_offset_int2": dict(act="identity", bits1=2, bits2=2, zp_mode="offset", zp_offset=1.5,
                                 dtype="f16", H=64, I=64, B=64),
    # qmoe.rs uses_separate_gate: silu beside fc3 is the gated form
    "silu_fc3_params": dict(act="silu", fc1_layout="separate", swiglu_limit=0.5, bias=True, dtype="bf16",
                            H=64, I=64, E=3, k=2),
    # qmoe.rs unfused SwiGLU: gate rows in fc1, up rows in a separate fc3
    "separate_fc3_bias_uint8": dict(fc1_layout="separate", bias=True, zp_mode="uint8", zp_lo=6, zp_hi=9,
                                    dtype="bf16", H=64, I=64, E=4, k=2),
}


@pytest.mark.parametrize("variant", list(SMALL_VARIANTS))
def test_layer_matches_brute_force(variant):
    cfg = CONFIGS["tiny"].with_(**SMALL_VARIANTS[variant])
    inp = make_inputs(cfg)
    got = O.forward(inp)
    ref = _brute_layer(inp)
    # Both round once into D at the end; fp64 sums may differ in the last bit
    # before that rounding, so allow one ulp of D.
    ulp = {"f32": 2.0 ** -23, "f16": 2.0 ** -10, "bf16": 2.0 ** -7}[cfg.dtype]
    np.testing.assert_allclose(got, ref, rtol=ulp, atol=1e-30)
    assert np.abs(got).max() > 1e-3     # not trivially zero


def test_single_expert_is_dense_quantised_glu():
    cfg = CONFIGS["tiny"].with_(E=1, k=1, H=64, I=32)
    inp = make_inputs(cfg)
    W1 = O.expert_weights(inp, 1, 0)
    W2 = O.expert_weights(inp, 2, 0)
    x = inp["x"].double().numpy()
    a = x @ W1.T
    h = O.silu(a[:, :32]) * a[:, 32:]
    ref = O.round_to_dtype(h @ W2.T, "f32")
    np.testing.assert_array_equal(O.forward(inp), ref)


def test_identity_like_weights_route_the_input_through():
    # Codes chosen so that W1 = s*[I; I] (gate|up) and W2 = s*I; with
    # k = E = 1: out = R(s * silu(s*x) * s*x).
    cfg = CONFIGS["tiny"].with_(E=1, k=1, H=32, I=32, B=32, zp_mode="sym")
    inp = make_inputs(cfg)
    eye = np.eye(32, dtype=np.int64)
    q1 = np.concatenate([eye, eye]) + 8                # code 9 on the diagonal, 8 elsewhere
    inp["fc1_codes"] = torch.from_numpy(pack_fields(q1, 4)[None])
    inp["fc2_codes"] = torch.from_numpy(pack_fields(eye + 8, 4)[None])
    s = 0.5
    inp["fc1_scales"] = torch.full((1, 64, 1), s)
    inp["fc2_scales"] = torch.full((1, 32, 1), s)
    x = inp["x"].double().numpy()
    ref = O.round_to_dtype(s * (O.silu(s * x) * (s * x)), "f32")
    np.testing.assert_array_equal(O.forward(inp), ref)


def test_canonical_configs_generate_valid_inputs():
    for name in ("tiny", "decode_many_expert_int4"):
        cfg = CONFIGS[name]
        inp = make_inputs(cfg)
        assert inp["fc1_codes"].shape == (cfg.E, 2 * cfg.I, cfg.H * cfg.bits1 // 8)
        assert inp["fc2_codes"].shape == (cfg.E, cfg.H, cfg.I * cfg.bits2 // 8)
        if cfg.zp_mode == "uint8":
            z = O.unpack_fields(inp["fc1_zp"].numpy(), cfg.bits1, cfg.H // cfg.B)
            assert z.min() >= cfg.zp_lo and z.max() <= cfg.zp_hi


def test_prefill_routing_is_skewed():
    # The skewed workload must give a Zipf-like load: expert 0 busiest.
    cfg = CONFIGS["prefill_int4"].with_(T=512)
    logits = make_inputs(cfg.with_(H=128, I=128))["logits"].numpy()
    ids = O.select_experts(logits, cfg.k)
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    assert counts[0] == counts.max() and counts[0] > 0.9 * 512
    assert counts[-8:].sum() < counts[:8].sum() / 20


# ---------------------------------------------------------------------------
# Planted mistakes: each must be caught by one of the pins above.
# ---------------------------------------------------------------------------
def _layer_pin_fails(monkeypatch, name, fake):
    monkeypatch.setattr(O, name, fake)
    cfg = CONFIGS["tiny"].with_(**SMALL_VARIANTS["uint8_int4_bf16"])
    inp = make_inputs(cfg)
    got = O.forward(inp)
    ref = _brute_layer(inp)
    ulp = 2.0 ** -7
    return not np.allclose(got, ref, rtol=ulp, atol=1e-30)


def test_planted_swapped_gate_up_is_caught(monkeypatch):
    real = O.glu
    assert _layer_pin_fails(monkeypatch, "glu",
                            lambda a, inter, act, *r: real(np.concatenate([a[:, inter:], a[:, :inter]], 1),
                                                           inter, act, *r))


def _variant_pin_fails(monkeypatch, variant, name, fake):
    monkeypatch.setattr(O, name, fake)
    cfg = CONFIGS["tiny"].with_(**SMALL_VARIANTS[variant])
    inp = make_inputs(cfg)
    ulp = {"f32": 2.0 ** -23, "f16": 2.0 ** -10, "bf16": 2.0 ** -7}[cfg.dtype]
    return not np.allclose(O.forward(inp), _brute_layer(inp), rtol=ulp, atol=1e-30)


def test_planted_swapped_fc1_fc3_is_caught(monkeypatch):
    # gate from fc3 and up from fc1 instead of the other way round
    cfg = CONFIGS["tiny"].with_(fc1_layout="separate", H=64, I=64)
    inp = make_inputs(cfg)
    ref = _brute_layer(inp)
    swapped = dict(inp)
    for part in ("codes", "scales", "zp", "bias"):
        swapped["fc1_" + part], swapped["fc3_" + part] = inp["fc3_" + part], inp["fc1_" + part]
    assert np.abs(O.forward(swapped) - ref).max() > 1e-3


def test_planted_dropped_bias_is_caught(monkeypatch):
    assert _variant_pin_fails(monkeypatch, "interleaved_bias_swiglu_params", "projection_bias",
                              lambda inputs, fc, e: 0.0)


def test_planted_ignored_interleave_is_caught(monkeypatch):
    real = O.split_gate_up
    assert _variant_pin_fails(monkeypatch, "interleaved_bias_swiglu_params", "split_gate_up",
                              lambda a, inter, layout="concat": real(a, inter, "concat"))


def test_planted_ignored_limit_is_caught(monkeypatch):
    real = O.swiglu
    assert _variant_pin_fails(monkeypatch, "interleaved_bias_swiglu_params", "swiglu",
                              lambda g, u, alpha=1.0, beta=0.0, limit=float("inf"): real(g, u, alpha, beta))


def test_planted_wrong_zero_point_is_caught(monkeypatch):
    real = O.zero_points
    assert _layer_pin_fails(monkeypatch, "zero_points",
                            lambda *a, **k: real(*a, **k) - 1.0)


def test_planted_unrounded_weights_are_caught(monkeypatch):
    real = O.dequantize

    def fake(*a, **k):
        a = list(a)
        a[5] = "f32" if len(a) > 5 else a[5]
        return real(*a, **k)
    assert _layer_pin_fails(monkeypatch, "dequantize", fake)


def test_planted_transposed_selection_order_is_caught(monkeypatch):
    real = O.select_experts
    assert _layer_pin_fails(monkeypatch, "select_experts",
                            lambda l, k: real(-np.asarray(l, np.float32), k))
