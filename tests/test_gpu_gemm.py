"""Parity of the tensor-core grouped GEMM path (tcgen05, A = dequantised
weights in TMEM, B = routed token rows) with the CPU oracle.  Setting the
GEMM threshold to 0 sends every expert with rows to it, so small shapes cover
the variant matrix (with the single-launch decode forward switched off); the
prefill workload runs at full size in test_gpu_parity.py."""
import numpy as np
import pytest
import torch

from oracle import qmoe_oracle as O
from qmoe_inputs import CONFIGS, make_inputs
from test_gpu_parity import check_out, check_routing, run_layer, separate_path

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qm():
    from weight_only_quantized_qmoe_gb300 import build
    build.build()
    import weight_only_quantized_qmoe_gb300 as q
    return q


BASE = CONFIGS["tiny"].with_(H=256, I=128, E=8, k=2, dtype="bf16", B=32, T=24)

GEMM_VARIANTS = {
    "int4_sym_bf16_B32": dict(),
    "int4_sym_f16_B128": dict(dtype="f16", B=128),
    "int4_uint8_B64": dict(zp_mode="uint8", zp_lo=6, zp_hi=9, B=64),
    "int2_offset_geglu_f16_B128": dict(bits1=2, bits2=2, zp_mode="offset", zp_offset=1.5,
                                       dtype="f16", act="geglu", B=128),
    "int2_K_fold_regression": dict(bits1=2, bits2=2, H=1024, I=512, B=64, T=20),
    "int3_sym_B32": dict(bits1=3, bits2=3),
    "int3_uint8_int4": dict(bits1=3, bits2=4, zp_mode="uint8", zp_lo=0, zp_hi=7),
    "odd_tiles_H96_I96": dict(H=96, I=96, B=32, T=30),
    "rows_over_256": dict(E=2, k=1, T=300),
    "many_experts": dict(E=64, k=6, T=50),
}


@pytest.mark.parametrize("name", list(GEMM_VARIANTS))
def test_gemm_variant_parity(qm, name):
    cfg = BASE.with_(**GEMM_VARIANTS[name])
    inp = make_inputs(cfg)
    layer, out = run_layer(qm, inp, path="gemm")
    check_routing(layer, inp, path="gemm")
    items, m_tile = layer.worklist(1, cfg.T)
    assert m_tile == 128 and len(items) > 0
    check_out(out, O.forward(inp), cfg.dtype)


def test_gemm_and_decode_classes_agree(qm):
    # The same forward through the decode kernel only and the GEMM only.
    cfg = BASE.with_(T=48, E=4, k=2)
    inp = make_inputs(cfg)
    _, out_dec = run_layer(qm, inp, path="decode")
    _, out_gemm = run_layer(qm, inp, path="gemm")
    ref = O.forward(inp)
    check_out(out_dec, ref, cfg.dtype)
    check_out(out_gemm, ref, cfg.dtype)


def test_mixed_classes_in_one_forward(qm):
    # Skewed routing: some experts above, some below the threshold.
    cfg = BASE.with_(T=200, E=16, k=2, zipf_bias=1.5)
    inp = make_inputs(cfg)
    layer, out = run_layer(qm, inp, path=separate_path(24))
    rt = check_routing(layer, inp, path=separate_path(24))
    assert (rt["counts"] > 24).any() and ((rt["counts"] > 0) & (rt["counts"] <= 24)).any()
    check_out(out, O.forward(inp), cfg.dtype)
