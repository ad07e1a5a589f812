"""Host-side tests of the C-ABI library (no GPU needed): it loads, exports
every function include/qmoe.h declares, and validates arguments before any
device work."""
import ctypes

import pytest

from weight_only_quantized_qmoe_gb300 import binding as b


@pytest.fixture(scope="module")
def lib():
    from weight_only_quantized_qmoe_gb300 import build
    build.build()
    return b.load()


def test_exports_every_declared_function(lib):
    names = b.header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(b._SIGS), "binding and header disagree"


def _create(**kw):
    args = dict(hidden=256, inter=128, experts=8, top_k=2, bits_fc1=4, bits_fc2=4, block_size=64,
                zp_mode=b.QMOE_ZP_SYMMETRIC, activation=b.QMOE_ACT_SWIGLU, dtype=b.QMOE_BF16)
    args.update(kw)
    return b.qmoe_create(**args)


def test_create_validates(lib):
    st, h = _create()
    assert st == b.QMOE_OK and h
    b.qmoe_destroy(h)
    for act in (b.QMOE_ACT_RELU, b.QMOE_ACT_GELU_TANH, b.QMOE_ACT_SILU, b.QMOE_ACT_IDENTITY):
        st, h = _create(activation=act)
        assert st == b.QMOE_OK and h, act
        # the fc1 row layouts are for gated activations only (silu beside a
        # separate fc3 is the gated form)
        assert b.qmoe_set_fc1_layout(h, b.QMOE_FC1_INTERLEAVED) == b.QMOE_ERR_INVALID_ARG
        want = b.QMOE_OK if act == b.QMOE_ACT_SILU else b.QMOE_ERR_INVALID_ARG
        assert b.qmoe_set_fc1_layout(h, b.QMOE_FC1_SEPARATE_FC3) == want
        assert b.qmoe_set_fc1_layout(h, b.QMOE_FC1_CONCAT) == b.QMOE_OK
        b.qmoe_destroy(h)
    for widths in ((8, 8), (8, 2), (3, 8), (1, 1), (1, 4)):
        st, h = _create(bits_fc1=widths[0], bits_fc2=widths[1])
        assert st == b.QMOE_OK and h, widths
        b.qmoe_destroy(h)
    for kw, want in [
        (dict(bits_fc1=5), b.QMOE_ERR_UNSUPPORTED),
        (dict(bits_fc2=7), b.QMOE_ERR_UNSUPPORTED),
        (dict(bits_fc1=0), b.QMOE_ERR_UNSUPPORTED),
        (dict(bits_fc2=6), b.QMOE_ERR_UNSUPPORTED),
        (dict(block_size=16), b.QMOE_ERR_UNSUPPORTED),
        (dict(top_k=9), b.QMOE_ERR_INVALID_ARG),
        (dict(top_k=0), b.QMOE_ERR_INVALID_ARG),
        (dict(hidden=200), b.QMOE_ERR_INVALID_ARG),
        (dict(inter=96, block_size=64), b.QMOE_ERR_INVALID_ARG),
        (dict(experts=2000, top_k=2), b.QMOE_ERR_UNSUPPORTED),
        (dict(zp_mode=7), b.QMOE_ERR_INVALID_ARG),
        (dict(activation=6), b.QMOE_ERR_INVALID_ARG),
        (dict(activation=-1), b.QMOE_ERR_INVALID_ARG),
        (dict(dtype=9), b.QMOE_ERR_INVALID_ARG),
    ]:
        st, h = _create(**kw)
        assert st == want, (kw, st)
        assert not h


def test_zero_point_offset_rules(lib):
    st, h = _create(zp_mode=b.QMOE_ZP_OFFSET, bits_fc1=2, bits_fc2=2, dtype=b.QMOE_F16)
    assert st == b.QMOE_OK
    assert b.qmoe_set_zero_point_offset(h, 1.5) == b.QMOE_OK
    assert b.qmoe_set_zero_point_offset(h, 1.3) == b.QMOE_ERR_UNSUPPORTED
    assert "requantize" in b.qmoe_last_error(h)
    assert b.qmoe_set_zero_point_offset(h, float("nan")) == b.QMOE_ERR_INVALID_ARG
    b.qmoe_destroy(h)
    st, h = _create()
    assert b.qmoe_set_zero_point_offset(h, 1.5) == b.QMOE_ERR_STATE
    b.qmoe_destroy(h)


def test_prepack_and_forward_state_checks(lib):
    st, h = _create(zp_mode=b.QMOE_ZP_UINT8)
    # zero points required in uint8 mode; checked before any device call
    assert b.qmoe_prepack(h, 1, 16, 16, 0, 0) == b.QMOE_ERR_INVALID_ARG
    assert b.qmoe_prepack(h, 4, 16, 16, 16, 0) == b.QMOE_ERR_INVALID_ARG
    assert b.qmoe_prepack(h, 3, 16, 16, 16, 0) == b.QMOE_ERR_STATE       # fc3 needs separate projections
    assert b.qmoe_prepack(h, 1, 0, 16, 16, 0) == b.QMOE_ERR_INVALID_ARG
    # T == 0: no work, OK; T > 0 before prepack: STATE
    assert b.qmoe_forward(h, 16, 16, 16, 0, 0) == b.QMOE_OK
    assert b.qmoe_forward(h, 16, 16, 16, 4, 0) == b.QMOE_ERR_STATE
    assert b.qmoe_forward(h, 16, 16, 16, -1, 0) == b.QMOE_ERR_INVALID_ARG
    assert b.qmoe_get_routing(h, 0, 0, 0, 0, 0) == b.QMOE_ERR_STATE
    assert "prepack" in b.qmoe_last_error(h) or "forward" in b.qmoe_last_error(h)
    st, m = b.qmoe_get_worklist(h, 2, 0, 0, 0, 0)
    assert st == b.QMOE_ERR_INVALID_ARG
    assert b.qmoe_set_trace_events(h, [1, 2]) == b.QMOE_ERR_INVALID_ARG
    assert b.qmoe_set_gemm_min_rows(h, -1) == b.QMOE_ERR_INVALID_ARG
    assert b.qmoe_set_wait_limit(h, -1) == b.QMOE_ERR_INVALID_ARG
    b.qmoe_destroy(h)


def test_activation_layout_and_bias_argument_checks(lib):
    st, h = _create()
    inf = float("inf")
    assert b.qmoe_set_swiglu_params(h, 1.702, 1.0, 7.0) == b.QMOE_OK
    assert b.qmoe_set_swiglu_params(h, 1.0, 0.0, inf) == b.QMOE_OK         # the defaults
    assert b.qmoe_set_swiglu_params(h, float("nan"), 0.0, 1.0) == b.QMOE_ERR_INVALID_ARG
    assert b.qmoe_set_swiglu_params(h, 0.0, 0.0, 1.0) == b.QMOE_ERR_INVALID_ARG
    assert b.qmoe_set_swiglu_params(h, 1.0, inf, 1.0) == b.QMOE_ERR_INVALID_ARG
    assert b.qmoe_set_swiglu_params(h, 1.0, 0.0, 0.0) == b.QMOE_ERR_INVALID_ARG
    assert b.qmoe_set_swiglu_params(h, 1.0, 0.0, -1.0) == b.QMOE_ERR_INVALID_ARG
    assert b.qmoe_set_fc1_layout(h, 1) == b.QMOE_OK
    assert b.qmoe_set_fc1_layout(h, 0) == b.QMOE_OK
    assert b.qmoe_set_fc1_layout(h, 3) == b.QMOE_ERR_INVALID_ARG
    assert b.qmoe_set_fc1_layout(h, -1) == b.QMOE_ERR_INVALID_ARG
    assert b.qmoe_set_bias(h, 4, 16, 0) == b.QMOE_ERR_INVALID_ARG
    # fc3 exists only beside a separate-gate fc1 (checked before any device call)
    assert b.qmoe_set_bias(h, 3, 16, 0) == b.QMOE_ERR_STATE
    assert b.qmoe_prepack(h, 3, 16, 16, None, None) == b.QMOE_ERR_STATE
    assert b.qmoe_set_bias(h, 1, 0, 0) == b.QMOE_OK                       # removing none is fine
    assert b.qmoe_set_fc1_layout(h, b.QMOE_FC1_SEPARATE_FC3) == b.QMOE_OK
    assert b.qmoe_set_bias(h, 3, 0, 0) == b.QMOE_OK                       # removing none is fine
    b.qmoe_destroy(h)


def test_status_strings(lib):
    assert b.qmoe_status_string(b.QMOE_OK) == "QMOE_OK"
    assert b.qmoe_status_string(b.QMOE_ERR_TIMEOUT) == "QMOE_ERR_TIMEOUT"
    assert b.qmoe_status_string(99) == "QMOE_ERR_UNKNOWN"
    assert lib.qmoe_last_error(None) == b"null layer"


def test_worklist_capacity_bounds_item_count(lib):
    st, h = _create(experts=64, top_k=8)
    for T in (1, 8, 100, 4096):
        cap0 = b.qmoe_worklist_capacity(h, 0, T)
        cap1 = b.qmoe_worklist_capacity(h, 1, T)
        R = T * 8
        # every expert with rows contributes ceil(c / tb) <= c / tb + 1 items
        assert cap0 >= min(64, R) and cap1 >= min(64, R)
    assert b.qmoe_worklist_capacity(h, 2, 4) == -1
    b.qmoe_destroy(h)
