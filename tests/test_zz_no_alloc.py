"""qmoe_forward_noalloc: the forward for callers that may not allocate device
memory when they run the layer (a runtime whose caching allocator owns the
whole device, a fixed memory plan decided before start-up).  Its workspace is
the library's static scratch array, so it must give qmoe_forward's result
(within the output tolerance) call after call, agree with the oracle, report
a bounded wait that ran out, and refuse sizes the array cannot hold.

This file is collected last on purpose: it runs after every other GPU test,
and also passes on its own in a fresh process."""
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


def _noalloc(qm, layer, x, logits, out):
    stream = torch.cuda.current_stream().cuda_stream
    return qm.binding.qmoe_forward_noalloc(layer.handle, x.data_ptr(), logits.data_ptr(),
                                           out.data_ptr(), x.shape[0], stream)


@pytest.mark.parametrize("cfg", [
    CONFIGS["decode_int2"],
    CONFIGS["decode_many_expert_int4"],
    CONFIGS["tiny"],                                        # fp32 activations
    CONFIGS["tiny"].with_(H=256, I=128, E=8, dtype="bf16", bits1=3, bits2=2, T=37),
], ids=["decode_int2", "many_expert_int4", "tiny_f32", "int3_int2_T37"])
def test_noalloc_matches_forward_on_two_calls(qm, cfg):
    inp = make_inputs(cfg)
    layer = qm.QMoELayer.from_config(cfg)
    x, logits = qm.load_inputs(layer, inp)
    ref = layer.forward(x, logits)
    torch.cuda.synchronize()
    ref64 = ref.float().cpu().numpy().astype(np.float64)
    tol = O.tolerance(cfg.dtype, np.abs(ref64).max())
    oracle = O.forward(inp)
    tol_o = O.tolerance(cfg.dtype, np.abs(oracle).max())
    for call in range(2):                                   # the array keeps old contents
        out = torch.full_like(x, float("nan"))
        assert _noalloc(qm, layer, x, logits, out) == qm.QMOE_OK, qm.qmoe_last_error(layer.handle)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        err = np.abs(got - ref64).max()
        assert err <= tol, f"call {call}: max|err| vs qmoe_forward {err:.3e} > {tol:.3e}"
        err_o = np.abs(got - oracle).max()
        assert err_o <= tol_o, f"call {call}: max|err| vs oracle {err_o:.3e} > {tol_o:.3e}"
    assert layer.poll() == 0
    layer.close()


def test_noalloc_reports_a_wait_that_ran_out(qm):
    # Host-injected failure (no GPU fault): the decode kernels arm their first
    # copy stage but never issue it, so the bounded waits run out.  The status
    # word in the static array stays set until a poll reads and clears it.
    cfg = CONFIGS["tiny"].with_(H=256, I=128, E=8, dtype="bf16", T=4)
    inp = make_inputs(cfg)
    layer = qm.QMoELayer.from_config(cfg)
    x, logits = qm.load_inputs(layer, inp)
    out = torch.empty_like(x)
    assert layer.poll() == 0
    layer.set_wait_limit(2000)
    layer.inject_stall(True)
    assert _noalloc(qm, layer, x, logits, out) == qm.QMOE_OK
    torch.cuda.synchronize()
    assert layer.poll() == qm.QMOE_ERR_TIMEOUT
    assert layer.poll() == 0                                # read and cleared
    layer.inject_stall(False)
    layer.set_wait_limit(0)
    assert _noalloc(qm, layer, x, logits, out) == qm.QMOE_OK
    torch.cuda.synchronize()
    assert layer.poll() == 0
    ref = O.forward(inp)
    err = np.abs(out.float().cpu().numpy().astype(np.float64) - ref).max()
    assert err <= O.tolerance(cfg.dtype, np.abs(ref).max())
    layer.close()


def test_noalloc_rejects_sizes_beyond_the_array(qm):
    cfg = CONFIGS["mixed_int3_int4"]                        # needs about 4.4 MB of scratch
    inp = make_inputs(cfg)
    layer = qm.QMoELayer.from_config(cfg)
    x, logits = qm.load_inputs(layer, inp)
    out = torch.empty_like(x)
    assert _noalloc(qm, layer, x, logits, out) == qm.QMOE_ERR_UNSUPPORTED
    msg = qm.qmoe_last_error(layer.handle)
    assert "scratch" in msg and "qmoe_forward" in msg
    assert _noalloc(qm, layer, x[:0], logits[:0], out) == qm.QMOE_OK   # no tokens, no work
    layer.close()
