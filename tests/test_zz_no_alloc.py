"""qmoe_forward_noalloc: the forward for callers that may not allocate device
memory when they run the layer (allocation-free graph capture, a framework
allocator that owns the whole device, fixed memory plans).  Its workspace is
the library's static scratch array, so it must give the same result as
qmoe_forward, call after call, and refuse sizes the array cannot hold.

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
    for call in range(2):                                   # the array keeps old contents
        out = torch.full_like(x, float("nan"))
        assert _noalloc(qm, layer, x, logits, out) == qm.QMOE_OK, qm.qmoe_last_error(layer.handle)
        torch.cuda.synchronize()
        err = np.abs(out.float().cpu().numpy().astype(np.float64) - ref64).max()
        assert err <= tol, f"call {call}: max|err| {err:.3e} > {tol:.3e}"
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
