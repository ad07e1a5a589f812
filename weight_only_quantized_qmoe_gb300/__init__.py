"""GB300 (sm_103a) weight-only block-quantised MoE layer forward (QMoE).

The compute lives in ``libqmoe.so`` (C ABI, ``include/qmoe.h``); this package
holds its ctypes binding (:mod:`.binding`, the C names) and :class:`QMoELayer`,
a convenience owner of one layer handle that takes torch CUDA tensors.
PyTorch is used only for device memory and streams.
"""
from __future__ import annotations

from . import binding
from .binding import *  # noqa: F401,F403  (the C-ABI names)

_DT = {"f32": binding.QMOE_F32, "f16": binding.QMOE_F16, "bf16": binding.QMOE_BF16}
_ZP = {"sym": binding.QMOE_ZP_SYMMETRIC, "uint8": binding.QMOE_ZP_UINT8,
       "offset": binding.QMOE_ZP_OFFSET}
_ACT = {"swiglu": binding.QMOE_ACT_SWIGLU, "geglu": binding.QMOE_ACT_GEGLU_TANH,
        "relu": binding.QMOE_ACT_RELU, "gelu": binding.QMOE_ACT_GELU_TANH, "silu": binding.QMOE_ACT_SILU,
        "identity": binding.QMOE_ACT_IDENTITY}


class QMoEError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{binding.qmoe_status_string(status)}: {msg}")
        self.status = status


def _ptr(t):
    return 0 if t is None else t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


class QMoELayer:
    """One QMoE layer on the current CUDA device.

    Parameters mirror ``qmoe_create``; string forms are accepted for
    ``zp_mode`` ("sym" | "uint8" | "offset"), ``activation`` ("swiglu" |
    "geglu" gated; "relu" | "gelu" | "silu" | "identity" non-gated) and
    ``dtype`` ("f32" | "f16" | "bf16").
    """

    def __init__(self, hidden, inter, experts, top_k, bits_fc1, bits_fc2, block_size,
                 zp_mode="sym", activation="swiglu", dtype="bf16", normalize=True,
                 zp_offset=None):
        zp = _ZP.get(zp_mode, zp_mode)
        act = _ACT.get(activation, activation)
        dt = _DT.get(dtype, dtype)
        st, h = binding.qmoe_create(hidden, inter, experts, top_k, bits_fc1, bits_fc2,
                                    block_size, zp, act, dt)
        if st != binding.QMOE_OK:
            raise QMoEError(st, "qmoe_create rejected the configuration")
        self.handle = h
        self.hidden, self.inter, self.experts, self.top_k = hidden, inter, experts, top_k
        self._check(binding.qmoe_set_routing(h, normalize))
        if zp_offset is not None:
            self._check(binding.qmoe_set_zero_point_offset(h, zp_offset))

    @classmethod
    def from_config(cls, cfg):
        layer = cls(cfg.H, cfg.I, cfg.E, cfg.k, cfg.bits1, cfg.bits2, cfg.B, cfg.zp_mode,
                    cfg.act, cfg.dtype, cfg.normalize,
                    cfg.zp_offset if cfg.zp_mode == "offset" else None)
        if getattr(cfg, "fc1_layout", "concat") != "concat":
            layer.set_fc1_layout(cfg.fc1_layout)
        if (getattr(cfg, "swiglu_alpha", 1.0), getattr(cfg, "swiglu_beta", 0.0),
                getattr(cfg, "swiglu_limit", float("inf"))) != (1.0, 0.0, float("inf")):
            layer.set_swiglu_params(cfg.swiglu_alpha, cfg.swiglu_beta, cfg.swiglu_limit)
        return layer

    def set_swiglu_params(self, alpha, beta, limit):
        self._check(binding.qmoe_set_swiglu_params(self.handle, alpha, beta, limit))

    def set_fc1_layout(self, layout):
        """"concat" | "interleaved" | "separate" (fc1 = gate rows, fc3 = up
        rows), or True / False for interleaved / concatenated."""
        codes = {"concat": binding.QMOE_FC1_CONCAT, "interleaved": binding.QMOE_FC1_INTERLEAVED,
                 "separate": binding.QMOE_FC1_SEPARATE_FC3, True: binding.QMOE_FC1_INTERLEAVED,
                 False: binding.QMOE_FC1_CONCAT}
        self._check(binding.qmoe_set_fc1_layout(self.handle, codes.get(layout, layout)))

    def set_bias(self, fc, bias, stream=None):
        """fp32 [E, N] device tensor (fc 1, 2, or 3 beside a separate fc1), or
        None to remove."""
        self._check(binding.qmoe_set_bias(self.handle, fc, _ptr(bias), _stream(stream)))

    def _check(self, st):
        if st != binding.QMOE_OK:
            raise QMoEError(st, binding.qmoe_last_error(self.handle))

    def reserve(self, max_tokens):
        self._check(binding.qmoe_reserve(self.handle, max_tokens))

    def set_gemm_min_rows(self, n):
        self._check(binding.qmoe_set_gemm_min_rows(self.handle, n))

    def set_fused_decode(self, mode):
        """QMOE_FUSED_OFF / QMOE_FUSED_ON / QMOE_FUSED_AUTO (default)."""
        self._check(binding.qmoe_set_fused_decode(self.handle, mode))

    def set_deterministic(self, mode):
        """Combine of the tensor-core path: 0 / False = fp32 reductions,
        1 / True = slot-ordered (bitwise deterministic), 2 = automatic (the
        default: ordered up to 64 tokens)."""
        self._check(binding.qmoe_set_deterministic(self.handle, int(mode)))

    def last_path(self):
        """QMOE_PATH_SEPARATE or QMOE_PATH_FUSED: the launch sequence of the
        last forward (QMOE_PATH_NONE before any)."""
        return binding.qmoe_last_forward_path(self.handle)

    def prepack(self, fc, codes, scales, zp=None, stream=None):
        self._check(binding.qmoe_prepack(self.handle, fc, _ptr(codes), _ptr(scales), _ptr(zp),
                                         _stream(stream)))

    def forward(self, x, logits, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty_like(x)
        self._check(binding.qmoe_forward(self.handle, _ptr(x), _ptr(logits), _ptr(out),
                                         x.shape[0], _stream(stream)))
        return out

    def forward_host(self, x_host, logits_host, out_host, stream=None):
        self._check(binding.qmoe_forward_host(self.handle, _ptr(x_host), _ptr(logits_host),
                                              _ptr(out_host), x_host.shape[0], _stream(stream)))
        return out_host

    def routing(self, T, stream=None):
        import torch
        R = T * self.top_k
        dev = torch.device("cuda")
        ids = torch.empty(R, dtype=torch.int32, device=dev)
        w = torch.empty(R, dtype=torch.float32, device=dev)
        perm = torch.empty(R, dtype=torch.int32, device=dev)
        offs = torch.empty(self.experts + 1, dtype=torch.int32, device=dev)
        self._check(binding.qmoe_get_routing(self.handle, _ptr(ids), _ptr(w), _ptr(perm),
                                             _ptr(offs), _stream(stream)))
        return ids, w, perm, offs

    def worklist(self, which, T, stream=None):
        import torch
        cap = binding.qmoe_worklist_capacity(self.handle, which, T)
        items = torch.empty((cap, 4), dtype=torch.int32, device="cuda")
        cnt = torch.empty(1, dtype=torch.int32, device="cuda")
        st, m_tile = binding.qmoe_get_worklist(self.handle, which, _ptr(items), _ptr(cnt), cap,
                                               _stream(stream))
        self._check(st)
        torch.cuda.synchronize()
        return items[: int(cnt.item())].cpu(), m_tile

    def set_trace_events(self, events):
        # torch only reports elapsed times of events it has seen recorded;
        # record each once here, the library re-records them every forward.
        for e in events or []:
            e.record()
        self._check(binding.qmoe_set_trace_events(
            self.handle, None if events is None else [e.cuda_event for e in events]))

    def poll(self):
        return binding.qmoe_poll_device_status(self.handle)

    def set_wait_limit(self, n):
        self._check(binding.qmoe_set_wait_limit(self.handle, n))

    def inject_stall(self, enable):
        self._check(binding.qmoe_debug_inject_stall(self.handle, enable))

    def close(self):
        if getattr(self, "handle", None):
            binding.qmoe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def load_inputs(layer: QMoELayer, inp: dict, device="cuda"):
    """Move one workload (qmoe_inputs.make_inputs) to the device and prepack
    it.  Returns (x, logits) device tensors."""
    for fc in (1, 2, 3):
        pre = f"fc{fc}_"
        if inp.get(pre + "codes") is None:
            continue      # fc3 only beside a separate-gate fc1
        codes = inp[pre + "codes"].to(device)
        scales = inp[pre + "scales"].to(device)
        zp = inp[pre + "zp"]
        zp = zp.to(device) if zp is not None else None
        layer.prepack(fc, codes, scales, zp)
        b = inp.get(pre + "bias")
        if b is not None:
            layer.set_bias(fc, b.to(device))
    import torch
    torch.cuda.synchronize()
    return inp["x"].to(device), inp["logits"].to(device)
