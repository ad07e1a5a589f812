"""Seeded synthetic inputs for the QMoE layer forward.

This module only *draws* data: it holds none of the layer's arithmetic
(no routing, dequantisation, projection or combine).  Both the CPU oracle's
tests and the CUDA path (tests, ``bench.py``, ``smoke()``) take their inputs
from here, so the two sides see the same bytes.

Workloads follow the shapes and value distributions of the QMoE pages:

* "Tiny" int4 SwiGLU case, and the H100 int2 GeGLU decode shape
  (hidden = inter = 2048, E = 8, top-2, block 128) from the onnxruntime PR
  "[CUDA] QMoE: fused int2 mixed-input GEMM + GeGLU activation + fractional
  zero-point" (Validation paragraph);
* a many-expert int4 decode with explicit uint8 zero points, a mixed-width
  int3/int4 case ("[CUDA] Add fast INT3 QMoE kernels ..." PR, Testing), and
  a skewed-routing int4 prefill.

Canonical (boundary) layout of the quantised expert tensors, as the
onnx-runtime-ep-cuda ``qmoe.rs`` page defines it (QuantizedExperts::validate
and ``decode_affine_weight``):

* ``codes``  uint8 ``[E, N, K*bits/8]``: each row is an LSB-first bit stream of
  K codes of ``bits`` bits (code d occupies bits [d*bits, d*bits+bits)).
* ``scales`` dtype D ``[E, N, K/B]``.
* ``zp``     uint8 ``[E, N, ceil((K/B)*bits/8)]``: LSB-first bit stream of the
  K/B per-block zero points, at the weight bit width (only in ``uint8`` mode).

fc1 rows are ``[gate (I rows) | up (I rows)]`` (concatenated gate/up), or
interleaved (row 2f = gate f, row 2f+1 = up f) when ``fc1_layout`` says so,
or, with ``fc1_layout == "separate"``, fc1 holds the I gate rows and a third
projection fc3 (keys ``fc3_*``, drawn after every other tensor) the I up rows.
Optional projection biases are float32 ``[E, N]`` in the same row order.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class QMoEConfig:
    """Shape, quantisation and distribution parameters of one workload."""

    name: str
    T: int                 # tokens
    H: int                 # hidden
    I: int                 # inter (fc1 has 2*I rows: gate | up)
    E: int                 # experts
    k: int                 # top_k
    normalize: bool        # renormalise the k routing weights
    bits1: int             # fc1 code width
    bits2: int             # fc2 code width
    B: int                 # quantisation block size along K
    zp_mode: str           # "sym" | "uint8" | "offset"
    dtype: str             # "f32" | "f16" | "bf16" (activations, scales, output)
    act: str               # gated "swiglu" | "geglu", or non-gated "relu" | "gelu" | "silu" | "identity"
    scale_lo: float
    scale_hi: float
    seed: int
    zp_offset: float = float("nan")
    zp_lo: int = 0
    zp_hi: int = 0
    logit_sigma: float = 1.0
    zipf_bias: float = 0.0  # logits[t, e] += zipf_bias * log(1 / (e + 1))
    # fc1 row order: "concat" ([gate (I rows) | up (I rows)]), "interleaved"
    # (row 2f = gate f, row 2f+1 = up f) or "separate" (fc1 = gate rows, a
    # third projection fc3 = up rows)
    fc1_layout: str = "concat"
    # SwiGLU attributes: h = min(g, L) * sigmoid(alpha * min(g, L)) * (clamp(u, -L, L) + beta)
    swiglu_alpha: float = 1.0
    swiglu_beta: float = 0.0
    swiglu_limit: float = float("inf")
    # fp32 projection biases ([E, 2I] for fc1 in its row order, [E, H] for fc2)
    bias: bool = False
    bias_sigma: float = 0.05

    def with_(self, **kw) -> "QMoEConfig":
        return dataclasses.replace(self, **kw)

    @property
    def R(self) -> int:
        return self.T * self.k


# The five workloads.  Seeds: 0 for the tiny case (as stated), 1..4 for the
# others in order.
CONFIGS = {
    "tiny": QMoEConfig(
        name="tiny", T=4, H=128, I=256, E=4, k=2, normalize=True, bits1=4, bits2=4,
        B=32, zp_mode="sym", dtype="f32", act="swiglu", scale_lo=0.005,
        scale_hi=0.02, seed=0),
    "decode_int2": QMoEConfig(
        name="decode_int2", T=8, H=2048, I=2048, E=8, k=2, normalize=True, bits1=2,
        bits2=2, B=128, zp_mode="offset", zp_offset=1.5, dtype="f16", act="geglu",
        scale_lo=0.01, scale_hi=0.05, seed=1),
    "decode_many_expert_int4": QMoEConfig(
        name="decode_many_expert_int4", T=32, H=2048, I=768, E=128, k=8,
        normalize=True, bits1=4, bits2=4, B=32, zp_mode="uint8", zp_lo=6, zp_hi=9,
        dtype="bf16", act="swiglu", scale_lo=0.005, scale_hi=0.02, logit_sigma=2.0,
        seed=2),
    "mixed_int3_int4": QMoEConfig(
        name="mixed_int3_int4", T=64, H=2880, I=2880, E=32, k=4, normalize=False,
        bits1=3, bits2=4, B=32, zp_mode="sym", dtype="bf16", act="swiglu",
        scale_lo=0.005, scale_hi=0.02, seed=3),
    "prefill_int4": QMoEConfig(
        name="prefill_int4", T=4096, H=4096, I=1536, E=64, k=8, normalize=True,
        bits1=4, bits2=4, B=128, zp_mode="sym", dtype="bf16", act="swiglu",
        scale_lo=0.002, scale_hi=0.01, zipf_bias=1.5, seed=4),
}


def pack_fields(values: np.ndarray, bits: int) -> np.ndarray:
    """Encode the last axis of ``values`` (ints < 2**bits) as an LSB-first bit
    stream of ``bits``-bit fields, padded with zero bits to whole bytes.

    This is the storage format of the boundary, not part of the layer's
    arithmetic; it is used here only to write explicit zero points and in
    tests that build hand-made code rows.
    """
    values = np.asarray(values, dtype=np.int64)
    n = values.shape[-1]
    nbytes = (n * bits + 7) // 8
    bitarr = ((values[..., :, None] >> np.arange(bits)) & 1).astype(np.uint8)
    bitarr = bitarr.reshape(values.shape[:-1] + (n * bits,))
    pad = nbytes * 8 - n * bits
    if pad:
        bitarr = np.concatenate(
            [bitarr, np.zeros(values.shape[:-1] + (pad,), np.uint8)], axis=-1)
    return np.packbits(bitarr, axis=-1, bitorder="little")


def zp_row_bytes(K: int, B: int, bits: int) -> int:
    return (K // B * bits + 7) // 8


def _cast(a: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DTYPES[dtype])


def _projection(rng, cfg: QMoEConfig, N: int, K: int, bits: int):
    codes = rng.integers(0, 256, size=(cfg.E, N, K * bits // 8), dtype=np.uint8)
    scales = _cast(rng.uniform(cfg.scale_lo, cfg.scale_hi,
                               size=(cfg.E, N, K // cfg.B)).astype(np.float32),
                   cfg.dtype)
    zp = None
    if cfg.zp_mode == "uint8":
        vals = rng.integers(cfg.zp_lo, cfg.zp_hi + 1, size=(cfg.E, N, K // cfg.B))
        zp = torch.from_numpy(pack_fields(vals, bits))
    return torch.from_numpy(codes), scales, zp


def make_inputs(cfg: QMoEConfig, T: Optional[int] = None) -> dict:
    """Draw one workload.  Fixed draw order: logits, x, fc1 codes, fc1 scales,
    fc1 zero points, fc2 codes, fc2 scales, fc2 zero points.

    Returns CPU torch tensors in the canonical layout (see module doc).
    """
    T = cfg.T if T is None else T
    rng = np.random.default_rng(cfg.seed)
    logits = rng.standard_normal((T, cfg.E), dtype=np.float32) * np.float32(cfg.logit_sigma)
    if cfg.zipf_bias:
        bias = (cfg.zipf_bias * np.log(1.0 / (np.arange(cfg.E) + 1.0))).astype(np.float32)
        logits = (logits + bias[None, :]).astype(np.float32)
    x = _cast(rng.standard_normal((T, cfg.H), dtype=np.float32), cfg.dtype)
    # a separate fc3 holds the up rows: fc1 then has only the I gate rows
    sep = cfg.fc1_layout == "separate"
    gated = cfg.act in ("swiglu", "geglu")
    n1 = cfg.I if (sep or not gated) else 2 * cfg.I
    fc1 = _projection(rng, cfg, n1, cfg.H, cfg.bits1)
    fc2 = _projection(rng, cfg, cfg.H, cfg.I, cfg.bits2)
    b1 = b2 = b3 = None
    if cfg.bias:   # drawn after everything else: the other streams do not move
        b1 = torch.from_numpy((rng.standard_normal((cfg.E, n1)) * cfg.bias_sigma).astype(np.float32))
        b2 = torch.from_numpy((rng.standard_normal((cfg.E, cfg.H)) * cfg.bias_sigma).astype(np.float32))
    fc3 = (None, None, None)
    if sep:        # after that, fc3 (codes, scales, zero points, bias)
        fc3 = _projection(rng, cfg, cfg.I, cfg.H, cfg.bits1)
        if cfg.bias:
            b3 = torch.from_numpy((rng.standard_normal((cfg.E, cfg.I)) * cfg.bias_sigma).astype(np.float32))
    return {
        "cfg": cfg.with_(T=T),
        "logits": torch.from_numpy(np.ascontiguousarray(logits)),
        "x": x,
        "fc1_codes": fc1[0], "fc1_scales": fc1[1], "fc1_zp": fc1[2],
        "fc2_codes": fc2[0], "fc2_scales": fc2[1], "fc2_zp": fc2[2],
        "fc3_codes": fc3[0], "fc3_scales": fc3[1], "fc3_zp": fc3[2],
        "fc1_bias": b1, "fc2_bias": b2, "fc3_bias": b3,
    }


def weight_bytes_per_expert(cfg: QMoEConfig) -> int:
    """Bytes of one expert's packed codes + scales + zero points (both fcs)."""
    esz = torch.tensor([], dtype=DTYPES[cfg.dtype]).element_size()
    total = 0
    n1 = 2 * cfg.I if cfg.act in ("swiglu", "geglu") else cfg.I
    for N, K, bits in ((n1, cfg.H, cfg.bits1), (cfg.H, cfg.I, cfg.bits2)):
        total += N * K * bits // 8 + N * (K // cfg.B) * esz
        if cfg.zp_mode == "uint8":
            total += N * zp_row_bytes(K, cfg.B, bits)
    return total


def expert_fc_bytes(cfg: QMoEConfig, fc: int) -> int:
    """Bytes of one expert's fc1 (fc=1) or fc2 (fc=2) codes + scales + zp."""
    esz = torch.tensor([], dtype=DTYPES[cfg.dtype]).element_size()
    n1 = 2 * cfg.I if cfg.act in ("swiglu", "geglu") else cfg.I
    N, K, bits = ((n1, cfg.H, cfg.bits1) if fc == 1 else (cfg.H, cfg.I, cfg.bits2))
    total = N * K * bits // 8 + N * (K // cfg.B) * esz
    if cfg.zp_mode == "uint8":
        total += N * zp_row_bytes(K, cfg.B, bits)
    return total


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = ["QMoEConfig", "CONFIGS", "DTYPES", "make_inputs", "pack_fields",
           "zp_row_bytes", "weight_bytes_per_expert", "expert_fc_bytes", "ceil_div"]
