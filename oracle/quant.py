"""Quantized MTP head for the oracle: the format named on "How OpenVINO MTP
Speculative Decoding Works Internally", "Why MTP gets its own quantization
configuration" (4-bit asymmetric, group size 64, INT8 symmetric backup).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages name the format but not its arithmetic; the reading used here (and
listed in the design notes) is the plain round-to-nearest one:

  INT4, per group of 64 consecutive input columns w_0..w_63:
      lo = min(min_i w_i, 0), hi = max(max_i w_i, 0)
      s  = (hi - lo) / 15, or 1 when that is 0
      z  = clamp(rint(-lo / s), 0, 15)
      q_i = clamp(rint(w_i / s) + z, 0, 15)
      dequantized w'_i = (q_i - z) * fp16(s)
  INT8 backup, per row (the shared embedding / LM head):
      s = max_i |w_i| / 127, or 1 when that is 0
      q_i = clamp(rint(w_i / s), -127, 127)
      dequantized w'_i = q_i * fp16(s)

Every step is IEEE float32 with round-half-to-even (numpy float32 arithmetic
and np.rint), so the integer codes are a deterministic function of the bf16
inputs; dequantization is exact in float64.
"""
from dataclasses import dataclass
from typing import Dict, Optional, Tuple

import numpy as np

from .mtp_oracle import MTPWeights64, widen

# projection tensors quantized to INT4 (the backup INT8 covers the table)
INT4_NAMES = ("w_eh", "w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down")


_ROWS = 4096        # rows quantized at a time (bounds the host memory used)


def _bf16_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> the same values as float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def quantize_int4_g64(w_bits: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """bf16 bits [R, C] (C % 64 == 0) -> packed codes [R, C/2] uint8 (column
    2k in the low nibble of byte k), fp16 scale bits [R, C/64] uint16, zero
    points [R, C/64] uint8."""
    R, C = w_bits.shape
    if R > _ROWS:
        parts = [quantize_int4_g64(w_bits[r:r + _ROWS]) for r in range(0, R, _ROWS)]
        return tuple(np.concatenate([p[i] for p in parts]) for i in range(3))
    w = _bf16_f32(w_bits).reshape(R, C // 64, 64)
    lo = np.minimum(w.min(axis=2), np.float32(0.0))
    hi = np.maximum(w.max(axis=2), np.float32(0.0))
    s = (hi - lo) / np.float32(15.0)
    s = np.where(s == np.float32(0.0), np.float32(1.0), s).astype(np.float32)
    z = np.clip(np.rint(-lo / s), np.float32(0.0), np.float32(15.0)).astype(np.float32)
    q = np.clip(np.rint(w / s[:, :, None]) + z[:, :, None], np.float32(0.0), np.float32(15.0)).astype(np.uint8)
    q = q.reshape(R, C // 2, 2)
    packed = (q[:, :, 0] | (q[:, :, 1] << 4)).astype(np.uint8)
    return packed, s.astype(np.float16).view(np.uint16), z.astype(np.uint8)


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """[R, C/2] bytes -> [R, C] codes."""
    R, half = packed.shape
    out = np.empty((R, 2 * half), dtype=np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def dequantize_int4_g64(packed: np.ndarray, scale_bits: np.ndarray, zeros: np.ndarray) -> np.ndarray:
    """Exact float64 values (q - z) * fp16(s)."""
    q = unpack_int4(packed).astype(np.float64)
    R, C = q.shape
    s = scale_bits.view(np.float16).astype(np.float64)
    z = zeros.astype(np.float64)
    return ((q.reshape(R, C // 64, 64) - z[:, :, None]) * s[:, :, None]).reshape(R, C)


def quantize_int8_rows(w_bits: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """bf16 bits [R, C] -> codes [R, C] int8, fp16 scale bits [R] uint16."""
    R = w_bits.shape[0]
    if R > _ROWS:
        parts = [quantize_int8_rows(w_bits[r:r + _ROWS]) for r in range(0, R, _ROWS)]
        return tuple(np.concatenate([p[i] for p in parts]) for i in range(2))
    w = _bf16_f32(w_bits)
    amax = np.abs(w).max(axis=1)
    s = amax / np.float32(127.0)
    s = np.where(s == np.float32(0.0), np.float32(1.0), s).astype(np.float32)
    q = np.clip(np.rint(w / s[:, None]), np.float32(-127.0), np.float32(127.0)).astype(np.int8)
    return q, s.astype(np.float16).view(np.uint16)


def dequantize_int8_rows(q: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """Exact float64 values q * fp16(s)."""
    return q.astype(np.float64) * scale_bits.view(np.float16).astype(np.float64)[:, None]


@dataclass
class QuantizedWeights64(MTPWeights64):
    """The oracle's head weights with the quantized format: projections
    dequantized to float64, the INT8 table kept as codes and widened on use
    (embed_stored / lm_stored hold the codes, *_scale the fp16 bits).  dtype
    stays "bf16": it is the KV cache's storage format."""
    embed_scale: Optional[np.ndarray] = None
    lm_scale: Optional[np.ndarray] = None

    def lm_chunk(self, r0: int, r1: int) -> np.ndarray:
        return dequantize_int8_rows(self.lm_stored[r0:r1], self.lm_scale[r0:r1])

    def embed_rows(self, ids: np.ndarray) -> np.ndarray:
        ids = np.asarray(ids)
        return dequantize_int8_rows(self.embed_stored[ids].reshape(-1, self.embed_stored.shape[1]),
                                    self.embed_scale[ids].reshape(-1)).reshape(ids.shape + (-1,))


def quantized_weights(w: Dict[str, np.ndarray], n_q: int, n_kv: int, head_dim: int, eps: float,
                      rope_theta: float) -> QuantizedWeights64:
    """Quantize the stored bf16 head weights ``w`` (synth.make_weights keys;
    the LM head is the embedding table) and return the oracle's view of the
    quantized head."""
    wd = {}
    for k, v in w.items():
        if k == "embed":
            continue
        if k in INT4_NAMES:
            wd[k] = dequantize_int4_g64(*quantize_int4_g64(v))
        else:
            wd[k] = widen(v, "bf16")
    q8, s8 = quantize_int8_rows(w["embed"])
    return QuantizedWeights64(embed_stored=q8, lm_stored=q8, embed_scale=s8, lm_scale=s8, dtype="bf16", n_q=n_q,
                              n_kv=n_kv, head_dim=head_dim, eps=eps, rope_theta=rope_theta, **wd)
