"""Pins of the oracle's quantized-head format (4-bit asymmetric, group size
64, INT8 symmetric backup; "How OpenVINO MTP Speculative Decoding Works
Internally", "Why MTP gets its own quantization configuration") against
hand-worked groups, exact-grid inputs, error bounds and the packing layout.
CPU only."""
import numpy as np

import oracle as O
from oracle import quant as Q
import synth


def bits(values):
    """bf16 bits of float32-exact bf16 values."""
    return synth.f32_to_bf16_bits(np.asarray(values, dtype=np.float32))


def test_int4_grid_group_is_reproduced_exactly():
    # values c*(j - 8), j = 0..15, repeated: lo = -8c, hi = 7c -> s = c, z = 8,
    # code = j; the grid is exact in bf16 and fp16, so dequantization is exact
    c = 0.125
    j = np.tile(np.arange(16), 4)
    w = bits(c * (j - 8))[None, :]
    q, s, z = Q.quantize_int4_g64(w)
    assert s.view(np.float16)[0, 0] == c and z[0, 0] == 8
    np.testing.assert_array_equal(Q.unpack_int4(q)[0], j)
    np.testing.assert_array_equal(Q.dequantize_int4_g64(q, s, z)[0], c * (j - 8))


def test_int4_all_positive_and_all_negative_groups_keep_zero_in_range():
    # zero is always representable: a positive group has z = 0, a negative one z = 15
    pos = bits(np.linspace(1.0, 15.0, 64).round(0))[None, :]       # 1..15
    q, s, z = Q.quantize_int4_g64(pos)
    assert z[0, 0] == 0 and s.view(np.float16)[0, 0] == 1.0
    np.testing.assert_array_equal(Q.dequantize_int4_g64(q, s, z)[0], np.linspace(1.0, 15.0, 64).round(0))
    neg = bits(-np.linspace(1.0, 15.0, 64).round(0))[None, :]
    q, s, z = Q.quantize_int4_g64(neg)
    assert z[0, 0] == 15
    np.testing.assert_array_equal(Q.dequantize_int4_g64(q, s, z)[0], -np.linspace(1.0, 15.0, 64).round(0))


def test_int4_zero_group_and_constant_group():
    w = np.zeros((1, 128), dtype=np.uint16)
    w[0, 64:] = bits(np.full(64, 3.0))
    q, s, z = Q.quantize_int4_g64(w)
    # all-zero group: scale 1, zero point 0, codes 0
    assert s.view(np.float16)[0, 0] == 1.0 and z[0, 0] == 0
    assert not Q.unpack_int4(q)[0, :64].any()
    # constant 3.0: s = 3/15 = 0.2, every code 15, value 15 * fp16(0.2)
    assert z[0, 1] == 0
    np.testing.assert_array_equal(Q.unpack_int4(q)[0, 64:], 15)
    np.testing.assert_array_equal(Q.dequantize_int4_g64(q, s, z)[0, 64:],
                                  15 * float(np.float16(np.float32(3.0) / np.float32(15.0))))


def test_int4_halfway_codes_round_to_even():
    # s = 1 (group spans 0..15), z = 0: 0.5 -> 0, 1.5 -> 2, 2.5 -> 2, 3.5 -> 4
    vals = np.zeros(64, dtype=np.float32)
    vals[0] = 15.0
    vals[1:5] = [0.5, 1.5, 2.5, 3.5]
    q, s, z = Q.quantize_int4_g64(bits(vals)[None, :])
    np.testing.assert_array_equal(Q.unpack_int4(q)[0, 1:5], [0, 2, 2, 4])


def test_int4_packing_low_nibble_first():
    c = 1.0
    j = np.tile(np.arange(16), 4)
    q, _, _ = Q.quantize_int4_g64(bits(c * j)[None, :])
    # byte k holds column 2k in bits 0..3 and column 2k+1 in bits 4..7
    np.testing.assert_array_equal(q[0, :8], [0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE])


def test_int4_random_groups_error_bound():
    rng_bits = synth.f32_to_bf16_bits(synth.normal(5, 3, (16, 512), dtype="f32") * np.float32(0.02))
    w = O.widen(rng_bits, "bf16")
    q, s, z = Q.quantize_int4_g64(rng_bits)
    codes = Q.unpack_int4(q)
    assert codes.max() <= 15
    deq = Q.dequantize_int4_g64(q, s, z)
    sg = np.repeat(s.view(np.float16).astype(np.float64), 64, axis=1)
    # round to nearest on the grid: half a step, plus the fp16 rounding of s
    # (relative 2^-11) times at most 15 steps
    assert np.all(np.abs(deq - w) <= sg * (0.5 + 15 * 2.0 ** -11) + 1e-12)
    # each group's extremes lie within a step of the grid ends
    wg = w.reshape(16, 8, 64)
    lo = np.minimum(wg.min(axis=2), 0)
    hi = np.maximum(wg.max(axis=2), 0)
    sf = s.view(np.float16).astype(np.float64)
    np.testing.assert_allclose(sf, (hi - lo) / 15, rtol=2.0 ** -10)


def test_int8_rows_exact_grid_zero_row_and_extremes():
    c = 2.0 ** -6
    j = np.arange(-127, 129) % 255 - 127        # covers -127..127
    w = np.zeros((3, 256), dtype=np.uint16)
    w[0] = bits(c * j)
    w[2] = bits(c * -j)
    q, s = Q.quantize_int8_rows(w)
    sf = s.view(np.float16).astype(np.float64)
    assert sf[0] == c and sf[2] == c and sf[1] == 1.0
    np.testing.assert_array_equal(q[0], j)
    np.testing.assert_array_equal(q[2], -j)
    assert not q[1].any()
    assert q.min() == -127 and q.max() == 127
    np.testing.assert_array_equal(Q.dequantize_int8_rows(q, s)[0], c * j)


def test_int8_random_rows_error_bound():
    b = synth.f32_to_bf16_bits(synth.normal(9, 4, (32, 384), dtype="f32") * np.float32(0.02))
    w = O.widen(b, "bf16")
    q, s = Q.quantize_int8_rows(b)
    deq = Q.dequantize_int8_rows(q, s)
    sf = s.view(np.float16).astype(np.float64)[:, None]
    assert np.all(np.abs(deq - w) <= sf * (0.5 + 127 * 2.0 ** -11) + 1e-12)
    # the row's largest magnitude maps to +-127
    np.testing.assert_array_equal(np.abs(q).max(axis=1), 127)


def test_quantized_weights_dequantize_table_on_use():
    cfg = synth.MTPShape("quant_pin_bf16", H=128, n_q=2, n_kv=1, head_dim=64, ffn=256, vocab=300, batch=1, K=2,
                         dtype="bf16", ctx_lo=4, ctx_hi=4, seed_index=60)
    w = synth.make_weights(cfg, norm="random")
    W = Q.quantized_weights(w, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    q8, s8 = Q.quantize_int8_rows(w["embed"])
    ids = np.array([0, 5, cfg.vocab - 1])
    full = Q.dequantize_int8_rows(q8, s8)
    np.testing.assert_array_equal(W.embed_rows(ids), full[ids])
    np.testing.assert_array_equal(W.lm_chunk(3, 17), full[3:17])
    # projections hold the exact INT4 dequantization, norms stay bf16
    np.testing.assert_array_equal(W.w_q, Q.dequantize_int4_g64(*Q.quantize_int4_g64(w["w_q"])))
    np.testing.assert_array_equal(W.w_norm_in, O.widen(w["w_norm_in"], "bf16"))
    assert W.dtype == "bf16"
