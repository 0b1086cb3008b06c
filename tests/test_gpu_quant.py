"""Quantized MTP head on the GPU (4-bit asymmetric group-64 projections, INT8
symmetric per-row embedding / LM head; "How OpenVINO MTP Speculative
Decoding Works Internally", "Why MTP gets its own quantization
configuration"), through the C ABI:

* the device quantizers give the oracle's codes, scales and zero points bit
  for bit (both sides compute in IEEE fp32 with round-half-to-even);
* drafting with the quantized head matches the oracle run on the exactly
  dequantized weights, under the same tolerances as the dense head."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import LOGIT_TOL, dev, host, make_context, upload_weights
from oracle import quant as Q
from test_gpu_draft import Case, check_forced, check_free

pytestmark = pytest.mark.gpu


def special_matrix(rows, cols, seed_stream):
    """Seeded N(0, 0.02) bf16 rows with hand-made groups planted: all zero,
    constant, halfway codes, all negative, large, tiny."""
    w = synth.f32_to_bf16_bits(synth.normal(70, seed_stream, (rows, cols), dtype="f32") * np.float32(0.02))
    f = lambda v: synth.f32_to_bf16_bits(np.asarray(v, dtype=np.float32))
    w[0, 0:64] = 0
    w[0, 64:128] = f(np.full(64, 3.0))
    ties = np.zeros(64, dtype=np.float32)
    ties[0] = 15.0
    ties[1:9] = [0.5, 1.5, 2.5, 3.5, 4.5, 5.5, 6.5, 7.5]
    w[1, 0:64] = f(ties)
    w[1, 64:128] = f(-np.abs(synth.normal(71, seed_stream, (64,), dtype="f32")))
    w[2, 0:64] = f(synth.normal(72, seed_stream, (64,), dtype="f32") * np.float32(3e4))
    w[2, 64:128] = f(synth.normal(73, seed_stream, (64,), dtype="f32") * np.float32(1e-20))
    w[3, :] = 0                                     # an all-zero row (INT8 scale 1)
    return w


@pytest.mark.parametrize("shape", [(300, 1024), (7, 4096), (64, 128)])
def test_int4_quantizer_matches_oracle_bitwise(shape):
    import mtp_self_speculative_gb300 as M
    R, C = shape
    w = special_matrix(R, C, 1)
    q = torch.empty((R, C // 2), dtype=torch.uint8, device="cuda")
    s = torch.empty((R, C // 64), dtype=torch.int16, device="cuda")
    z = torch.empty((R, C // 64), dtype=torch.uint8, device="cuda")
    M.mtp_quantize_int4_g64(dev(w), q, s, z)
    torch.cuda.synchronize()
    oq, os_, oz = Q.quantize_int4_g64(w)
    np.testing.assert_array_equal(host(q), oq)
    np.testing.assert_array_equal(host(s).view(np.uint16), os_)
    np.testing.assert_array_equal(host(z), oz)


@pytest.mark.parametrize("shape", [(513, 4096), (5, 100), (1, 8192)])
def test_int8_quantizer_matches_oracle_bitwise(shape):
    import mtp_self_speculative_gb300 as M
    R, C = shape
    w = special_matrix(R, C, 2) if C >= 128 and R >= 4 else \
        synth.f32_to_bf16_bits(synth.normal(74, 3, shape, dtype="f32") * np.float32(0.02))
    q = torch.empty((R, C), dtype=torch.int8, device="cuda")
    s = torch.empty((R,), dtype=torch.int16, device="cuda")
    M.mtp_quantize_int8_rows(dev(w), q, s)
    torch.cuda.synchronize()
    oq, os_ = Q.quantize_int8_rows(w)
    np.testing.assert_array_equal(host(q), oq)
    np.testing.assert_array_equal(host(s).view(np.uint16), os_)


def test_quantized_config_checks():
    """The quantized head needs bf16 weights, at most 4 requests per call and
    row lengths that are multiples of 1024; anything else is refused at
    creation."""
    import mtp_self_speculative_gb300 as M
    ok = synth.MTPShape("q_ok", H=1024, n_q=8, n_kv=2, head_dim=128, ffn=2048, vocab=999, batch=1, K=2,
                        dtype="bf16", ctx_lo=4, ctx_hi=4, seed_index=61)
    wdev = upload_weights(synth.make_weights(ok))
    ctx = make_context(ok, wdev, max_batch=4, weight_format="int4_g64")
    M.mtp_destroy(ctx)
    for kw in ({"max_batch": 5}, ):
        with pytest.raises(RuntimeError):
            make_context(ok, wdev, weight_format="int4_g64", **kw)
    bad_h = synth.MTPShape("q_bad_h", H=768, n_q=6, n_kv=2, head_dim=128, ffn=2048, vocab=999, batch=1, K=2,
                           dtype="bf16", ctx_lo=4, ctx_hi=4, seed_index=61)
    with pytest.raises(RuntimeError):
        make_context(bad_h, upload_weights(synth.make_weights(bad_h)), weight_format="int4_g64")
    with pytest.raises(RuntimeError):
        make_context(ok, None, weight_format="int4_g64")


SMALL_Q = dict(H=1024, n_q=8, n_kv=2, head_dim=128, ffn=2048, vocab=5003, K=3, dtype="bf16", ctx_lo=0, ctx_hi=64,
               paged_shuffle=True, seed_index=62)


@pytest.mark.parametrize("lens", [[33], [0, 17], [5, 16, 40], [1, 30, 2, 64]])
def test_quantized_small_batch(lens):
    """Quantized head, B = 1..4 (the 1-, 2- and 4-row kernel variants), odd
    vocabulary (a lone last LM row), random norm weights; forced and free
    chains against the oracle, then a bitwise-repeatable second run."""
    cfg = synth.MTPShape("small_q4", batch=len(lens), **SMALL_Q)
    case = Case(cfg, norm="random", lens=lens, weight_format="int4_g64")
    sub = list(range(len(lens)))
    _, _, ids, logits = check_forced(case, sub, LOGIT_TOL)
    check_free(case, sub, ids, logits, LOGIT_TOL)
    ids2, logits2, _, _ = case.gpu_draft(forced=True)
    np.testing.assert_array_equal(ids2, ids)
    np.testing.assert_array_equal(logits2, logits)


def test_quantized_wide_rows_batch4():
    """F = 12288 at B = 4: the largest staged input of the down projection
    next to its ring; q_dim != H (48 query heads of 128, 8 per kv head)."""
    cfg = synth.MTPShape("wide_q4", H=2048, n_q=48, n_kv=6, head_dim=128, ffn=12288, vocab=7001, batch=4, K=2,
                         dtype="bf16", ctx_lo=1, ctx_hi=90, paged_shuffle=True, seed_index=63)
    case = Case(cfg, norm="random", lens=[90, 1, 40, 17], weight_format="int4_g64")
    check_forced(case, [0, 1, 2, 3], LOGIT_TOL)


@pytest.mark.slow
def test_quantized_qwen3_8b_b1_full_size():
    """Qwen3-8B-shaped head with the quantized format, B = 1, context 4096,
    K = 5: the quantized bench workload and its launch configuration."""
    case = Case(synth.QWEN3_8B_B1, weight_format="int4_g64")
    _, _, ids, logits = check_forced(case, [0], LOGIT_TOL)
    check_free(case, [0], ids, logits, LOGIT_TOL)


def test_quantized_device_errors():
    """pending != 0 on entry and a too-short block table on the quantized
    kernels: reported through the error word, the cache untouched, and the
    context drafts correctly afterwards."""
    import mtp_self_speculative_gb300 as M
    from gpu_util import download_kv, upload_kv
    cfg = synth.MTPShape("err_q4", batch=2, **dict(SMALL_Q, ctx_lo=150, ctx_hi=200, seed_index=64))
    case = Case(cfg, norm="random", weight_format="int4_g64")
    ids = torch.empty((2, 3), dtype=torch.int32, device="cuda")
    kv = case.kv0.copy()
    kv.pending[:] = [0, 1]
    kvd = upload_kv(kv)
    M.mtp_draft(case.ctx, *case.inputs, kvd, 3, ids)
    assert M.mtp_get_device_error(case.ctx) == M.MTP_ERR_DEVICE_ARGS
    got = download_kv(kvd)
    np.testing.assert_array_equal(got.pending, [3, 1])
    L1 = int(kv.seq_len[1])
    from gpu_util import kv_slots
    gk, gv = kv_slots(got, 1, 0, L1 + 3)
    ok, ov = kv_slots(kv, 1, 0, L1 + 3)
    np.testing.assert_array_equal(gk, ok)
    np.testing.assert_array_equal(gv, ov)
    kv = case.kv0.copy()
    kv.block_table = kv.block_table[:, :8].copy()      # room for 128 slots only
    kvd = upload_kv(kv)
    M.mtp_draft(case.ctx, *case.inputs, kvd, 3, ids)
    assert M.mtp_get_device_error(case.ctx) == M.MTP_ERR_CAPACITY
    got = download_kv(kvd)
    np.testing.assert_array_equal(got.k_pool, kv.k_pool)
    check_forced(case, [0, 1], LOGIT_TOL)
