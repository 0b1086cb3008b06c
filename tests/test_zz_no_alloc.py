"""The allocation-free verify entry point, checked against mtp_verify.

Some callers cannot allocate device memory where they verify drafts (their
device memory belongs to a fixed plan or another framework's pool, or they
cannot afford cudaMalloc's device-wide synchronisation), so they cannot create
a context either.  mtp_verify_noalloc serves them with a fixed scratch array
inside the library.  This file is collected last so that a failure here does
not hide any other test; it passes alone in a fresh process and after the
rest of the suite."""
import ctypes

import numpy as np
import pytest

import synth


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from mtp_self_speculative_gb300 import _lib
    lib = _lib.load()
    # B * (max_k + 1) > 65536, B > 4096, max_k > 100: rejected before any device work
    assert lib.mtp_verify_noalloc(None, 8192, 100, 1, 8, 1, 1, 1, 1, 8, 1, 1, 1) == _lib.MTP_ERR_INVALID
    assert lib.mtp_verify_noalloc(None, 4096, 100, 1, 16, 1, 1, 1, 1, 16, 1, 1, 1) == _lib.MTP_ERR_INVALID
    assert lib.mtp_verify_noalloc(None, 4, 100, 1, 101, 1, 1, 1, 1, 101, 1, 1, 1) == _lib.MTP_ERR_INVALID
    assert lib.mtp_verify_noalloc(None, 4, 100, 5, 4, 1, 1, 1, 1, 4, 1, 1, 1) == _lib.MTP_ERR_INVALID
    assert lib.mtp_verify_noalloc(None, 4, 100, 1, 4, None, 1, 1, 1, 4, 1, 1, 1) == _lib.MTP_ERR_INVALID


def _both(cfg, vi, ctx, M, torch, dev, host):
    B = len(vi.num_drafts)
    outs = []
    from gpu_util import Guarded
    for fn in ("ctx", "noalloc"):
        acc = Guarded((B,), torch.int32, fill=-9)
        bon = Guarded((B,), torch.int32, fill=-9)
        args = (dev(vi.logits), dev(vi.row_offsets), dev(vi.drafts), dev(vi.num_drafts), acc.t, bon.t)
        if fn == "ctx":
            M.mtp_verify(ctx, *args)
        else:
            M.mtp_verify_noalloc(*args, vocab=cfg.vocab, max_k=vi.max_k)
        torch.cuda.synchronize()
        acc.check("accepted")
        bon.check("bonus")
        outs.append((host(acc.t), host(bon.t)))
    return outs


@pytest.mark.gpu
def test_noalloc_verify_matches_context_verify_twice():
    import torch
    import mtp_self_speculative_gb300 as M
    from gpu_util import dev, host, make_context

    # two calls in a row on the 64-request bf16 workload (ragged K_b in 1..8)
    cfg = synth.VERIFY_B64
    vi = synth.make_verify_inputs(cfg)
    ctx = make_context(cfg, None, max_batch=cfg.batch, max_k=vi.max_k)
    for _ in range(2):
        (a_ctx, b_ctx), (a_na, b_na) = _both(cfg, vi, ctx, M, torch, dev, host)
        np.testing.assert_array_equal(a_na, a_ctx)     # integer outputs: bit-exact
        np.testing.assert_array_equal(b_na, b_ctx)
    assert M.mtp_get_device_error(ctx) == 0

    # a smaller float32 call next: the shared scratch must not carry the
    # previous call's keys or counters into this one
    cfg2 = synth.TINY_F32
    ctx2 = make_context(cfg2, None, max_batch=1, max_k=3)
    for seed in (5, 6):
        vi2 = synth.make_verify_inputs(cfg2, num_drafts=np.array([3]), seed=seed, len_mode="uniform")
        (a_ctx, b_ctx), (a_na, b_na) = _both(cfg2, vi2, ctx2, M, torch, dev, host)
        np.testing.assert_array_equal(a_na, a_ctx)
        np.testing.assert_array_equal(b_na, b_ctx)


@pytest.mark.gpu
def test_noalloc_malformed_rows_give_minus_one_for_those_requests_only():
    """Request 1 claims one row too many, so request 2 is left one short:
    both get accepted = bonus = -1 (the documented device-side result, there
    being no error word without a context); requests 0 and 3 still get the
    oracle's results.  A second, well-formed call right after it is exact
    again."""
    import torch
    import mtp_self_speculative_gb300 as M
    import oracle as O
    from gpu_util import Guarded, dev, host

    cfg = synth.shrink(synth.VERIFY_B64, vocab=3001, batch=4)
    vi = synth.make_verify_inputs(cfg)
    ro = vi.row_offsets.copy()
    ro[2] += 1
    acc_o, bon_o = O.verify(vi.logits, vi.row_offsets, vi.drafts, vi.num_drafts, "bf16")
    for offsets, bad in ((ro, {1, 2}), (vi.row_offsets, set())):
        acc = Guarded((4,), torch.int32, fill=-9)
        bon = Guarded((4,), torch.int32, fill=-9)
        M.mtp_verify_noalloc(dev(vi.logits), dev(offsets), dev(vi.drafts), dev(vi.num_drafts), acc.t, bon.t,
                             vocab=cfg.vocab, max_k=vi.max_k)
        torch.cuda.synchronize()
        acc.check("accepted")
        bon.check("bonus")
        a, b_ = host(acc.t), host(bon.t)
        for r in range(4):
            if r in bad:
                assert (a[r], b_[r]) == (-1, -1), r
            else:
                assert (a[r], b_[r]) == (acc_o[r], bon_o[r]), r
