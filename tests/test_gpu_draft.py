"""GPU MTP draft vs the float64 oracle, through the C ABI.

Parity is checked on the same seeded inputs: both sides draft with the same
given token chain (so every step is comparable), logits within the stated
normwise tolerance, draft ids equal except at the oracle's near-ties, the
appended KV entries within tolerance, every other KV slot bit-identical.  The
free-running GPU chain is checked against the free-running oracle chain up to
the first (legitimate) near-tie divergence."""
import re

import numpy as np
import pytest
import torch

import oracle as O
import synth
from gpu_util import (F32_LOGIT_TOL, LOGIT_TOL, Guarded, check_ids, check_ids_are_argmax_of_own_logits,
                      check_logits, dev, download_kv, exact_floor, host, kv_slots, make_context, oracle_weights,
                      upload_kv, upload_weights)

pytestmark = pytest.mark.gpu


class Case:
    def __init__(self, cfg, norm="ones", lens=None, K=None, chain_stream=77, tc_min_batch=0, persistent_max_batch=0,
                 weight_format="dense"):
        self.cfg = cfg
        self.weight_format = weight_format
        self._W = None
        self.K = K or cfg.K
        self.w = synth.make_weights(cfg, norm=norm)
        self.lens = synth.context_lengths(cfg) if lens is None else np.asarray(lens, dtype=np.int32)
        self.B = len(self.lens)
        self.kv0 = synth.make_kv(cfg, self.lens, extra_slots=self.K + 3)
        self.di = synth.make_draft_inputs(cfg, self.w, self.lens)
        self.chain = synth.uniform_int(cfg.seed, chain_stream, (self.B, max(self.K - 1, 1)), 0, cfg.vocab)
        self.wdev = upload_weights(self.w)
        self.ctx = make_context(cfg, self.wdev, max_batch=self.B, max_k=self.K,
                                max_pos=int(self.lens.max()) + self.K + 8, tc_min_batch=tc_min_batch,
                                persistent_max_batch=persistent_max_batch, weight_format=weight_format)
        self.inputs = (dev(self.di.hidden), dev(self.di.embeds), dev(self.di.positions))

    def gpu_draft(self, forced=True, kvd=None):
        import mtp_self_speculative_gb300 as M
        cfg, B, K = self.cfg, self.B, self.K
        kvd = upload_kv(self.kv0) if kvd is None else kvd
        ids = Guarded((B, K), torch.int32, fill=-7)
        logits = Guarded((B, K, cfg.vocab), torch.float32)
        hout = Guarded((B, cfg.H), torch.float32)
        chain = dev(self.chain[:, :K - 1].copy()) if (forced and K > 1) else None
        M.mtp_draft(self.ctx, *self.inputs, kvd, K, ids.t, logits.t, hout.t, chain_ids=chain)
        torch.cuda.synchronize()
        assert M.mtp_get_device_error(self.ctx) == 0
        for g, name in ((ids, "draft_ids"), (logits, "logits"), (hout, "hidden_out")):
            g.check(name)
        ids_h, logits_h = host(ids.t), host(logits.t)
        check_ids_are_argmax_of_own_logits(ids_h, logits_h)
        return ids_h, logits_h, host(hout.t), kvd

    def oracle(self, subset, forced=True, kv=None):
        """Oracle draft on ``subset``; appends into ``kv`` (default: a copy of
        the initial cache)."""
        cfg = self.cfg
        if self._W is None:
            self._W = oracle_weights(cfg, self.w, self.weight_format)
        W = self._W
        kv = self.kv0.copy() if kv is None else kv
        view = synth.KVState(kv.k_pool, kv.v_pool, kv.block_table[subset], kv.seq_len[subset].copy(),
                             np.zeros(len(subset), dtype=np.int32), kv.block_size)
        chain = self.chain[subset, :self.K - 1] if (forced and self.K > 1) else None
        res = O.draft(W, O.widen(self.di.hidden[subset], cfg.dtype), O.widen(self.di.embeds[subset], cfg.dtype),
                      self.di.positions[subset], view, self.K, chain_ids=chain)
        return res, view


def check_forced(case, subset, tol, inplace=False):
    """Forced-chain parity on the requests in ``subset``.  ``inplace`` lets
    the oracle append into the initial cache itself (large caches; the case
    is not used afterwards)."""
    cfg, K = case.cfg, case.K
    ids, logits, hout, kvd = case.gpu_draft(forced=True)
    prefix = {b: kv_slots(case.kv0, b, 0, int(case.lens[b])) for b in subset}
    res, view = case.oracle(subset, forced=True, kv=case.kv0 if inplace else None)
    worst = check_logits(logits[subset], res.logits, tol)
    exact = check_ids(ids[subset], res.logits)
    n_steps = len(subset) * K
    assert exact >= (n_steps if tol <= F32_LOGIT_TOL else exact_floor(n_steps)), (exact, n_steps)
    e_h = np.max(np.abs(hout[subset] - res.hidden_out), axis=-1) / np.max(np.abs(res.hidden_out), axis=-1)
    assert np.max(e_h) <= tol
    got = download_kv(kvd)
    np.testing.assert_array_equal(got.seq_len, case.lens)
    np.testing.assert_array_equal(got.pending, K)
    for i, b in enumerate(subset):
        L = int(case.lens[b])
        gk, gv = kv_slots(got, b, 0, L + K)
        ok, ov = kv_slots(view, i, L, L + K)
        np.testing.assert_array_equal(gk[:L], prefix[b][0])
        np.testing.assert_array_equal(gv[:L], prefix[b][1])
        for g_app, o_app in ((gk[L:], ok), (gv[L:], ov)):
            a = O.widen(g_app, cfg.dtype)
            o = O.widen(o_app, cfg.dtype)
            err = np.max(np.abs(a - o), axis=-1) / np.maximum(np.max(np.abs(o), axis=-1), 1e-30)
            assert np.max(err) <= tol
        # the rest of the request's blocks stays zero
        nblk = (L + K + cfg.block_size - 1) // cfg.block_size
        tail = L + K
        cap = nblk * cfg.block_size
        if cap > tail:
            zk, zv = kv_slots(got, b, tail, cap)
            assert not zk.any() and not zv.any()
    return worst, exact, ids, logits


def check_free(case, subset, forced_ids, forced_logits, tol):
    """Free-running chain: step 1 equals the forced run bitwise; ids follow the
    oracle's own chain until the first near-tie."""
    ids, logits, _, _ = case.gpu_draft(forced=False)
    np.testing.assert_array_equal(ids[:, 0], forced_ids[:, 0])
    np.testing.assert_array_equal(logits[:, 0], forced_logits[:, 0])
    # a fresh copy of the initial KV for the oracle's own run
    kv = case.kv0.copy()
    res, _ = case.oracle(subset, forced=False, kv=kv)
    for i, b in enumerate(subset):
        for k in range(case.K):
            check_logits(logits[b, k][None], res.logits[i, k][None], tol)
            check_ids(ids[b, k][None], res.logits[i, k][None])
            if ids[b, k] != res.ids[i, k]:
                break            # legitimate near-tie: later steps follow different tokens


# ------------------------------------------------------------------ small

def test_tiny_f32_head_parity_and_invariants():
    """Tiny fp32 head (H=256, 4q/2kv, d=64, F=1024, V=4096, L=128, K=3) with
    non-unit norm weights so that a dropped norm weight shows."""
    import mtp_self_speculative_gb300 as M
    case = Case(synth.TINY_F32, norm="random")
    worst, exact, ids, logits = check_forced(case, [0], F32_LOGIT_TOL)
    check_free(case, [0], ids, logits, F32_LOGIT_TOL)
    # determinism: a second forced run is bitwise identical
    ids2, logits2, _, _ = case.gpu_draft(forced=True)
    np.testing.assert_array_equal(ids2, ids)
    np.testing.assert_array_equal(logits2, logits)
    # draft then full rollback leaves the cache bitwise as it was
    _, _, _, kvd = case.gpu_draft(forced=False)
    M.mtp_kv_rollback(case.ctx, kvd)
    got = download_kv(kvd)
    for f in ("k_pool", "v_pool", "seq_len", "pending"):
        np.testing.assert_array_equal(getattr(got, f), getattr(case.kv0, f), err_msg=f)


@pytest.mark.parametrize("path", ["cuda_cores", "tensor_cores"])
def test_ragged_bf16_block_edges(path):
    """bf16, G=4 heads per kv head, d=128, odd vocab; contexts 0, 1, 15, 16,
    17, 33 and 100 tokens (block boundaries, an empty cache).  Run on both
    the register-streaming CUDA-core kernels (B=7 in two groups of at most 4)
    and the tcgen05 path."""
    cfg = synth.MTPShape("ragged_bf16", H=512, n_q=8, n_kv=2, head_dim=128, ffn=1536, vocab=5003, batch=7, K=4,
                         dtype="bf16", ctx_lo=0, ctx_hi=100, paged_shuffle=True, seed_index=50)
    case = Case(cfg, norm="random", lens=[0, 1, 15, 16, 17, 33, 100],
                tc_min_batch=1 if path == "tensor_cores" else 1 << 20)
    _, _, ids, logits = check_forced(case, list(range(7)), LOGIT_TOL)
    check_free(case, list(range(7)), ids, logits, LOGIT_TOL)


@pytest.mark.parametrize("path", ["streamed", "persistent"])
@pytest.mark.parametrize("lens", [[33], [0, 17], [5, 16, 40], [1, 30, 2, 64]])
def test_small_batch_bf16(lens, path):
    """bf16 batches of 1..4 on both small-batch paths: the per-step
    TMA-streamed CUDA-core kernels (1, 2 and 4 batch rows per pass) and the
    persistent kernel that runs all K steps in one cooperative launch."""
    cfg = synth.MTPShape("small_bf16", H=512, n_q=8, n_kv=2, head_dim=128, ffn=1536, vocab=5003, batch=len(lens), K=3,
                         dtype="bf16", ctx_lo=0, ctx_hi=64, paged_shuffle=True, seed_index=53)
    case = Case(cfg, norm="random", lens=lens, persistent_max_batch=-1 if path == "streamed" else 4)
    _, _, ids, logits = check_forced(case, list(range(len(lens))), LOGIT_TOL)
    check_free(case, list(range(len(lens))), ids, logits, LOGIT_TOL)
    ids2, logits2, _, _ = case.gpu_draft(forced=True)
    np.testing.assert_array_equal(ids2, ids)
    np.testing.assert_array_equal(logits2, logits)


@pytest.mark.parametrize("path", ["streamed", "persistent"])
def test_small_batch_multi_chunk_rows(path):
    """Rows wider than one 4096-column chunk in every projection (H = 4608,
    q_dim = 6144, F = 9216: RMSNorm statistics over several chunks, partial
    sums carried across chunks), 8 query heads per kv head, K = 3, B = 2."""
    cfg = synth.MTPShape("wide_bf16", H=4608, n_q=48, n_kv=6, head_dim=128, ffn=9216, vocab=20001, batch=2, K=3,
                         dtype="bf16", ctx_lo=1, ctx_hi=200, paged_shuffle=True, seed_index=54)
    case = Case(cfg, norm="random", lens=[200, 37], persistent_max_batch=-1 if path == "streamed" else 4)
    _, _, ids, logits = check_forced(case, [0, 1], LOGIT_TOL)
    check_free(case, [0, 1], ids, logits, LOGIT_TOL)


def test_tensor_core_path_batch_40_gqa8():
    """tcgen05 path with N = 48 (40 requests padded), 8 q heads per kv head,
    a vocabulary that ends mid-tile, and more tiles than SMs in the LM head."""
    cfg = synth.MTPShape("tc_b40", H=768, n_q=16, n_kv=2, head_dim=128, ffn=2048, vocab=40000, batch=40, K=3,
                         dtype="bf16", ctx_lo=1, ctx_hi=300, paged_shuffle=True, seed_index=52)
    case = Case(cfg, norm="random")
    _, _, ids, logits = check_forced(case, list(range(40)), LOGIT_TOL)
    check_free(case, [0, 13, 39], ids, logits, LOGIT_TOL)
    ids2, logits2, _, _ = case.gpu_draft(forced=True)
    np.testing.assert_array_equal(ids2, ids)
    np.testing.assert_array_equal(logits2, logits)


def test_gqa_eight_heads_per_kv_head_f32():
    cfg = synth.MTPShape("gqa8_f32", H=256, n_q=16, n_kv=2, head_dim=64, ffn=512, vocab=2048, batch=3, K=2,
                         dtype="f32", ctx_lo=40, ctx_hi=300, seed_index=51)
    case = Case(cfg, norm="random")
    check_forced(case, [0, 1, 2], F32_LOGIT_TOL)


@pytest.mark.parametrize("path", ["streamed", "persistent", "tensor_cores"])
def test_device_errors_bf16(path):
    """pending != 0 on entry and a block table that is too short are reported
    through the error word; the request's cache is left untouched at every
    step (a request that starts with pending != 0 is never appended to), and
    the context drafts correctly afterwards."""
    import mtp_self_speculative_gb300 as M
    cfg = synth.MTPShape("err_bf16", H=512, n_q=8, n_kv=2, head_dim=128, ffn=1536, vocab=5003, batch=2, K=3,
                         dtype="bf16", ctx_lo=150, ctx_hi=200, seed_index=55)
    case = Case(cfg, norm="random", persistent_max_batch=4 if path == "persistent" else -1,
                tc_min_batch=1 if path == "tensor_cores" else 1 << 20)
    ids = torch.empty((2, 3), dtype=torch.int32, device="cuda")
    kv = case.kv0.copy()
    kv.pending[:] = 1
    kvd = upload_kv(kv)
    M.mtp_draft(case.ctx, *case.inputs, kvd, 3, ids)
    assert M.mtp_get_device_error(case.ctx) == M.MTP_ERR_DEVICE_ARGS
    got = download_kv(kvd)
    np.testing.assert_array_equal(got.k_pool, kv.k_pool)
    np.testing.assert_array_equal(got.v_pool, kv.v_pool)
    np.testing.assert_array_equal(got.pending, kv.pending)
    kv = case.kv0.copy()
    kv.block_table = kv.block_table[:, :8].copy()      # room for 128 slots only
    kvd = upload_kv(kv)
    M.mtp_draft(case.ctx, *case.inputs, kvd, 3, ids)
    assert M.mtp_get_device_error(case.ctx) == M.MTP_ERR_CAPACITY
    got = download_kv(kvd)
    np.testing.assert_array_equal(got.k_pool, kv.k_pool)
    # the context still drafts correctly afterwards
    check_forced(case, [0, 1], LOGIT_TOL)


def test_device_errors_leave_no_fault():
    """pending != 0 on entry and a block table too short are reported through
    the error word; the writes are skipped."""
    import mtp_self_speculative_gb300 as M
    cfg = synth.TINY_F32
    case = Case(cfg)
    kv = case.kv0.copy()
    kv.pending[:] = 1
    kvd = upload_kv(kv)
    ids = torch.empty((1, 3), dtype=torch.int32, device="cuda")
    M.mtp_draft(case.ctx, *case.inputs, kvd, 3, ids)
    assert M.mtp_get_device_error(case.ctx) == M.MTP_ERR_DEVICE_ARGS
    got = download_kv(kvd)
    np.testing.assert_array_equal(got.k_pool, kv.k_pool)
    np.testing.assert_array_equal(got.pending, kv.pending)
    kv = case.kv0.copy()
    kv.block_table = kv.block_table[:, :8].copy()      # room for 128 slots only
    kvd = upload_kv(kv)
    M.mtp_draft(case.ctx, *case.inputs, kvd, 3, ids)
    assert M.mtp_get_device_error(case.ctx) == M.MTP_ERR_CAPACITY
    got = download_kv(kvd)
    np.testing.assert_array_equal(got.k_pool, kv.k_pool)


# ------------------------------------------------------------- full sizes

@pytest.mark.slow
@pytest.mark.parametrize("path", ["streamed", "persistent"])
def test_qwen3_8b_b1_full_size(path):
    """Qwen3-8B-shaped head, bf16, B=1, context 4096, K=5 -- the bench's
    workload and launch configuration (streamed per-step kernels), and the
    same on the persistent kernel."""
    case = Case(synth.QWEN3_8B_B1, persistent_max_batch=4 if path == "persistent" else 0)
    worst, exact, ids, logits = check_forced(case, [0], LOGIT_TOL)
    check_free(case, [0], ids, logits, LOGIT_TOL)


@pytest.mark.slow
@pytest.mark.parametrize("B", [2, 3, 4])
def test_qwen3_8b_small_batch_full_size(B):
    """Qwen3-8B-shaped head at 2, 3 and 4 requests (tree expansions, small
    batches), bf16, ragged paged contexts, K=3: the tensor-core short
    projections at their real chunking (4096- and 2048-column chunks, eh_proj
    accumulating its two halves apart, a 4-request tile with one empty row at
    B=3) and the tensor-core LM head; every request checked."""
    import dataclasses
    cfg = dataclasses.replace(synth.QWEN3_8B_B1, name="qwen3_8b_mtp_b%d" % B, batch=B, K=3, ctx_lo=1, ctx_hi=4096,
                              paged_shuffle=True, seed_index=57)
    case = Case(cfg, lens=[4096, 1, 2500, 17][:B], persistent_max_batch=-1)
    worst, exact, ids, logits = check_forced(case, list(range(B)), LOGIT_TOL)
    check_free(case, list(range(B)), ids, logits, LOGIT_TOL)


@pytest.mark.slow
def test_qwen3_8b_cb32_ragged_paged():
    """Continuous batching: B=32, contexts uniform in 512..8192 in shuffled
    16-token blocks, K=5; every request checked."""
    case = Case(synth.QWEN3_8B_CB32)
    check_forced(case, list(range(32)), LOGIT_TOL, inplace=True)


@pytest.mark.slow
def test_qwen3_32b_b128_sampled():
    """Qwen3-32B-shaped head, B=128, context 16384 each, K=3: the whole batch
    runs on the GPU; a seeded sample of 8 requests is checked against the
    oracle (requests are independent given the shared weights)."""
    case = Case(synth.QWEN3_32B_B128)
    subset = sorted(set(synth.uniform_int(case.cfg.seed, 88, (8,), 0, 128).tolist()))
    check_forced(case, subset, LOGIT_TOL, inplace=True)


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_runs_out_and_reports_timeout(which):
    """A bounded wait whose condition never comes true (a shared-memory
    barrier nobody arrives at; a grid-barrier counter nobody increments)
    gives up, reports MTP_ERR_TIMEOUT through the error word, and leaves the
    context usable: the error reads once, then the head drafts correctly."""
    import time
    import mtp_self_speculative_gb300 as M
    case = Case(synth.TINY_F32)
    t = time.perf_counter()
    M.mtp_selftest_wait_timeout(case.ctx, which)
    assert M.mtp_get_device_error(case.ctx) == M.MTP_ERR_TIMEOUT
    elapsed = time.perf_counter() - t
    assert elapsed < 30.0
    if which == 1:
        assert elapsed >= 1.9          # the counter wait is bounded by 2 s of the GPU timer
    assert M.mtp_get_device_error(case.ctx) == 0
    check_forced(case, [0], F32_LOGIT_TOL)



@pytest.mark.parametrize("n_q", [8, 16, 32])
def test_long_context_small_batch_split_combine_bf16(n_q):
    """Contexts of 2500 and 3001 tokens at B = 2 with 2, 4 and 8 query heads
    per kv head: the tensor-core attention splits each (request, kv head)
    over many CTAs and merges the splits (several lanes per output item for
    2 and 4 heads per kv head), on both small-batch paths' step kernels."""
    cfg = synth.MTPShape("long_ctx_bf16", H=1024, n_q=n_q, n_kv=4, head_dim=128, ffn=2048, vocab=5003, batch=2,
                         K=3, dtype="bf16", ctx_lo=2500, ctx_hi=3001, paged_shuffle=True, seed_index=56)
    case = Case(cfg, norm="random", lens=[3001, 2500], persistent_max_batch=-1)
    _, _, ids, logits = check_forced(case, [0, 1], LOGIT_TOL)
    check_free(case, [0, 1], ids, logits, LOGIT_TOL)



@pytest.mark.parametrize("B", [1, 4, 24])
def test_lm_head_weighted_ranges_are_bit_identical(B, monkeypatch):
    """The 1-4-request LM heads size each CTA's range of vocabulary rows by
    its SM's measured streaming rate, claimed through a packed (ticket, next
    unit) counter.  Every logit is one warp's (1 request) or one tile
    column's (2-4 requests) dot product whichever CTA owns its row, so
    repeated drafts -- whose ranges change as the rate table settles -- and
    drafts over equal ranges give the same logits and ids bit for bit, and
    both match the oracle.  The tcgen05 LM head (24 requests) takes equal
    ranges in 16-row units, so a CTA's last 128-row tile is often short and
    its unused accumulator rows hold stale stage data that must not reach
    the argmax.  60001 rows give every CTA many units and a last unit of one
    row."""
    cfg = synth.MTPShape("balance_bf16", H=512, n_q=8, n_kv=2, head_dim=128, ffn=1536, vocab=60001, batch=B, K=3,
                         dtype="bf16", ctx_lo=40, ctx_hi=90, seed_index=58)
    got = {}
    for bal in ("1", "0"):
        monkeypatch.setenv("MTP_LM_BALANCE", bal)
        case = Case(cfg, norm="random", persistent_max_batch=-1, tc_min_batch=1 if B > 4 else 0)
        _, _, ids, logits = check_forced(case, list(range(B)), LOGIT_TOL)
        for _ in range(3):
            ids2, logits2, _, _ = case.gpu_draft(forced=True)
            np.testing.assert_array_equal(ids2, ids)
            np.testing.assert_array_equal(logits2, logits)
        got[bal] = (ids, logits)
    np.testing.assert_array_equal(got["1"][0], got["0"][0])
    np.testing.assert_array_equal(got["1"][1], got["0"][1])


@pytest.mark.parametrize("dtype,vocab", [("bf16", 60001), ("bf16", 201), ("f32", 4099)])
def test_deferred_argmax_matches_last_cta_argmax(dtype, vocab, monkeypatch):
    """One request: in every step but the last the LM head leaves one argmax
    key per CTA and the next step's eh_proj reduces them (writing the draft
    id and the pending count itself).  Forced and free-running drafts give
    the same ids, logits, hidden rows and cache as the LM head's own last-CTA
    argmax, bit for bit, and match the oracle.  201 rows launch fewer CTAs
    than there are SMs."""
    cfg = synth.MTPShape("defer_" + dtype, H=512, n_q=8, n_kv=2, head_dim=128, ffn=1536, vocab=vocab, batch=1, K=5,
                         dtype=dtype, ctx_lo=40, ctx_hi=90, seed_index=61)
    import mtp_self_speculative_gb300 as M
    tol = F32_LOGIT_TOL if dtype == "f32" else LOGIT_TOL
    got = {}
    for defer in ("1", "0"):
        monkeypatch.setenv("MTP_LM_DEFER", defer)
        case = Case(cfg, norm="random", persistent_max_batch=-1)
        _, _, ids, logits = check_forced(case, [0], tol)
        check_free(case, [0], ids, logits, tol)
        free = case.gpu_draft(forced=False)
        got[defer] = (ids, logits, free[0], free[1], free[2], download_kv(free[3]))
        # every draft call (forced, free, free again: three) defers K-1 of
        # its K steps, or none
        deferred = M.mtp_path_count(case.ctx, M.MTP_PATH_LM_DEFERRED)
        assert deferred == (3 * (cfg.K - 1) if defer == "1" else 0), deferred
    a, b = got["1"], got["0"]
    for x, y in zip(a[:5], b[:5]):
        np.testing.assert_array_equal(x, y)
    for f in ("k_pool", "v_pool", "seq_len", "pending"):
        np.testing.assert_array_equal(getattr(a[5], f), getattr(b[5], f), err_msg=f)


@pytest.mark.parametrize("cluster", ["1", "0"])
@pytest.mark.parametrize("n_q,lens", [(8, [200]), (8, [200, 0, 37]), (16, [150, 3]), (2, [90, 180])])
def test_attention_split_combine_in_a_cluster(cluster, n_q, lens, monkeypatch, capfd):
    """One block per split (up to 14 splits) so that every request's splits
    form one thread-block cluster that combines them through distributed
    shared memory (cluster=1), or write partials to HBM for the last CTA
    (cluster=0).  Requests of 0+k and 3+k tokens leave most CTAs of their
    cluster without blocks; G = 4, 8 and 1 query heads per kv head.  Both
    forms match the oracle.  The plan trace shows which form ran: with at
    most four clusters needed they all fit on the GPU at once, so the cluster
    form is the one tested."""
    monkeypatch.setenv("MTP_ATTN_CLUSTER", cluster)
    monkeypatch.setenv("MTP_ATTN_BPS", "1")
    monkeypatch.setenv("MTP_ATTN_TRACE", "1")
    cfg = synth.MTPShape("cluster_bf16", H=512, n_q=n_q, n_kv=2, head_dim=128, ffn=1536, vocab=5003,
                         batch=len(lens), K=3, dtype="bf16", ctx_lo=0, ctx_hi=200, seed_index=62)
    case = Case(cfg, norm="random", lens=lens, persistent_max_batch=-1)
    subset = list(range(len(lens)))
    _, _, ids, logits = check_forced(case, subset, LOGIT_TOL)
    check_free(case, subset, ids, logits, LOGIT_TOL)
    import mtp_self_speculative_gb300 as M
    launched = M.mtp_path_count(case.ctx, M.MTP_PATH_ATTN_CLUSTER)
    plans = [ln for ln in capfd.readouterr().err.splitlines() if ln.startswith("attention cluster:")]
    if cluster == "0":
        assert not plans and launched == 0
    else:
        assert plans, "no attention cluster plan was made"
        fit, needed = (int(w) for w in re.findall(r"(\d+) clusters fit, (\d+) needed", plans[-1])[0])
        assert (launched > 0) == (fit >= needed), (launched, plans[-1])
        if needed <= 4:
            assert launched > 0, plans[-1]
