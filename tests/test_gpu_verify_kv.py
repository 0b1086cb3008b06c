"""GPU verification and KV edits vs the oracle: bit-exact accepted counts,
bonus ids, pools, lengths.  Calls go through the C ABI."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from gpu_util import Guarded, dev, download_kv, host, make_context, upload_kv

pytestmark = pytest.mark.gpu


def _verify_gpu(ctx, vi, B):
    import mtp_self_speculative_gb300 as M
    acc = Guarded((B,), torch.int32, fill=-9)
    bon = Guarded((B,), torch.int32, fill=-9)
    M.mtp_verify(ctx, dev(vi.logits), dev(vi.row_offsets), dev(vi.drafts), dev(vi.num_drafts), acc.t, bon.t)
    torch.cuda.synchronize()
    assert M.mtp_get_device_error(ctx) == 0
    acc.check("accepted")
    bon.check("bonus")
    return host(acc.t), host(bon.t)


def test_verify_rollback_b64_bit_exact():
    """64 requests, K_b uniform in 1..8, bf16 [rows, 151936] logits with a +8
    spike per row; drafts copy the spikes for a geometric(0.8) prefix."""
    cfg = synth.VERIFY_B64
    vi = synth.make_verify_inputs(cfg)
    ctx = make_context(cfg, None, max_batch=cfg.batch, max_k=vi.max_k)
    acc, bon = _verify_gpu(ctx, vi, cfg.batch)
    acc_o, bon_o = O.verify(vi.logits, vi.row_offsets, vi.drafts, vi.num_drafts, "bf16")
    np.testing.assert_array_equal(acc, acc_o)
    np.testing.assert_array_equal(bon, bon_o)
    # the recipe's planted prefix is what the oracle accepts (spikes dominate)
    assert np.mean(acc_o == vi.accept_len) > 0.95


def test_verify_tiny_f32_many_seeds():
    """Tiny fp32 head: logits [1, 4, 4096], prefix length uniform over 0..3."""
    cfg = synth.TINY_F32
    ctx = make_context(cfg, None, max_batch=1, max_k=3)
    seen = set()
    for seed in range(40):
        vi = synth.make_verify_inputs(cfg, num_drafts=np.array([3]), seed=1000 + seed, len_mode="uniform")
        acc, bon = _verify_gpu(ctx, vi, 1)
        acc_o, bon_o = O.verify(vi.logits, vi.row_offsets, vi.drafts, vi.num_drafts, "f32")
        np.testing.assert_array_equal(acc, acc_o)
        np.testing.assert_array_equal(bon, bon_o)
        seen.add(int(acc_o[0]))
    assert seen == {0, 1, 2, 3}


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_verify_edges_unaligned_vocab_zero_drafts_and_ties(dtype):
    cfg = synth.MTPShape("edge", H=0, n_q=2, n_kv=2, head_dim=64, ffn=0, vocab=1001, batch=7, K=6, dtype=dtype,
                         ctx_lo=1, ctx_hi=1, seed_index=40)
    nd = np.array([0, 1, 6, 3, 0, 5, 2], dtype=np.int32)
    vi = synth.make_verify_inputs(cfg, num_drafts=nd)
    # plant exact ties in some rows: the lowest id must win
    lg = vi.logits.copy()
    lg[0, 17] = lg[0, 900] = lg[0, vi.planted[0]]
    lg[3, 1000] = lg[3, vi.planted[3]]
    vi.logits = lg
    ctx = make_context(cfg, None, max_batch=cfg.batch, max_k=6)
    acc, bon = _verify_gpu(ctx, vi, cfg.batch)
    acc_o, bon_o = O.verify(vi.logits, vi.row_offsets, vi.drafts, vi.num_drafts, dtype)
    np.testing.assert_array_equal(acc, acc_o)
    np.testing.assert_array_equal(bon, bon_o)
    # all drafts equal the argmax rows -> K_b accepted + bonus of row K_b
    r = O.argmax_lowest(O.widen(vi.logits, dtype))
    full = np.full_like(vi.drafts, -1)
    for b in range(cfg.batch):
        full[b, :nd[b]] = r[vi.row_offsets[b]:vi.row_offsets[b] + nd[b]]
    vi.drafts = full
    acc, bon = _verify_gpu(ctx, vi, cfg.batch)
    np.testing.assert_array_equal(acc, nd)
    np.testing.assert_array_equal(bon, r[vi.row_offsets[1:] - 1])


def _adversarial_rows(V, dtype, seed):
    """Rows that stress the argmax scan: a constant row, a row of -inf, -0/+0
    as the maximum in both orders, the maximum repeated at spread-out ids,
    record-breaking values at every 1000th id, a maximum in the first and in
    the last element, and plain normal rows.  Seeded numpy, float64 values
    exact in the stored dtype."""
    rng = np.random.default_rng(seed)
    rows = []
    rows.append(np.full(V, 0.5))
    rows.append(np.full(V, -np.inf))
    r = -1.0 - rng.random(V); r[V // 2] = -0.0; r[3] = 0.0; rows.append(r)
    r = -1.0 - rng.random(V); r[V - 7] = 0.0; r[101] = -0.0; rows.append(r)
    r = rng.standard_normal(V); at = rng.choice(V, 9, replace=False); r[at] = 6.0; rows.append(r)
    r = rng.standard_normal(V) - 10.0; r[::1000] = np.arange(len(r[::1000])) * 0.25; rows.append(r)
    r = rng.standard_normal(V); r[0] = 9.0; rows.append(r)
    r = rng.standard_normal(V); r[V - 1] = 9.0; rows.append(r)
    while len(rows) < 24:
        rows.append(rng.standard_normal(V))
    z = np.stack(rows)
    if dtype == "bf16":
        return synth.f32_to_bf16_bits(z.astype(np.float32))
    return z.astype(np.float32)


@pytest.mark.parametrize("dtype,V", [("bf16", 151936), ("f32", 151936), ("bf16", 40009), ("f32", 1001)])
def test_verify_adversarial_rows_all_accepted(dtype, V):
    """Every row's argmax is observed: the drafts are the oracle's argmaxes,
    so the GPU accepts all K_b drafts only if every row agrees.  The rows
    ([24, V], odd V gives misaligned row starts) are cut by the flat split of
    the scan at many points inside rows."""
    import mtp_self_speculative_gb300 as M
    lg = _adversarial_rows(V, dtype, seed=77 + V)
    nd = np.array([4, 0, 7, 2, 6], dtype=np.int32)           # 24 rows
    ro = np.concatenate([[0], np.cumsum(nd + 1)]).astype(np.int32)
    r = O.argmax_lowest(O.widen(lg, dtype))
    assert r[0] == 0 and r[1] == 0 and r[2] == 3 and r[3] == 101
    drafts = np.full((len(nd), 8), -1, dtype=np.int32)
    for b in range(len(nd)):
        drafts[b, :nd[b]] = r[ro[b]:ro[b] + nd[b]]
    cfg = synth.MTPShape("adv", H=0, n_q=2, n_kv=2, head_dim=64, ffn=0, vocab=V, batch=len(nd), K=8,
                         dtype=dtype, ctx_lo=1, ctx_hi=1, seed_index=41)
    ctx = make_context(cfg, None, max_batch=len(nd), max_k=8)
    acc = Guarded((len(nd),), torch.int32, fill=-9)
    bon = Guarded((len(nd),), torch.int32, fill=-9)
    M.mtp_verify(ctx, dev(lg), dev(ro), dev(drafts), dev(nd), acc.t, bon.t)
    torch.cuda.synchronize()
    assert M.mtp_get_device_error(ctx) == 0
    acc.check("accepted")
    bon.check("bonus")
    acc_o, bon_o = O.verify(lg, ro, drafts, nd, dtype)
    np.testing.assert_array_equal(acc_o, nd)
    np.testing.assert_array_equal(host(acc.t), acc_o)
    np.testing.assert_array_equal(host(bon.t), bon_o)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_verify_nan_entries_are_passed_over(dtype):
    """NaN logits are not candidates (the library's stated behaviour; the
    pages never meet NaN): the argmax is that of the other entries, and a row
    of NaN only gives r = -1."""
    import mtp_self_speculative_gb300 as M
    V = 3000
    z = np.zeros((3, V))
    z[0, :] = np.nan
    z[1, :] = -1.0; z[1, 0] = np.nan; z[1, 2999] = np.nan; z[1, 1234] = 2.0; z[1, 1500:1600] = np.nan
    z[2, :] = -2.0; z[2, 7] = np.nan; z[2, 2048] = 0.5
    lg = synth.f32_to_bf16_bits(z.astype(np.float32)) if dtype == "bf16" else z.astype(np.float32)
    nd = np.array([0, 1], dtype=np.int32)      # request 0: row 0; request 1: rows 1, 2
    ro = np.array([0, 1, 3], dtype=np.int32)
    drafts = np.array([[-1], [1234]], dtype=np.int32)
    cfg = synth.MTPShape("nan", H=0, n_q=2, n_kv=2, head_dim=64, ffn=0, vocab=V, batch=2, K=1,
                         dtype=dtype, ctx_lo=1, ctx_hi=1, seed_index=42)
    ctx = make_context(cfg, None, max_batch=2, max_k=1)
    acc = Guarded((2,), torch.int32, fill=-9)
    bon = Guarded((2,), torch.int32, fill=-9)
    M.mtp_verify(ctx, dev(lg), dev(ro), dev(drafts), dev(nd), acc.t, bon.t)
    torch.cuda.synchronize()
    acc.check("accepted")
    bon.check("bonus")
    np.testing.assert_array_equal(host(acc.t), [0, 1])
    np.testing.assert_array_equal(host(bon.t), [-1, 2048])
    assert M.mtp_get_device_error(ctx) == 0


def test_verify_inconsistent_offsets_sets_error():
    import mtp_self_speculative_gb300 as M
    cfg = synth.shrink(synth.VERIFY_B64, vocab=512, batch=4)
    vi = synth.make_verify_inputs(cfg)
    ro = vi.row_offsets.copy()
    ro[2] += 1                          # request 1 claims one row too many
    ctx = make_context(cfg, None, max_batch=4, max_k=vi.max_k)
    acc = Guarded((4,), torch.int32, fill=-9)
    bon = Guarded((4,), torch.int32, fill=-9)
    M.mtp_verify(ctx, dev(vi.logits), dev(ro), dev(vi.drafts), dev(vi.num_drafts), acc.t, bon.t)
    assert M.mtp_get_device_error(ctx) == M.MTP_ERR_DEVICE_ARGS
    assert host(acc.t)[1] == -1 and host(bon.t)[1] == -1
    acc.check("accepted")
    bon.check("bonus")
    assert M.mtp_get_device_error(ctx) == 0     # cleared


def _drafted_kv(cfg, num_drafts):
    """KV with seq_len committed entries plus num_drafts[b] drafted ones."""
    lens = synth.context_lengths(cfg)
    kv = synth.make_kv(cfg, lens, extra_slots=int(num_drafts.max()) + 1, prefill_slots=lens + num_drafts)
    kv.pending = num_drafts.astype(np.int32).copy()
    return kv


def test_commit_after_verify_b64_bit_exact():
    import mtp_self_speculative_gb300 as M
    cfg = synth.VERIFY_B64
    vi = synth.make_verify_inputs(cfg)
    kv0 = _drafted_kv(cfg, vi.num_drafts)
    kvd = upload_kv(kv0)
    ctx = make_context(cfg, None, max_batch=cfg.batch, max_k=vi.max_k)
    acc = Guarded((cfg.batch,), torch.int32, fill=-9)
    bon = Guarded((cfg.batch,), torch.int32, fill=-9)
    M.mtp_verify(ctx, dev(vi.logits), dev(vi.row_offsets), dev(vi.drafts), dev(vi.num_drafts), acc.t, bon.t)
    M.mtp_kv_commit_accepted(ctx, kvd, acc.t, extra=1)
    torch.cuda.synchronize()
    assert M.mtp_get_device_error(ctx) == 0
    acc.check("accepted")
    bon.check("bonus")
    got = download_kv(kvd)
    acc_o, _ = O.verify(vi.logits, vi.row_offsets, vi.drafts, vi.num_drafts, "bf16")
    kv_o = kv0.copy()
    O.kv_commit(kv_o, np.minimum(acc_o + 1, vi.num_drafts), "bf16")
    np.testing.assert_array_equal(got.seq_len, kv_o.seq_len)
    np.testing.assert_array_equal(got.pending, kv_o.pending)
    np.testing.assert_array_equal(got.k_pool, kv_o.k_pool)
    np.testing.assert_array_equal(got.v_pool, kv_o.v_pool)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_commit_rollback_truncate_bit_exact(dtype):
    import mtp_self_speculative_gb300 as M
    cfg = synth.MTPShape("kv", H=0, n_q=4, n_kv=2, head_dim=64 if dtype == "f32" else 128, ffn=0, vocab=64,
                         batch=6, K=7, dtype=dtype, ctx_lo=0, ctx_hi=40, paged_shuffle=True, seed_index=41)
    nd = np.array([0, 1, 7, 3, 7, 2], dtype=np.int32)
    kv0 = _drafted_kv(cfg, nd)
    ctx = make_context(cfg, None, max_batch=6, max_k=7)
    n_keep = np.array([0, 1, 4, 3, 7, 0], dtype=np.int32)
    kvd = upload_kv(kv0)
    M.mtp_kv_commit(ctx, kvd, dev(n_keep))
    torch.cuda.synchronize()
    assert M.mtp_get_device_error(ctx) == 0
    kv_o = kv0.copy()
    O.kv_commit(kv_o, n_keep, dtype)
    got = download_kv(kvd)
    for f in ("k_pool", "v_pool", "seq_len", "pending"):
        np.testing.assert_array_equal(getattr(got, f), getattr(kv_o, f), err_msg=f)
    # rollback: everything drafted disappears
    kvd = upload_kv(kv0)
    M.mtp_kv_rollback(ctx, kvd)
    kv_o = kv0.copy()
    O.kv_rollback(kv_o, dtype)
    got = download_kv(kvd)
    for f in ("k_pool", "v_pool", "seq_len", "pending"):
        np.testing.assert_array_equal(getattr(got, f), getattr(kv_o, f), err_msg=f)
    # truncate to a shorter common prefix
    kvd = upload_kv(kv0)
    new_len = np.maximum(kv0.seq_len - 5, 0).astype(np.int32)
    M.mtp_kv_truncate(ctx, kvd, dev(new_len))
    kv_o = kv0.copy()
    O.kv_truncate(kv_o, new_len, dtype)
    got = download_kv(kvd)
    for f in ("k_pool", "v_pool", "seq_len", "pending"):
        np.testing.assert_array_equal(getattr(got, f), getattr(kv_o, f), err_msg=f)
    assert M.mtp_get_device_error(ctx) == 0


def test_commit_more_than_pending_is_rejected_on_device():
    import mtp_self_speculative_gb300 as M
    cfg = synth.MTPShape("kv", H=0, n_q=2, n_kv=2, head_dim=64, ffn=0, vocab=64, batch=2, K=3, dtype="bf16",
                         ctx_lo=5, ctx_hi=5, seed_index=42)
    nd = np.array([2, 2], dtype=np.int32)
    kv0 = _drafted_kv(cfg, nd)
    kvd = upload_kv(kv0)
    ctx = make_context(cfg, None, max_batch=2, max_k=3)
    M.mtp_kv_commit(ctx, kvd, dev(np.array([1, 3], dtype=np.int32)))
    assert M.mtp_get_device_error(ctx) == M.MTP_ERR_DEVICE_ARGS
    got = download_kv(kvd)
    assert list(got.seq_len) == [6, 5] and list(got.pending) == [0, 2]   # request 1 untouched
