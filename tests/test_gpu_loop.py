"""The speculative loop on the GPU (draft -> synthetic verifier -> verify ->
commit -> advance, all enqueued by mtp_spec_loop) against the oracle's loop
and against plain greedy decoding with the same verifier ("How OpenVINO MTP
Speculative Decoding Works Internally": the speculative result equals the
main model's greedy result).  Token ids, accepted counts, positions and
prefix hashes are compared exactly; the synthetic verifier's rows and the
state advance bit for bit."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import loop as L
import synth
from gpu_util import dev, host, make_context, upload_kv, upload_weights

pytestmark = pytest.mark.gpu


def as_i64(u: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u, dtype=np.uint64).view(np.int64)).cuda()


def stored_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    return O.bf16_bits_of(x) if dtype == "bf16" else x.astype(np.float32)


def widen_gpu(t: torch.Tensor, dtype: str) -> np.ndarray:
    return O.widen(host(t), dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_synth_target_rows_bit_exact(dtype):
    import mtp_self_speculative_gb300 as M
    cfg = synth.MTPShape("st_rows", H=256, n_q=4, n_kv=2, head_dim=64, ffn=512, vocab=5003, batch=3, K=4,
                         dtype=dtype, ctx_lo=4, ctx_hi=4, seed_index=71)
    ctx = make_context(cfg, None)
    B, K = 3, 4
    h = synth.loop_start_hashes(cfg, B)
    last = synth.uniform_int(cfg.seed, 98, (B,), 0, cfg.vocab)
    drafts = synth.uniform_int(cfg.seed, 97, (B, K), 0, cfg.vocab)
    drafts[0, :] = last[0]                   # a request whose drafts repeat its last token
    thr = int(0.6 * 2 ** 53)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    for k in (K, 0):
        logits = torch.empty((B * (k + 1), cfg.vocab), dtype=tdt, device="cuda")
        offs = torch.empty(B + 1, dtype=torch.int32, device="cuda")
        M.mtp_synth_target(ctx, as_i64(h), dev(last), dev(drafts[:, :k].copy()) if k else None, k, thr, logits, offs)
        got = widen_gpu(logits, dtype)
        np.testing.assert_array_equal(host(offs), np.arange(B + 1) * (k + 1))
        for b in range(B):
            hh, ll = int(h[b]), int(last[b])
            for j in range(k + 1):
                if j:
                    hh, ll = L.fold(hh, int(drafts[b, j - 1])), int(drafts[b, j - 1])
                np.testing.assert_array_equal(got[b * (k + 1) + j], L.target_row(hh, ll, thr, cfg.vocab, dtype))


def test_loop_advance_bit_exact():
    import mtp_self_speculative_gb300 as M
    cfg = synth.MTPShape("adv", H=512, n_q=8, n_kv=2, head_dim=64, ffn=512, vocab=3001, batch=3, K=3,
                         dtype="bf16", ctx_lo=4, ctx_hi=4, seed_index=72)
    w = synth.make_weights(cfg)
    ctx = make_context(cfg, upload_weights(w))
    B, K, cap = 3, 3, 6
    h = synth.loop_start_hashes(cfg, B)
    drafts = synth.uniform_int(cfg.seed, 96, (B, K), 0, cfg.vocab)
    acc = np.array([0, 3, 1], dtype=np.int32)
    bonus = np.array([5, 3000, 17], dtype=np.int32)
    out_len0 = np.array([0, 4, 2], dtype=np.int32)       # request 1 overflows its 6-token buffer
    pos0 = np.array([10, 20, 30], dtype=np.int32)
    t = dict(seq_hash=as_i64(h), last_tok=dev(np.zeros(B, np.int32)), positions=dev(pos0),
             hidden=torch.zeros((B, cfg.H), dtype=torch.bfloat16, device="cuda"),
             embeds=torch.zeros((B, cfg.H), dtype=torch.bfloat16, device="cuda"),
             out_tokens=torch.full((B, cap), -1, dtype=torch.int32, device="cuda"), out_len=dev(out_len0))
    M.mtp_loop_advance(ctx, K, dev(drafts), dev(acc), dev(bonus), **t)
    assert M.mtp_get_device_error(ctx) == M.MTP_ERR_CAPACITY
    out = host(t["out_tokens"])
    for b in range(B):
        emitted = [int(x) for x in drafts[b, :acc[b]]] + [int(bonus[b])]
        hh = int(h[b])
        for x in emitted:
            hh = L.fold(hh, x)
        assert int(host(t["seq_hash"]).view(np.uint64)[b]) == hh
        assert int(host(t["last_tok"])[b]) == bonus[b]
        assert int(host(t["positions"])[b]) == pos0[b] + acc[b] + 1
        assert int(host(t["out_len"])[b]) == out_len0[b] + len(emitted)
        n0 = int(out_len0[b])
        keep = emitted[:max(0, cap - n0)]
        np.testing.assert_array_equal(out[b, n0:n0 + len(keep)], keep)
        np.testing.assert_array_equal(host(t["hidden"])[b], O.bf16_bits_of(L.target_hidden(hh, cfg.H, "bf16")))
        np.testing.assert_array_equal(host(t["embeds"])[b], w["embed"][bonus[b]])
    # an accepted count past K leaves the request unchanged and reports it
    M.mtp_loop_advance(ctx, K, dev(drafts), dev(np.array([4, 0, 0], np.int32)), dev(bonus), **t)
    assert M.mtp_get_device_error(ctx) == M.MTP_ERR_DEVICE_ARGS


def _run_loop(cfg, w, K, iters, thr, weight_format="dense", lens=None):
    """GPU loop and oracle loop from the same start; returns both states."""
    import mtp_self_speculative_gb300 as M
    lens = synth.context_lengths(cfg) if lens is None else np.asarray(lens, dtype=np.int32)
    B = len(lens)
    kv0 = synth.make_kv(cfg, lens, extra_slots=K * iters + K + 1)
    h0 = synth.loop_start_hashes(cfg, B)
    last0 = synth.uniform_int(cfg.seed, 95, (B,), 0, cfg.vocab)
    ctx = make_context(cfg, upload_weights(w), max_batch=B, max_k=max(K, 1),
                       max_pos=int(lens.max()) + (K + 1) * iters + 8, weight_format=weight_format)
    lp = M.SpecLoop(ctx, B, K, thr, out_cap=(K + 1) * iters)
    lp.seq_hash.copy_(as_i64(h0))
    lp.last_tok.copy_(dev(last0))
    lp.positions.copy_(dev(lens))
    hid0 = np.stack([L.target_hidden(int(h0[b]), cfg.H, cfg.dtype) for b in range(B)])
    lp.hidden.copy_(dev(stored_bits(hid0, cfg.dtype)))
    lp.embeds.copy_(dev(w["embed"][last0]))
    kvd = upload_kv(kv0) if K > 0 else None
    M.mtp_spec_loop(ctx, kvd, lp, iters)
    torch.cuda.synchronize()
    assert M.mtp_get_device_error(ctx) == 0
    n = host(lp.out_len)
    gpu = [list(host(lp.out_tokens)[b, :n[b]]) for b in range(B)]
    # oracle
    if weight_format == "int4_g64":
        from oracle import quant
        W = quant.quantized_weights(w, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
        dense_rows = lambda ids: O.widen(w["embed"][np.asarray(ids)], cfg.dtype)
    else:
        W = O.MTPWeights64.from_stored(w, cfg.dtype, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
        dense_rows = None
    st = L.LoopState([int(x) for x in h0], [int(x) for x in last0], [int(x) for x in lens], [[] for _ in range(B)])
    acc = None
    if K > 0:
        acc = L.spec_loop(W, kv0.copy(), st, K, thr, iters, cfg.dtype, embed_rows=dense_rows)
    greedy = [L.greedy(int(h0[b]), int(last0[b]), thr, cfg.vocab, len(gpu[b])) for b in range(B)]
    return lp, gpu, st, acc, greedy, lens


@pytest.mark.parametrize("K", [3, 0])
def test_spec_loop_tiny_f32(K):
    cfg = synth.MTPShape("loop_f32", H=256, n_q=4, n_kv=2, head_dim=64, ffn=512, vocab=4096, batch=2, K=3,
                         dtype="f32", ctx_lo=5, ctx_hi=40, seed_index=73)
    w = synth.copy_head(cfg, synth.make_weights(cfg, norm="ones"))
    iters = 10
    lp, gpu, st, acc, greedy, lens = _run_loop(cfg, w, K, iters, int(0.7 * 2 ** 53))
    for b in range(2):
        assert gpu[b] == greedy[b]
        if K:
            assert gpu[b] == st.out[b]
            assert int(host(lp.positions)[b]) == st.position[b]
            assert int(host(lp.seq_hash).view(np.uint64)[b]) == st.seq_hash[b]
        else:
            assert len(gpu[b]) == iters
    if K:
        np.testing.assert_array_equal(host(lp.accepted), acc[-1])
        assert acc.max() > 0 and (acc < K).any()


def test_spec_loop_bf16_ragged_batch():
    cfg = synth.MTPShape("loop_bf16", H=512, n_q=8, n_kv=2, head_dim=128, ffn=1536, vocab=5003, batch=3, K=4,
                         dtype="bf16", ctx_lo=0, ctx_hi=60, paged_shuffle=True, seed_index=74)
    w = synth.copy_head(cfg, synth.make_weights(cfg, norm="random"))
    lp, gpu, st, acc, greedy, lens = _run_loop(cfg, w, 4, 8, int(0.8 * 2 ** 53), lens=[0, 17, 60])
    for b in range(3):
        assert gpu[b] == st.out[b] == greedy[b]
    assert acc.max() > 0


def test_spec_loop_quantized_head():
    cfg = synth.MTPShape("loop_q4", H=1024, n_q=8, n_kv=2, head_dim=128, ffn=2048, vocab=5003, batch=2, K=3,
                         dtype="bf16", ctx_lo=3, ctx_hi=50, paged_shuffle=True, seed_index=75)
    w = synth.copy_head(cfg, synth.make_weights(cfg, norm="random"))
    lp, gpu, st, acc, greedy, lens = _run_loop(cfg, w, 3, 8, int(0.8 * 2 ** 53), weight_format="int4_g64")
    for b in range(2):
        assert gpu[b] == st.out[b] == greedy[b]
    assert acc.max() > 0


@pytest.mark.slow
def test_spec_loop_qwen3_8b_b1():
    """Qwen3-8B-shaped head with the copy recipe, B = 1, context 4096, K = 5:
    the loop bench's workload."""
    cfg = synth.QWEN3_8B_B1
    w = synth.copy_head(cfg, synth.make_weights(cfg, norm="ones"))
    lp, gpu, st, acc, greedy, lens = _run_loop(cfg, w, 5, 4, int(0.8 * 2 ** 53))
    assert gpu[0] == st.out[0] == greedy[0]
