"""Dynamic draft length on the GPU ("Speculative Decoding" (OpenVINO GenAI),
"Fast Draft", "Backend Differences"): the draft confidence against the
oracle's on the same logits, the confidence stop inside the speculative loop
(output still equal to greedy decoding), and a host-driven loop whose draft
count follows the acceptance-driven rule."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import dynamic as D
from oracle import loop as L
import synth
from gpu_util import dev, host, make_context, upload_kv, upload_weights
from test_gpu_loop import as_i64, stored_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("weight_format", ["dense", "int4_g64"])
def test_draft_confidence_matches_oracle_on_the_same_logits(weight_format):
    import mtp_self_speculative_gb300 as M
    cfg = synth.MTPShape("conf", H=1024, n_q=8, n_kv=2, head_dim=128, ffn=2048, vocab=5003, batch=3, K=4,
                         dtype="bf16", ctx_lo=5, ctx_hi=70, paged_shuffle=True, seed_index=76)
    w = synth.make_weights(cfg, norm="random")
    lens = synth.context_lengths(cfg)
    kv = upload_kv(synth.make_kv(cfg, lens, extra_slots=cfg.K + 1))
    di = synth.make_draft_inputs(cfg, w, lens)
    ctx = make_context(cfg, upload_weights(w), weight_format=weight_format)
    B, K, V = 3, cfg.K, cfg.vocab
    ids = torch.empty((B, K), dtype=torch.int32, device="cuda")
    logits = torch.empty((B, K, V), dtype=torch.float32, device="cuda")
    M.mtp_draft(ctx, dev(di.hidden), dev(di.embeds), dev(di.positions), kv, K, ids, logits)
    conf = torch.empty((B, K), dtype=torch.float32, device="cuda")
    z = host(logits).astype(np.float64)
    want = D.draft_confidence(z)
    for tau in np.quantile(want, [0.1, 0.5, 0.9]):
        nd = torch.empty(B, dtype=torch.int32, device="cuda")
        M.mtp_draft_confidence(ctx, logits, float(tau), conf, nd)
        torch.cuda.synchronize()
        got = host(conf).astype(np.float64)
        np.testing.assert_allclose(got, want, rtol=1e-5)
        exp = D.num_drafts_from_confidence(want, tau)
        near = np.abs(want - tau) <= 1e-5 * tau
        for b in range(B):
            if not near[b, :exp[b] + 1 if exp[b] < K else K].any():
                assert int(host(nd)[b]) == exp[b]
    assert M.mtp_get_device_error(ctx) == 0


def test_spec_loop_confidence_stop_equals_greedy():
    import mtp_self_speculative_gb300 as M
    cfg = synth.MTPShape("loop_conf", H=512, n_q=8, n_kv=2, head_dim=128, ffn=1536, vocab=5003, batch=2, K=4,
                         dtype="bf16", ctx_lo=3, ctx_hi=40, paged_shuffle=True, seed_index=77)
    w = synth.make_weights(cfg, norm="random")
    B, K, iters, thr = 2, cfg.K, 8, int(0.7 * 2 ** 53)
    lens = synth.context_lengths(cfg)
    kv = upload_kv(synth.make_kv(cfg, lens, extra_slots=K * iters + K + 1))
    h0 = synth.loop_start_hashes(cfg, B)
    last0 = synth.uniform_int(cfg.seed, 95, (B,), 0, cfg.vocab)
    ctx = make_context(cfg, upload_weights(w), max_batch=B, max_k=K, max_pos=int(lens.max()) + (K + 1) * iters + 8)
    # probe the confidences of a first draft to place the threshold at their median
    probe = M.SpecLoop(ctx, B, K, thr, out_cap=8, conf_threshold=1e-12)
    lp = M.SpecLoop(ctx, B, K, thr, out_cap=(K + 1) * iters, conf_threshold=1.0)
    for loop in (probe, lp):
        loop.seq_hash.copy_(as_i64(h0))
        loop.last_tok.copy_(dev(last0))
        loop.positions.copy_(dev(lens))
        loop.hidden.copy_(dev(stored_bits(np.stack([L.target_hidden(int(h0[b]), cfg.H, "bf16") for b in range(B)]),
                                          "bf16")))
        loop.embeds.copy_(dev(w["embed"][last0]))
    kv_probe = upload_kv(synth.make_kv(cfg, lens, extra_slots=K * iters + K + 1))
    M.mtp_spec_loop(ctx, kv_probe, probe, 1)
    torch.cuda.synchronize()
    lp.conf_threshold = float(np.median(host(probe.conf)))
    proposed = []
    for _ in range(iters):
        M.mtp_spec_loop(ctx, kv, lp, 1)
        torch.cuda.synchronize()
        proposed.extend(host(lp.num_drafts).tolist())
    assert M.mtp_get_device_error(ctx) == 0
    assert min(proposed) < K and max(proposed) > 0
    n = host(lp.out_len)
    for b in range(B):
        toks = host(lp.out_tokens)[b, :n[b]].tolist()
        assert toks == L.greedy(int(h0[b]), int(last0[b]), thr, cfg.vocab, len(toks))


def test_adaptive_draft_count_host_loop():
    """A host-driven loop (one synchronisation per step, as a serving loop
    reads its tokens) whose draft count follows mtp_adapt_k; the copy head and
    a sticky verifier make full acceptances and rejections both happen."""
    import mtp_self_speculative_gb300 as M
    cfg = synth.MTPShape("loop_adapt", H=512, n_q=8, n_kv=2, head_dim=128, ffn=1536, vocab=5003, batch=1, K=8,
                         dtype="bf16", ctx_lo=20, ctx_hi=20, seed_index=78)
    w = synth.copy_head(cfg, synth.make_weights(cfg, norm="ones"))
    K_max, iters, thr = 8, 12, int(0.75 * 2 ** 53)
    lens = synth.context_lengths(cfg)
    kv = upload_kv(synth.make_kv(cfg, lens, extra_slots=K_max * iters + K_max + 1))
    h0 = synth.loop_start_hashes(cfg, 1)
    last0 = synth.uniform_int(cfg.seed, 95, (1,), 0, cfg.vocab)
    ctx = make_context(cfg, upload_weights(w), max_batch=1, max_k=K_max,
                       max_pos=int(lens.max()) + (K_max + 1) * iters + 8)
    lp = M.SpecLoop(ctx, 1, K_max, thr, out_cap=(K_max + 1) * iters)
    lp.seq_hash.copy_(as_i64(h0))
    lp.last_tok.copy_(dev(last0))
    lp.positions.copy_(dev(lens))
    lp.hidden.copy_(dev(stored_bits(L.target_hidden(int(h0[0]), cfg.H, "bf16")[None], "bf16")))
    lp.embeds.copy_(dev(w["embed"][last0]))
    K, Ks, accs = 3, [], []
    flat = lp.drafts.view(-1)
    for _ in range(iters):
        drafts = flat[:K].view(1, K)
        M.mtp_draft(ctx, lp.hidden, lp.embeds, lp.positions, kv, K, drafts)
        nd = torch.full((1,), K, dtype=torch.int32, device="cuda")
        M.mtp_synth_target(ctx, lp.seq_hash, lp.last_tok, drafts, K, thr, lp.target_logits[:K + 1],
                           lp.row_offsets, num_drafts=nd)
        M.mtp_verify(ctx, lp.target_logits[:K + 1], lp.row_offsets, drafts, nd, lp.accepted, lp.bonus)
        M.mtp_kv_commit_accepted(ctx, kv, lp.accepted, extra=1)
        M.mtp_loop_advance(ctx, K, drafts, lp.accepted, lp.bonus, lp.seq_hash, lp.last_tok, lp.positions,
                           lp.hidden, lp.embeds, lp.out_tokens, lp.out_len)
        a = int(host(lp.accepted)[0])          # the serving loop's one read per step
        Ks.append(K)
        accs.append(a)
        K_next = M.mtp_adapt_k(K, a, K, 1, K_max)
        assert K_next == D.next_k(K, a, K, 1, K_max)
        K = K_next
    assert M.mtp_get_device_error(ctx) == 0
    assert len(set(Ks)) > 1                     # the count did move
    n = int(host(lp.out_len)[0])
    toks = host(lp.out_tokens)[0, :n].tolist()
    assert toks == L.greedy(int(h0[0]), int(last0[0]), thr, cfg.vocab, n)
    assert n == sum(accs) + iters
