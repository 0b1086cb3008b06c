"""Tree drafting on the GPU ("Speculative Decoding" (OpenVINO GenAI), "Tree
Drafting", "How Tree Drafting Works") against the oracle: the packed trees
(tokens, parents, depths) on an fp32 head, including a request whose tree
crosses a cache block; the request's own cache touched only at the root's
slot while drafting; verification and commit; branching factor 1 equal to
chain drafting on the GPU; and the tree loop equal to greedy decoding."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import loop as L
from oracle import tree as T
import synth
from gpu_util import Guarded, dev, download_kv, host, kv_slots, make_context, upload_kv, upload_weights
from test_gpu_loop import as_i64, stored_bits

pytestmark = pytest.mark.gpu


def with_scratch(kv: synth.KVState, n: int):
    """The cache with n zero blocks appended to the pools; returns it and
    their ids."""
    z = np.zeros((n,) + kv.k_pool.shape[1:], dtype=kv.k_pool.dtype)
    out = synth.KVState(np.concatenate([kv.k_pool, z]), np.concatenate([kv.v_pool, z]), kv.block_table.copy(),
                        kv.seq_len.copy(), kv.pending.copy(), kv.block_size)
    return out, np.arange(kv.k_pool.shape[0], kv.k_pool.shape[0] + n, dtype=np.int32)


F32 = dict(H=256, n_q=4, n_kv=2, head_dim=64, ffn=512, vocab=4096, K=3, dtype="f32", paged_shuffle=True)


def _tree_case(bf=3, td=3, n_assist=8, lens=(31, 40, 16), seed=81, weights=None):
    import mtp_self_speculative_gb300 as M
    B = len(lens)
    cfg = synth.MTPShape("tree_g", batch=B, ctx_lo=min(lens), ctx_hi=max(lens), seed_index=seed, **F32)
    w = synth.make_weights(cfg, norm="random") if weights is None else weights(cfg)
    lens = np.asarray(lens, dtype=np.int32)
    kv0, scratch = with_scratch(synth.make_kv(cfg, lens, extra_slots=td + 20), (td - 1) * B * bf * 2)
    di = synth.make_draft_inputs(cfg, w, lens)
    ctx = make_context(cfg, upload_weights(w), max_batch=max(B * bf, B), max_k=max(td, 2),
                       max_pos=int(lens.max()) + 64)
    tree = M.TreeDraft(ctx, B, bf, td, n_assist, kv0.block_table.shape[1], dev(scratch))
    W = O.MTPWeights64.from_stored(w, cfg.dtype, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    return cfg, w, W, kv0, di, ctx, tree, lens


def test_tree_draft_matches_oracle_f32():
    import mtp_self_speculative_gb300 as M
    bf, td, n_assist = 3, 3, 8
    cfg, w, W, kv0, di, ctx, tree, lens = _tree_case(bf, td, n_assist)
    kvd = upload_kv(kv0)
    M.mtp_draft_tree(ctx, dev(di.hidden), dev(di.embeds), dev(di.positions), kvd, tree)
    torch.cuda.synchronize()
    assert M.mtp_get_device_error(ctx) == 0
    got = download_kv(kvd)
    checked = 0
    for b in range(len(lens)):
        kv1 = T._one_request_kv(kv0, b)
        tr = T.tree_draft_one(W, O.widen(di.hidden[b], "f32"), O.widen(di.embeds[b], "f32"), int(di.positions[b]),
                              kv1, bf, td, n_assist)
        L0 = int(lens[b])
        if tr.min_margin > 1e-4:
            np.testing.assert_array_equal(host(tree.tokens)[b], tr.tokens)
            np.testing.assert_array_equal(host(tree.parents)[b], tr.parents)
            np.testing.assert_array_equal(host(tree.depths)[b], tr.depths)
            checked += 1
        # the request's own cache: only the root's slot was written
        gk, gv = kv_slots(got, b, 0, L0 + td + 1)
        ok, ov = kv_slots(kv0, b, 0, L0 + td + 1)
        np.testing.assert_array_equal(np.delete(gk, L0, axis=0), np.delete(ok, L0, axis=0))
        np.testing.assert_array_equal(np.delete(gv, L0, axis=0), np.delete(ov, L0, axis=0))
        err = np.max(np.abs(gk[L0] - tr.root_k)) / np.max(np.abs(tr.root_k))
        assert err <= 1e-3
    np.testing.assert_array_equal(got.pending, 1)
    np.testing.assert_array_equal(got.seq_len, lens)
    assert checked >= 2
    # layer 1 is the MTP step from the verifier state: its nodes are the top
    # candidates of that step's logits, exactly (the same LM-head kernel
    # writes the logits of a one-step mtp_draft on the same inputs)
    ids = Guarded((len(lens), 1), torch.int32)
    z = Guarded((len(lens), 1, cfg.vocab), torch.float32)
    M.mtp_draft(ctx, dev(di.hidden), dev(di.embeds), dev(di.positions), upload_kv(kv0), 1, ids.t, z.t)
    torch.cuda.synchronize()
    ids.check("draft_ids")
    z.check("logits")
    zh = host(z.t)[:, 0]
    dep = host(tree.depths)
    for b in range(len(lens)):
        first = sorted(int(t) for t in host(tree.tokens)[b][dep[b] == 1])
        order = np.lexsort((np.arange(cfg.vocab), -zh[b].astype(np.float64)))   # value desc, id asc
        assert 1 <= len(first) <= bf
        assert first == sorted(order[:len(first)].tolist())
        assert int(host(ids.t)[b, 0]) == int(order[0])


def test_tree_verify_and_commit_match_oracle_f32():
    import mtp_self_speculative_gb300 as M
    bf, td, n_assist = 3, 3, 8
    cfg, w, W, kv0, di, ctx, tree, lens = _tree_case(bf, td, n_assist, seed=82, lens=(47, 18))
    B = len(lens)
    kvd = upload_kv(kv0)
    M.mtp_draft_tree(ctx, dev(di.hidden), dev(di.embeds), dev(di.positions), kvd, tree)
    h0 = synth.loop_start_hashes(cfg, B)
    # a verifier that follows each tree's first path: plant a sticky prediction
    last = di.token_ids.astype(np.int32)
    thr = int(0.9 * 2 ** 53)
    logits = torch.empty((B * (1 + n_assist), cfg.vocab), dtype=torch.float32, device="cuda")
    offs = torch.empty(B + 1, dtype=torch.int32, device="cuda")
    M.mtp_synth_target_tree(ctx, tree, as_i64(h0), dev(last), thr, logits, offs)
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    bonus = torch.empty(B, dtype=torch.int32, device="cuda")
    path = torch.full((B, td), -1, dtype=torch.int32, device="cuda")
    M.mtp_verify_tree(ctx, tree, logits, acc, bonus, path)
    M.mtp_tree_commit(ctx, kvd, tree, acc)
    torch.cuda.synchronize()
    assert M.mtp_get_device_error(ctx) == 0
    np.testing.assert_array_equal(host(offs), np.arange(B + 1) * (1 + n_assist))
    got = download_kv(kvd)
    tok, par = host(tree.tokens), host(tree.parents)
    checked = 0
    for b in range(B):
        # oracle predictions along the GPU's tree, and the oracle's walk
        preds = [L.predict(int(h0[b]), int(last[b]), thr, cfg.vocab)]
        for i in range(n_assist):
            h = int(h0[b])
            for t in T.node_prefix_tokens(i, tok[b], par[b]):
                h = L.fold(h, t)
            preds.append(L.predict(h, int(tok[b, i]), thr, cfg.vocab))
        z = host(logits)[b * (1 + n_assist):(b + 1) * (1 + n_assist)]
        np.testing.assert_array_equal(O.argmax_lowest(z), preds)
        a, nodes, bo = T.verify_tree(np.array(preds), tok[b], par[b])
        assert int(host(acc)[b]) == a and int(host(bonus)[b]) == bo
        np.testing.assert_array_equal(host(path)[b, :a], tok[b][nodes])
        # the oracle tree on the same inputs, and its commit
        kv1 = T._one_request_kv(kv0, b)
        tr = T.tree_draft_one(W, O.widen(di.hidden[b], "f32"), O.widen(di.embeds[b], "f32"), int(di.positions[b]),
                              kv1, bf, td, n_assist)
        if tr.min_margin <= 1e-4:
            continue                 # the oracle's own tree has a near-tie: the GPU may pick either side
        np.testing.assert_array_equal(tok[b], tr.tokens)
        checked += 1
        kvc = kv0.copy()
        kept = T.commit_tree(kvc, b, tr, nodes)
        L0 = int(lens[b])
        assert int(got.seq_len[b]) == L0 + kept and int(got.pending[b]) == 0
        gk, gv = kv_slots(got, b, L0, L0 + kept)
        ok, ov = kv_slots(kvc, b, L0, L0 + kept)
        for g_, o_ in ((gk, ok), (gv, ov)):
            e = np.max(np.abs(g_ - o_), axis=(1, 2)) / np.maximum(np.max(np.abs(o_), axis=(1, 2)), 1e-30)
            assert np.max(e) <= 1e-3
        zk, zv = kv_slots(got, b, L0 + kept, L0 + td + 1)
        assert not zk.any() and not zv.any()
    assert checked >= 1          # both requests of this seed have oracle margins above 1e-4


def test_branching_one_equals_chain_drafting_bf16():
    import mtp_self_speculative_gb300 as M
    cfg = synth.MTPShape("tree_chain", H=512, n_q=8, n_kv=2, head_dim=128, ffn=1536, vocab=5003, batch=2, K=4,
                         dtype="bf16", ctx_lo=5, ctx_hi=60, paged_shuffle=True, seed_index=83)
    w = synth.make_weights(cfg, norm="random")
    lens = np.array([15, 60], dtype=np.int32)
    kv0, scratch = with_scratch(synth.make_kv(cfg, lens, extra_slots=cfg.K + 8), (cfg.K - 1) * 2 * 2)
    di = synth.make_draft_inputs(cfg, w, lens)
    ctx = make_context(cfg, upload_weights(w), max_batch=2, max_k=cfg.K, max_pos=128, persistent_max_batch=-1)
    tree = M.TreeDraft(ctx, 2, 1, cfg.K, cfg.K, kv0.block_table.shape[1], dev(scratch))
    M.mtp_draft_tree(ctx, dev(di.hidden), dev(di.embeds), dev(di.positions), upload_kv(kv0), tree)
    ids = torch.empty((2, cfg.K), dtype=torch.int32, device="cuda")
    M.mtp_draft(ctx, dev(di.hidden), dev(di.embeds), dev(di.positions), upload_kv(kv0), cfg.K, ids)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(tree.tokens), host(ids))
    np.testing.assert_array_equal(host(tree.parents), [[-1, 0, 1, 2]] * 2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tree_loop_equals_greedy(dtype):
    import mtp_self_speculative_gb300 as M
    bf, td, n_assist, iters = 2, 4, 8, 8
    shape = dict(F32) if dtype == "f32" else dict(H=512, n_q=8, n_kv=2, head_dim=128, ffn=1536, vocab=5003, K=4,
                                                   dtype="bf16", paged_shuffle=True)
    lens = np.array([20, 33], dtype=np.int32)
    B = 2
    cfg = synth.MTPShape("tree_loop", batch=B, ctx_lo=20, ctx_hi=33, seed_index=84, **shape)
    w = synth.copy_head(cfg, synth.make_weights(cfg, norm="ones"))
    kv0, scratch = with_scratch(synth.make_kv(cfg, lens, extra_slots=(td + 1) * iters + td + 2),
                                (td - 1) * B * bf * 2)
    ctx = make_context(cfg, upload_weights(w), max_batch=B * bf, max_k=td,
                       max_pos=int(lens.max()) + (td + 1) * iters + 8)
    tree = M.TreeDraft(ctx, B, bf, td, n_assist, kv0.block_table.shape[1], dev(scratch))
    thr = int(0.8 * 2 ** 53)
    lp = M.SpecLoop(ctx, B, td, thr, out_cap=(td + 1) * iters)
    lp.target_logits = torch.zeros((B * (1 + n_assist), cfg.vocab), dtype=lp.target_logits.dtype, device="cuda")
    h0 = synth.loop_start_hashes(cfg, B)
    last0 = synth.uniform_int(cfg.seed, 95, (B,), 0, cfg.vocab)
    lp.seq_hash.copy_(as_i64(h0))
    lp.last_tok.copy_(dev(last0))
    lp.positions.copy_(dev(lens))
    lp.hidden.copy_(dev(stored_bits(np.stack([L.target_hidden(int(h0[b]), cfg.H, dtype) for b in range(B)]), dtype)))
    lp.embeds.copy_(dev(w["embed"][last0]))
    kvd = upload_kv(kv0)
    M.mtp_tree_loop(ctx, kvd, lp, tree, iters)
    torch.cuda.synchronize()
    assert M.mtp_get_device_error(ctx) == 0
    n = host(lp.out_len)
    accs = 0
    for b in range(B):
        toks = host(lp.out_tokens)[b, :n[b]].tolist()
        assert toks == L.greedy(int(h0[b]), int(last0[b]), thr, cfg.vocab, len(toks))
        assert int(host(lp.positions)[b]) == int(lens[b]) + len(toks)
        accs += len(toks) - iters
    assert accs > 0
    got = download_kv(kvd)
    assert (got.pending == 0).all() and (got.seq_len > lens).all()
