"""Pins of the oracle's tree drafting ("Speculative Decoding" (OpenVINO
GenAI), "Tree Drafting", "How Tree Drafting Works"): the validation rules,
the candidate count, branching factor 1 reproducing chain drafting (tokens
and cache entries), tree invariants, tree verification against brute force
over all paths, and the tree loop against greedy decoding.  CPU only."""
import numpy as np
import pytest

import oracle as O
from oracle import loop as L
from oracle import tree as T
import synth


def test_validation_rules():
    assert T.tree_is_valid(2, 3, 10) and not T.tree_is_valid(2, 3, 11)      # 2*2*2 + 2 = 10 candidates
    assert not T.tree_is_valid(2, 3, 2)                                    # n_assist >= tree_depth
    assert T.tree_is_valid(1, 5, 5) and not T.tree_is_valid(1, 5, 6)       # a chain supplies td
    assert T.tree_is_valid(4, 1, 4) and not T.tree_is_valid(4, 1, 5)


def _case(K=4, V=512, seed=80, copy=False):
    cfg = synth.MTPShape("tree_t", H=128, n_q=4, n_kv=2, head_dim=32, ffn=256, vocab=V, batch=1, K=K,
                         dtype="f32", ctx_lo=21, ctx_hi=21, seed_index=seed)
    w = synth.make_weights(cfg, norm="random")
    if copy:
        w = synth.copy_head(cfg, w)
    W = O.MTPWeights64.from_stored(w, "f32", cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    lens = synth.context_lengths(cfg)
    kv = synth.make_kv(cfg, lens, extra_slots=2 * K + 4)
    di = synth.make_draft_inputs(cfg, w, lens)
    return cfg, W, kv, di


@pytest.mark.parametrize("bf,td", [(2, 3), (3, 2), (3, 3), (4, 1)])
def test_candidate_count_and_tree_invariants(bf, td):
    cfg, W, kv, di = _case()
    n = bf * bf * (td - 1) + bf
    tr = T.tree_draft_one(W, O.widen(di.hidden[0], "f32"), O.widen(di.embeds[0], "f32"), int(di.positions[0]),
                          kv, bf, td, max(td, n - 1))
    assert len(tr.cands) == n
    # packed parents first, depth one more than the parent's, scores not increasing along a path
    for i in range(len(tr.tokens)):
        p = int(tr.parents[i])
        assert p < i
        assert tr.depths[i] == (1 if p < 0 else tr.depths[p] + 1)
        if p >= 0:
            assert tr.scores[i] <= tr.scores[p] + 1e-12
    # children of one node carry distinct tokens
    for p in set(tr.parents.tolist()):
        kids = tr.tokens[tr.parents == p]
        assert len(set(kids.tolist())) == len(kids)
    # the packed nodes are the best n_assist candidates
    best = sorted(c.score for c in tr.cands)[::-1][:len(tr.tokens)]
    np.testing.assert_allclose(sorted(tr.scores)[::-1], best, rtol=1e-12)


def test_branching_factor_one_is_chain_drafting():
    K = 4
    cfg, W, kv, di = _case(K=K)
    h, e, pos = O.widen(di.hidden, "f32"), O.widen(di.embeds, "f32"), di.positions
    tr = T.tree_draft_one(W, h[0], e[0], int(pos[0]), kv, 1, K, K)
    kv_chain = kv.copy()
    res = O.draft(W, h, e, pos, kv_chain, K)
    np.testing.assert_array_equal(tr.tokens, res.ids[0])
    np.testing.assert_array_equal(tr.parents, [-1, 0, 1, 2])
    # the root's and the expanded nodes' cache entries are chain drafting's
    L0 = int(kv.seq_len[0])
    np.testing.assert_allclose(tr.root_k, T._entry(kv_chain, L0)[0], rtol=1e-12, atol=1e-12)
    for d in range(1, K):
        c = tr.cands[tr.selected[d - 1]]
        assert c.expanded
        np.testing.assert_allclose(c.entry_k, T._entry(kv_chain, L0 + d)[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(c.entry_v, T._entry(kv_chain, L0 + d)[1], rtol=1e-12, atol=1e-12)
    # committing an accepted path of a = 2 equals chain drafting's commit of min(a + 1, K)
    kv_t = kv.copy()
    T.commit_tree(kv_t, 0, tr, [0, 1])
    O.kv_commit(kv_chain, np.array([3], dtype=np.int32), "f32")
    np.testing.assert_array_equal(kv_t.seq_len, kv_chain.seq_len)
    np.testing.assert_allclose(kv_t.k_pool, kv_chain.k_pool, rtol=1e-12, atol=1e-12)


def test_tree_verify_matches_bruteforce():
    rng = np.random.default_rng(5)
    for _ in range(300):
        n = int(rng.integers(1, 12))
        parents = np.array([int(rng.integers(-1, i)) for i in range(n)], dtype=np.int32)
        tokens = np.empty(n, dtype=np.int32)
        for i in range(n):       # distinct tokens among siblings, from a small alphabet
            used = {int(tokens[j]) for j in range(i) if parents[j] == parents[i]}
            tokens[i] = int(rng.choice([t for t in range(6) if t not in used]))
        preds = rng.integers(0, 6, size=n + 1)
        a, path, bonus = T.verify_tree(preds, tokens, parents)
        assert (a, bonus) == T.verify_tree_bruteforce(preds, tokens, parents)
        assert len(path) == a


def test_tree_loop_equals_greedy():
    cfg, W, kv, di = _case(K=3, V=512, copy=True)
    kv = synth.make_kv(cfg, synth.context_lengths(cfg), extra_slots=40)
    h0 = [int(synth.loop_start_hashes(cfg, 1)[0])]
    last0 = [7]
    st = L.LoopState(list(h0), list(last0), [int(cfg.ctx_lo)], [[]])
    thr = int(0.7 * 2 ** 53)
    acc = T.tree_spec_loop(W, kv, st, 2, 3, 6, thr, 8, "f32")
    assert st.out[0] == L.greedy(h0[0], last0[0], thr, W.lm_rows, len(st.out[0]))
    assert acc.max() > 0
    assert st.position[0] == cfg.ctx_lo + len(st.out[0])
