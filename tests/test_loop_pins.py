"""Pins of the oracle's speculative loop and its synthetic verifier: the
SplitMix64 finaliser against published outputs, the verifier rows, and the
greedy-equivalence invariant ("How OpenVINO MTP Speculative Decoding Works
Internally": speculative output equals plain greedy output of the main
model; "Speculative Decoding" (OpenVINO GenAI), "Overview") for drafters that
are always, sometimes and never right.  CPU only."""
import numpy as np

import oracle as O
from oracle import loop as L
import synth

GOLDEN = 0x9E3779B97F4A7C15


def test_mix64_gives_published_splitmix64_outputs():
    # SplitMix64 from state 1234567: output n = mix(1234567 + (n + 1) * GOLDEN)
    states = np.array([(1234567 + (n + 1) * GOLDEN) % 2 ** 64 for n in range(5)], dtype=np.uint64)
    np.testing.assert_array_equal(
        L.mix64(states),
        np.array([6457827717110365317, 3203168211198807973, 9817491932198370423,
                  4593380528125082431, 16408922859458223821], dtype=np.uint64))


def test_target_row_has_a_unique_planted_argmax_and_bounded_noise():
    V = 5003
    for h in (1, 2 ** 63 + 5, 123456789):
        for dtype in ("bf16", "f32"):
            z = L.target_row(h, 17, 2 ** 52, V, dtype)
            p = L.predict(h, 17, 2 ** 52, V)
            assert z[p] == 8.0 and np.sum(z == 8.0) == 1
            rest = np.delete(z, p)
            assert rest.min() >= -0.5 and rest.max() <= 0.5     # bf16 may round up to 0.5
            assert int(O.argmax_lowest(z[None])[0]) == p
    # bf16 storage: every value is a bf16 value
    z = L.target_row(99, 3, 0, V, "bf16")
    np.testing.assert_array_equal(O.round_to_bf16(z), z)


def test_sticky_threshold_extremes():
    V = 1000
    hs = L.mix64(np.arange(1, 200, dtype=np.uint64))
    assert all(L.predict(int(h), 42, 2 ** 53, V) == 42 for h in hs)      # always the last token
    other = [L.predict(int(h), 42, 0, V) for h in hs]                    # never sticky
    assert sum(t == 42 for t in other) <= 2


def _loop_case(copy=True, B=2, K=3, V=4096, iters=12):
    cfg = synth.MTPShape("loop_t", H=256, n_q=4, n_kv=2, head_dim=64, ffn=512, vocab=V, batch=B, K=K,
                         dtype="f32", ctx_lo=5, ctx_hi=40, seed_index=70)
    w = synth.make_weights(cfg, norm="ones")
    if copy:
        w = synth.copy_head(cfg, w)
    W = O.MTPWeights64.from_stored(w, "f32", cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    lens = synth.context_lengths(cfg)
    kv = synth.make_kv(cfg, lens, extra_slots=K * iters + K)
    h0 = [int(x) for x in synth.loop_start_hashes(cfg, B)]
    last0 = [int(x) for x in synth.uniform_int(cfg.seed, 99, (B,), 0, V)]
    st = L.LoopState(list(h0), list(last0), [int(x) for x in lens], [[] for _ in range(B)])
    return cfg, W, kv, st, h0, last0, lens


def _check_equivalence(W, kv, st, h0, last0, K, thr, iters, dtype="f32"):
    acc = L.spec_loop(W, kv, st, K, thr, iters, dtype)
    V = W.lm_rows
    for b in range(len(h0)):
        g = L.greedy(h0[b], last0[b], thr, V, len(st.out[b]))
        assert st.out[b] == g
        assert len(st.out[b]) == int(np.sum(acc[:, b])) + iters
    return acc


def test_spec_loop_equals_greedy_with_sometimes_right_drafts():
    cfg, W, kv, st, h0, last0, lens = _loop_case(copy=True)
    K = cfg.K
    lens0 = np.array(lens)
    acc = _check_equivalence(W, kv, st, h0, last0, K, int(0.7 * 2 ** 53), 12)
    assert acc.max() > 0                       # some drafts were accepted
    assert (acc < K).any()                      # and some were rejected
    # bookkeeping: positions advanced by the emitted counts, hashes folded
    for b in range(len(h0)):
        assert st.position[b] == int(lens0[b]) + len(st.out[b])
        h = h0[b]
        for t in st.out[b]:
            h = L.fold(h, t)
        assert st.seq_hash[b] == h


def test_spec_loop_all_accepted_when_the_target_repeats():
    cfg, W, kv, st, h0, last0, lens = _loop_case(copy=True, B=1)
    acc = _check_equivalence(W, kv, st, h0, last0, cfg.K, 2 ** 53, 2)
    assert (acc == cfg.K).all()
    assert st.out[0] == [last0[0]] * len(st.out[0])


def test_spec_loop_equals_greedy_with_random_drafts():
    cfg, W, kv, st, h0, last0, lens = _loop_case(copy=False)
    _check_equivalence(W, kv, st, h0, last0, cfg.K, int(0.7 * 2 ** 53), 2)


def test_spec_loop_with_confidence_stop_equals_greedy():
    """The confidence stop changes how many drafts are proposed, never the
    output: with a threshold at the median draft confidence some steps
    propose fewer than K drafts and the tokens still equal greedy decoding."""
    from oracle import dynamic as D
    cfg, W, kv, st, h0, last0, lens = _loop_case(copy=False, B=2)
    kv_probe = kv.copy()
    res = O.draft(W, np.ones((2, cfg.H)), W.embed_rows(np.array(last0)), np.array(st.position, dtype=np.int32),
                  kv_probe, cfg.K)
    tau = float(np.median(D.draft_confidence(res.logits)))
    acc = L.spec_loop(W, kv, st, cfg.K, int(0.7 * 2 ** 53), 6, "f32", conf_tau=tau)
    for b in range(2):
        assert st.out[b] == L.greedy(h0[b], last0[b], int(0.7 * 2 ** 53), W.lm_rows, len(st.out[b]))
