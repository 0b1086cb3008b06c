"""Pins of the float64 oracle against closed forms, invariants, brute force
and the worked examples of the pages -- never against a retyped copy of its
own formulas.  CPU only."""
import itertools
import math
import os

import numpy as np
import pytest

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------ number formats

def test_round_to_bf16_ties_and_exact_values():
    one = 1.0
    ulp = 2.0 ** -7                       # bf16 spacing in [1, 2)
    assert O.round_to_bf16(np.array([one]))[0] == one
    assert O.round_to_bf16(np.array([one + ulp / 2]))[0] == one            # tie -> even
    assert O.round_to_bf16(np.array([one + 3 * ulp / 2]))[0] == one + 2 * ulp  # tie -> even
    assert O.round_to_bf16(np.array([one + ulp / 2 + 1e-9]))[0] == one + ulp
    assert O.round_to_bf16(np.array([-3.0]))[0] == -3.0


def test_round_to_bf16_matches_library_rounding_on_float32_inputs():
    torch = pytest.importorskip("torch")
    x = synth.normal(7, 1, (20000,), dtype="f32").astype(np.float64) * 3.0
    x = x.astype(np.float32).astype(np.float64)   # float32-exact inputs
    lib = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_to_bf16(x), lib)
    bits = O.bf16_bits_of(O.round_to_bf16(x))
    np.testing.assert_array_equal(bits, synth.f32_to_bf16_bits(x.astype(np.float32)))


def test_widen_bf16_bits():
    bits = np.array([0x3F80, 0xBF80, 0x4000, 0x0000, 0x3F00], dtype=np.uint16)
    np.testing.assert_array_equal(O.widen(bits, "bf16"), [1.0, -1.0, 2.0, 0.0, 0.5])


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_vector_closed_form():
    c, eps, n = 3.0, 1e-6, 64
    w = np.linspace(0.5, 1.5, n)
    y = O.rmsnorm(np.full(n, c), w, eps)
    np.testing.assert_allclose(y, w * c / math.sqrt(c * c + eps), rtol=1e-15)


def test_rmsnorm_unit_rms_and_scale_invariance():
    x = np.array([3.0, -4.0, 0.0, 0.0])       # mean square = 25/4
    y = O.rmsnorm(x, np.ones(4), 0.0)
    np.testing.assert_allclose(y, [1.2, -1.6, 0.0, 0.0], rtol=1e-15)
    np.testing.assert_allclose(O.rmsnorm(1000 * x, np.ones(4), 0.0), y, rtol=1e-14)


# ------------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    x = np.arange(16, dtype=np.float64).reshape(2, 8)
    np.testing.assert_array_equal(O.rope(x, 0, 1e6), x)


def test_rope_first_pair_turns_by_position_radians():
    # pair 0 has inv_freq theta^0 = 1: at position p it turns by p radians,
    # in the positive sense (x0 + i x_{d/2}) * exp(i p)
    x = np.array([[1.0, 0.0]])
    np.testing.assert_allclose(O.rope(x, 1, 1e6), [[math.cos(1.0), math.sin(1.0)]], rtol=1e-15)
    x = np.array([[0.0, 1.0]])
    np.testing.assert_allclose(O.rope(x, 2, 1e6), [[-math.sin(2.0), math.cos(2.0)]], rtol=1e-15)


def test_rope_frequency_of_second_pair():
    # d = 4, theta = 100: pair 1 has inv_freq 100^(-2/4) = 0.1 -> 1 rad at p=10
    x = np.array([[0.0, 1.0, 0.0, 0.0]])   # pair 1 = (x[1], x[3])
    y = O.rope(x, 10, 100.0)
    np.testing.assert_allclose(y, [[0.0, math.cos(1.0), 0.0, math.sin(1.0)]], atol=1e-15)


def test_rope_preserves_pair_norms_and_is_relative():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, 128))
    k = rng.standard_normal((1, 128))
    for p in (1, 77, 4096):
        y = O.rope(q, p, 1e6)
        n0 = q[0, :64] ** 2 + q[0, 64:] ** 2
        n1 = y[0, :64] ** 2 + y[0, 64:] ** 2
        np.testing.assert_allclose(n1, n0, rtol=1e-12)
    dot = lambda m, n: float(O.rope(q, m, 1e6)[0] @ O.rope(k, n, 1e6)[0])
    assert dot(100, 40) == pytest.approx(dot(1060, 1000), rel=1e-9)
    assert dot(5, 5) == pytest.approx(float(q[0] @ k[0]), rel=1e-12)


# -------------------------------------------------------------- attention

def test_attention_single_key_returns_its_value():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((4, 8))
    k = rng.standard_normal((1, 2, 8))
    v = rng.standard_normal((1, 2, 8))
    o = O.attention(q, k, v)
    # group = 2: heads 0,1 read kv head 0; heads 2,3 read kv head 1
    np.testing.assert_allclose(o, v[0, [0, 0, 1, 1]], rtol=1e-15)


def test_attention_identical_keys_average_values():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((2, 8))
    k = np.repeat(rng.standard_normal((1, 1, 8)), 5, axis=0)
    v = rng.standard_normal((5, 1, 8))
    np.testing.assert_allclose(O.attention(q, k, v), np.repeat(v.mean(0), 2, axis=0), rtol=1e-13)


def test_attention_two_keys_logistic_weight():
    d = 4
    q = np.array([[1.0, 0.0, 0.0, 0.0]])
    k = np.array([[[2.0, 0, 0, 0]], [[0.0, 0, 0, 0]]])      # scores 2/sqrt(4)=1 and 0
    v = np.array([[[1.0, 0, 0, 0]], [[0.0, 1.0, 0, 0]]])
    w1 = 1.0 / (1.0 + math.exp(-1.0))
    np.testing.assert_allclose(O.attention(q, k, v), [[w1, 1 - w1, 0, 0]], rtol=1e-14)
    assert d == 4


def test_attention_dominant_key_selects_its_value():
    q = np.array([[50.0, 0, 0, 0]])
    k = np.zeros((3, 1, 4))
    k[1, 0, 0] = 10.0                                          # score 250 vs 0
    v = np.arange(12, dtype=np.float64).reshape(3, 1, 4)
    np.testing.assert_allclose(O.attention(q, k, v), v[1], rtol=1e-12)


def test_attention_gqa_group_mapping():
    n_q, n_kv, d = 8, 2, 4
    q = np.ones((n_q, d))
    k = np.zeros((1, n_kv, d))
    v = np.stack([np.full(d, 10.0), np.full(d, 20.0)])[None]
    o = O.attention(q, k, v)
    np.testing.assert_array_equal(o[:4], 10.0)
    np.testing.assert_array_equal(o[4:], 20.0)


def test_attention_order_of_slots_is_irrelevant():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((4, 16))
    k = rng.standard_normal((9, 2, 16))
    v = rng.standard_normal((9, 2, 16))
    perm = rng.permutation(9)
    np.testing.assert_allclose(O.attention(q, k, v), O.attention(q, k[perm], v[perm]), rtol=1e-12)


# -------------------------------------------------------------- MLP / proj

def test_silu_known_value():
    # sigmoid(1) = e/(1+e) = 0.7310585786300049
    np.testing.assert_allclose(O.silu(np.array([1.0, 0.0])), [0.7310585786300049, 0.0], rtol=1e-15)


def test_swiglu_scalar_network_by_hand():
    n = np.array([[2.0]])
    out = O.swiglu_mlp(n, np.array([[0.5]]), np.array([[3.0]]), np.array([[-2.0]]))
    # silu(1) * 6 * -2
    np.testing.assert_allclose(out, [[0.7310585786300049 * 6.0 * -2.0]], rtol=1e-14)


def test_swiglu_zero_gate_is_passthrough():
    rng = np.random.default_rng(4)
    n = rng.standard_normal((3, 16))
    out = O.swiglu_mlp(n, np.zeros((32, 16)), rng.standard_normal((32, 16)), rng.standard_normal((16, 32)))
    np.testing.assert_array_equal(out, 0.0)


def _tiny_weights(H=32, n_q=4, n_kv=2, d=8, F=64, V=64, seed=9, norm="random"):
    cfg = synth.MTPShape("t", H=H, n_q=n_q, n_kv=n_kv, head_dim=d, ffn=F, vocab=V, batch=1, K=3,
                         dtype="f32", ctx_lo=5, ctx_hi=5, seed_index=seed)
    w = synth.make_weights(cfg, norm=norm)
    return cfg, w


def test_eh_proj_concat_order_hidden_first():
    cfg, w = _tiny_weights()
    H = cfg.H
    W = O.MTPWeights64.from_stored(w, "f32", cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    rng = np.random.default_rng(5)
    h = rng.standard_normal((2, H))
    e = rng.standard_normal((2, H))
    W.w_eh = np.concatenate([np.eye(H), np.zeros((H, H))], axis=1)
    np.testing.assert_allclose(O.eh_proj(h, e, W), O.rmsnorm(h, W.w_norm_h, W.eps), rtol=1e-14)
    W.w_eh = np.concatenate([np.zeros((H, H)), np.eye(H)], axis=1)
    np.testing.assert_allclose(O.eh_proj(h, e, W), O.rmsnorm(e, W.w_norm_e, W.eps), rtol=1e-14)


# ---------------------------------------------------------- LM head, argmax

def test_argmax_ties_to_lowest_id():
    z = np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0]])
    np.testing.assert_array_equal(O.argmax_lowest(z), [1, 0])


def test_argmax_brute_force_small_vocab():
    for vals in itertools.product([0.0, 1.0, 2.0], repeat=4):
        z = np.array(vals)
        best = max(vals)
        assert O.argmax_lowest(z[None])[0] == min(i for i, x in enumerate(vals) if x == best)


def test_top2_gap():
    assert O.top2_gap(np.array([[1.0, 4.0, 3.5, -1.0]]))[0] == 0.5
    assert O.top2_gap(np.array([[2.0, 2.0]]))[0] == 0.0


def test_lm_head_self_dot_recovers_table_row():
    cfg, w = _tiny_weights(H=256, V=4096, norm="ones")
    W = O.MTPWeights64.from_stored(w, "f32", cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    ids = np.array([0, 17, 4095])
    z = O.lm_head(W.embed_rows(ids) * 7.0, W)
    np.testing.assert_array_equal(O.argmax_lowest(z), ids)


# ---------------------------------------------------------------- verify

def _load_golden():
    cases = []
    with open(os.path.join(GOLDEN, "accept_rule_examples.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            d, t, a, bonus = [p.strip() for p in line.split("|")]
            cases.append(([int(x) for x in d.split()], [int(x) for x in t.split()], int(a), int(bonus)))
    return cases


def _logits_with_argmax(tokens, V):
    rows = np.zeros((len(tokens), V), dtype=np.float32)
    rows[np.arange(len(tokens)), tokens] = 1.0
    return rows


def test_verify_golden_examples():
    cases = _load_golden()
    assert len(cases) >= 8
    for drafts, target, a, bonus in cases:
        K = len(drafts)
        V = 16
        logits = _logits_with_argmax(target, V)
        dr = np.array([drafts + [-1] * (4 - K)], dtype=np.int32)
        acc, bon = O.verify(logits, np.array([0, K + 1]), dr, np.array([K]), "f32")
        assert (acc[0], bon[0]) == (a, bonus), (drafts, target)
        n_seq, emitted = O.verify_sequential(np.array(target), np.array(drafts, dtype=np.int64))
        assert n_seq == a and emitted[-1] == bonus and emitted[:a] == drafts[:a]


def test_verify_brute_force_against_sequential_statement():
    V = 3
    for K in range(0, 4):
        for drafts in itertools.product(range(V), repeat=K):
            for target in itertools.product(range(V), repeat=K + 1):
                logits = _logits_with_argmax(list(target), V)
                dr = np.array([list(drafts) + [-1] * (3 - K)], dtype=np.int32)
                acc, bon = O.verify(logits, np.array([0, K + 1]), dr, np.array([K]), "f32")
                n_seq, emitted = O.verify_sequential(np.array(target), np.array(drafts))
                assert acc[0] == n_seq
                assert bon[0] == emitted[-1]
                assert len(emitted) == acc[0] + 1


def test_verify_accept_invariants_and_ragged_rows():
    cfg = synth.shrink(synth.VERIFY_B64, vocab=512, batch=12)
    vi = synth.make_verify_inputs(cfg)
    acc, bon = O.verify(vi.logits, vi.row_offsets, vi.drafts, vi.num_drafts, "bf16")
    # drafts equal to the row argmax everywhere -> K accepted + bonus of row K
    R = vi.logits.shape[0]
    r = O.argmax_lowest(O.widen(vi.logits, "bf16"))
    full = np.full_like(vi.drafts, -1)
    for b in range(cfg.batch):
        K_b = int(vi.num_drafts[b])
        full[b, :K_b] = r[vi.row_offsets[b]:vi.row_offsets[b] + K_b]
    acc2, bon2 = O.verify(vi.logits, vi.row_offsets, full, vi.num_drafts, "bf16")
    np.testing.assert_array_equal(acc2, vi.num_drafts)
    np.testing.assert_array_equal(bon2, r[vi.row_offsets[1:] - 1])
    # first-position mismatch -> 0 accepted, bonus = argmax of row 0
    miss = full.copy()
    for b in range(cfg.batch):
        miss[b, 0] = (r[vi.row_offsets[b]] + 1) % cfg.vocab
    acc3, bon3 = O.verify(vi.logits, vi.row_offsets, miss, vi.num_drafts, "bf16")
    np.testing.assert_array_equal(acc3, 0)
    np.testing.assert_array_equal(bon3, r[vi.row_offsets[:-1]])
    # rows after the first mismatch do not matter
    mutated = vi.logits.copy()
    for b in range(cfg.batch):
        for j in range(int(acc[b]) + 1, int(vi.num_drafts[b]) + 1):
            mutated[vi.row_offsets[b] + j] = mutated[vi.row_offsets[b] + j][::-1]
    acc4, bon4 = O.verify(mutated, vi.row_offsets, vi.drafts, vi.num_drafts, "bf16")
    np.testing.assert_array_equal(acc4, acc)
    np.testing.assert_array_equal(bon4, bon)
    assert R == int(vi.row_offsets[-1])


def test_synthetic_accept_length_matches_geometric_mean():
    # E[min(G, K)] = sum_{n=1..K} alpha^n for the planted-prefix recipe
    cfg = synth.shrink(synth.VERIFY_B64, vocab=64, batch=4000, k_lo=5, k_hi=5, K=5)
    vi = synth.make_verify_inputs(cfg, spike=50.0)
    acc, _ = O.verify(vi.logits, vi.row_offsets, vi.drafts, vi.num_drafts, "bf16")
    np.testing.assert_array_equal(acc, vi.accept_len)
    expect = synth.expected_accept_len(5, 0.8)
    assert expect == pytest.approx(2.68928)
    sd = np.std(acc) / math.sqrt(len(acc))
    assert abs(acc.mean() - expect) < 4 * sd


# -------------------------------------------------------------- KV cache

def _tiny_state(lens=(5, 21, 16), K=3, dtype="bf16", seed=11):
    cfg = synth.MTPShape("t", H=32, n_q=4, n_kv=2, head_dim=8, ffn=64, vocab=64, batch=len(lens), K=K,
                         dtype=dtype, ctx_lo=1, ctx_hi=1, paged_shuffle=True, seed_index=seed)
    w = synth.make_weights(cfg, norm="random")
    kv = synth.make_kv(cfg, np.array(lens), extra_slots=K + 2)
    return cfg, w, kv


def _run_draft(cfg, w, kv, K, chain=None):
    W = O.MTPWeights64.from_stored(w, cfg.dtype, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    di = synth.make_draft_inputs(cfg, w, kv.seq_len)
    return O.draft(W, O.widen(di.hidden, cfg.dtype), O.widen(di.embeds, cfg.dtype), di.positions, kv, K, chain)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_draft_then_rollback_is_bitwise_noop(dtype):
    cfg, w, kv = _tiny_state(dtype=dtype)
    before = kv.copy()
    _run_draft(cfg, w, kv, 3)
    np.testing.assert_array_equal(kv.pending, 3)
    assert not np.array_equal(kv.k_pool, before.k_pool)
    O.kv_rollback(kv, dtype)
    np.testing.assert_array_equal(kv.k_pool.view(np.uint8), before.k_pool.view(np.uint8))
    np.testing.assert_array_equal(kv.v_pool.view(np.uint8), before.v_pool.view(np.uint8))
    np.testing.assert_array_equal(kv.seq_len, before.seq_len)
    np.testing.assert_array_equal(kv.pending, 0)


def test_commit_keeps_prefix_and_zeroes_rest():
    cfg, w, kv = _tiny_state()
    L0 = kv.seq_len.copy()
    _run_draft(cfg, w, kv, 3)
    drafted = kv.copy()
    n_keep = np.array([0, 2, 3], dtype=np.int32)
    O.kv_commit(kv, n_keep, "bf16")
    np.testing.assert_array_equal(kv.seq_len, L0 + n_keep)
    np.testing.assert_array_equal(kv.pending, 0)
    for b in range(3):
        k_now, _ = O.kv_read_slots(kv, b, int(L0[b]) + 3, "bf16")
        k_dr, _ = O.kv_read_slots(drafted, b, int(L0[b]) + 3, "bf16")
        keep = int(L0[b] + n_keep[b])
        np.testing.assert_array_equal(k_now[:keep], k_dr[:keep])
        np.testing.assert_array_equal(k_now[keep:], 0.0)
    # every slot at or beyond seq_len is zero in the pool
    used = set()
    for b in range(3):
        for s in range(int(kv.seq_len[b])):
            used.add((int(kv.block_table[b, s // 16]), s % 16))
    for blk in range(kv.k_pool.shape[0]):
        for off in range(16):
            if (blk, off) not in used:
                assert not kv.k_pool[blk, :, off].any() and not kv.v_pool[blk, :, off].any()


def test_truncate_restores_prefix_state():
    cfg, w, kv = _tiny_state()
    before = kv.copy()
    _run_draft(cfg, w, kv, 3)
    O.kv_commit(kv, np.array([1, 3, 2], dtype=np.int32), "bf16")
    O.kv_truncate(kv, before.seq_len, "bf16")
    np.testing.assert_array_equal(kv.k_pool, before.k_pool)
    np.testing.assert_array_equal(kv.v_pool, before.v_pool)
    np.testing.assert_array_equal(kv.seq_len, before.seq_len)


def test_draft_appends_one_slot_per_step_and_attends_to_it():
    cfg, w, kv = _tiny_state(lens=(0,), K=2)
    res = _run_draft(cfg, w, kv, 2)
    k, v = O.kv_read_slots(kv, 0, 2, "bf16")
    assert np.abs(k).sum() > 0 and np.abs(v).sum() > 0
    assert res.logits.shape == (1, 2, cfg.vocab)


# -------------------------------------------- whole-step wiring (closed form)

def test_draft_chain_repeats_input_token_through_shared_embedding():
    """W_eh = [0 | I], W_o = 0, W_down = 0: x = RMSNorm(e), the layer adds
    nothing, so the logits are E . RMSNorm(RMSNorm(e)) and the self-dot of the
    input row wins.  Each later step embeds the previous draft, so the chain
    repeats the input token (recursion through the shared embedding, tied LM
    head)."""
    cfg, w = _tiny_weights(H=256, n_q=4, n_kv=2, d=64, F=128, V=4096, norm="ones")
    W = O.MTPWeights64.from_stored(w, "f32", cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    H = cfg.H
    W.w_eh = np.concatenate([np.zeros((H, H)), np.eye(H)], axis=1)
    W.w_o = np.zeros_like(W.w_o)
    W.w_down = np.zeros_like(W.w_down)
    kv = synth.make_kv(cfg, np.array([7]), extra_slots=5)
    tok = np.array([1234])
    rng = np.random.default_rng(0)
    res = O.draft(W, rng.standard_normal((1, H)), W.embed_rows(tok), np.array([7]), kv, 4)
    np.testing.assert_array_equal(res.ids, [[1234] * 4])


def test_draft_recursion_carries_pre_final_norm_hidden():
    """Embedding half of W_eh = 0 and the hidden half a coordinate
    permutation P that swaps the two halves of the coordinates: x = P RMSNorm(h).
    With the layer adding nothing, step k's state is P^k h up to scale.  Table
    rows are planted so that E[t_k] = P^k E[t_0]; the draft chain must walk
    t_1, t_2, t_3.  The final norm weight is zero on the second half, so a
    recursion on the post-final-norm state would leave only second-half
    coordinates after P, which the final norm then erases (all-zero logits,
    argmax 0)."""
    cfg, w = _tiny_weights(H=256, n_q=4, n_kv=2, d=64, F=128, V=4096, norm="ones")
    W = O.MTPWeights64.from_stored(w, "f32", cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    H = cfg.H
    rng = np.random.default_rng(1)
    half = H // 2
    perm = np.concatenate([half + rng.permutation(half), rng.permutation(half)])
    P = np.eye(H)[perm]
    W.w_eh = np.concatenate([P, np.zeros((H, H))], axis=1)
    W.w_o = np.zeros_like(W.w_o)
    W.w_down = np.zeros_like(W.w_down)
    W.w_norm_f = np.where(np.arange(H) < half, 1.0, 0.0)
    E = W.embed_stored.copy()
    chain = [11, 222, 3333, 4000]
    for a, b in zip(chain[:-1], chain[1:]):
        E[b] = P @ E[a]
    W.embed_stored = E
    W.lm_stored = E
    kv = synth.make_kv(cfg, np.array([3]), extra_slots=5)
    res = O.draft(W, W.embed_rows(np.array([chain[0]])) * 40.0, W.embed_rows(np.array([5])),
                  np.array([3]), kv, 3)
    np.testing.assert_array_equal(res.ids, [chain[1:]])
    # the wrong recursion (normed and weighted state) loses the chain
    h = W.embed_rows(np.array([chain[0]]))
    x1 = O.rmsnorm(h, W.w_norm_h, W.eps) @ P.T
    wrong = O.rmsnorm(O.rmsnorm(x1, W.w_norm_f, W.eps), W.w_norm_h, W.eps) @ P.T
    assert O.argmax_lowest(O.lm_head(wrong, W))[0] == 0 != chain[2]


def test_chain_ids_override_the_recursive_embedding():
    cfg, w = _tiny_weights(H=256, n_q=4, n_kv=2, d=64, F=128, V=4096, norm="ones")
    W = O.MTPWeights64.from_stored(w, "f32", cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    H = cfg.H
    W.w_eh = np.concatenate([np.zeros((H, H)), np.eye(H)], axis=1)
    W.w_o = np.zeros_like(W.w_o)
    W.w_down = np.zeros_like(W.w_down)
    kv = synth.make_kv(cfg, np.array([2]), extra_slots=5)
    res = O.draft(W, np.ones((1, H)), W.embed_rows(np.array([9])), np.array([2]), kv, 3,
                  chain_ids=np.array([[100, 200]]))
    np.testing.assert_array_equal(res.ids, [[9, 100, 200]])


def test_requests_are_independent():
    cfg, w, kv = _tiny_state(lens=(5, 21, 16))
    W = O.MTPWeights64.from_stored(w, "bf16", cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    di = synth.make_draft_inputs(cfg, w, kv.seq_len)
    kv_all = kv.copy()
    res_all = O.draft(W, O.widen(di.hidden, "bf16"), O.widen(di.embeds, "bf16"), di.positions, kv_all, 3)
    for b in range(3):
        kv_b = kv.copy()
        kv_b.block_table = kv.block_table[b:b + 1]
        kv_b.seq_len = kv.seq_len[b:b + 1].copy()
        kv_b.pending = kv.pending[b:b + 1].copy()
        res_b = O.draft(W, O.widen(di.hidden[b:b + 1], "bf16"), O.widen(di.embeds[b:b + 1], "bf16"),
                        di.positions[b:b + 1], kv_b, 3)
        np.testing.assert_allclose(res_b.logits[0], res_all.logits[b], rtol=1e-12, atol=1e-12)
