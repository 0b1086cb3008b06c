"""Pins of how the oracle's draft step wires its attention into the step, and
an independent restatement of the whole step.  CPU only.

What each pin fixes (sources: "MTP (Multi-Token Prediction)", "Architecture":
a standard decoder layer run once per recursive step; "How OpenVINO MTP
Speculative Decoding Works Internally", "Why the MTP graph is a single decoder
layer": its own one-layer cache, appended by every step):

* the attention span of draft step k: the committed entries plus drafted
  entries 1..k, its own entry included (step k of a request with L committed
  entries attends over exactly L + k slots);
* the rotary position of draft step k: positions[b] + k - 1 for the query and
  the key it appends;
* the attention primitive against an explicit softmax(Q K^T / sqrt(d)) V with
  the GQA groups expanded by repetition;
* the whole step a1..a7 against a second float64 program written in another
  form (complex rotation, masked attention over the logical sequence, split
  halves of W_eh) at the tiny fp32 workload's shape.

Every pin comes with a test that plants a plausible mistake in the oracle (on
the CPU, by replacing one of its module functions for the duration of the
test) and checks that the pin then fails.
"""
import math

import numpy as np
import pytest

import oracle as O
import oracle.mtp_oracle as OM
import synth


def _f32_cfg(H=256, n_q=4, n_kv=2, d=64, F=128, V=4096, seed=60, paged=True):
    return synth.MTPShape("pin", H=H, n_q=n_q, n_kv=n_kv, head_dim=d, ffn=F, vocab=V, batch=1, K=3,
                          dtype="f32", ctx_lo=1, ctx_hi=1, paged_shuffle=paged, seed_index=seed)


def _weights64(cfg, norm="ones"):
    w = synth.make_weights(cfg, norm=norm)
    return O.MTPWeights64.from_stored(w, "f32", cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)


def _kv(cfg, L, extra=8):
    return synth.make_kv(cfg, np.array([L], dtype=np.int32), extra_slots=extra)


def _stored(kv, L_total, which):
    """Raw float32 entries of request 0's first L_total slots, [T, n_kv, d],
    read straight from the pool through the block table."""
    pool = kv.k_pool if which == "k" else kv.v_pool
    out = []
    for s in range(L_total):
        out.append(pool[int(kv.block_table[0, s // kv.block_size]), :, s % kv.block_size, :])
    return np.stack(out).astype(np.float64)


# ------------------------------------------------------- (a) attention span

def _span_pin(L, K):
    """With W_q = 0 every score is 0, so the attention output of draft step k
    is the plain mean of the values over exactly the slots it attends to.
    W_o = I and W_down = 0 make the step's output hidden state x_k + o_k,
    so o_k = hidden_out - x_k is observable.  The expected values are built
    independently: the L prefilled values come from the generator in logical
    order, and the drafted value of step j is W_v RMSNorm(x_j), rounded to
    float32 like the cache, with x_j recomputed from the (pinned) eh_proj and
    the previous run's hidden output and draft id.  A span one slot too long
    (a zero slot joins the mean) or one too short (the step's own entry is
    missing) fails."""
    cfg = _f32_cfg()
    W = _weights64(cfg)
    H, d = cfg.H, cfg.head_dim
    assert cfg.q_dim == H
    W.w_q = np.zeros_like(W.w_q)
    W.w_o = np.eye(H)
    W.w_down = np.zeros_like(W.w_down)
    rng = np.random.default_rng(100 + L)
    h0 = rng.standard_normal((1, H))
    tok0 = np.array([77])
    pos = np.array([L + 3])                    # positions need not equal the slot count
    prefill_v = synth.normal(cfg.seed, synth.stream_id("v_pool"), (L, cfg.n_kv, d), dtype="f32",
                             offset=0).astype(np.float64) if L else np.zeros((0, cfg.n_kv, d))
    h_prev, e_prev = h0, W.embed_rows(tok0)
    drafted_v = []
    group = cfg.n_q // cfg.n_kv
    for k in range(1, K + 1):
        kv = _kv(cfg, L)
        res = O.draft(W, h0, W.embed_rows(tok0), pos, kv, k)
        x_k = O.eh_proj(h_prev, e_prev, W)
        v_k = (O.rmsnorm(x_k, W.w_norm_in, W.eps) @ W.w_v.T).astype(np.float32).astype(np.float64)
        drafted_v.append(v_k.reshape(cfg.n_kv, d))
        vals = np.concatenate([prefill_v, np.stack(drafted_v)], axis=0)   # [L + k, n_kv, d]
        assert vals.shape[0] == L + k
        expect = vals.mean(axis=0)[np.arange(cfg.n_q) // group].reshape(-1)
        o_k = (res.hidden_out - x_k)[0]
        np.testing.assert_allclose(o_k, expect, rtol=1e-10, atol=1e-12)
        # the step's own appended value is in the cache at slot L + k - 1
        np.testing.assert_array_equal(_stored(kv, L + k, "v")[L + k - 1], drafted_v[-1])
        h_prev = res.hidden_out
        e_prev = W.embed_rows(res.ids[:, k - 1])


@pytest.mark.parametrize("L", [0, 14])
def test_draft_attention_span_is_committed_plus_drafted_including_own(L):
    """L = 0: step 1 sees only its own entry (o = v_1 exactly), step 2 the
    mean of v_1 and v_2, step 3 of three.  L = 14 with K = 3 crosses a
    16-slot block boundary of a shuffled pool."""
    _span_pin(L, 3)


def test_span_pin_fails_when_the_span_is_one_slot_too_long(monkeypatch):
    real = OM.kv_read_slots
    monkeypatch.setattr(OM, "kv_read_slots", lambda kv, b, n, dt: real(kv, b, n + 1, dt))
    with pytest.raises(AssertionError):
        _span_pin(0, 3)


def test_span_pin_fails_when_the_own_entry_is_left_out(monkeypatch):
    real = OM.kv_read_slots
    monkeypatch.setattr(OM, "kv_read_slots", lambda kv, b, n, dt: real(kv, b, n - 1, dt))
    with pytest.raises((AssertionError, ValueError)):     # L = 0: step 1 has no key at all
        _span_pin(14, 3)
    with pytest.raises((AssertionError, ValueError)):
        _span_pin(0, 3)


# ---------------------------------------------------- (b) rotary position

def _position_pin(K, p=1000, A=8.0):
    """One prefilled key at slot 0, written as if rotated for position p - 1:
    A (cos(p-1) e_0 + sin(p-1) e_{d/2}) (pair 0 turns by 1 radian per
    position).  W_eh = [I | 0], unit norm weights and h = e_0 make the
    normalised input sqrt(H) e_0 at step 1; W_q reads only input coordinate 0,
    so every query head is a multiple of e_0 before rotation; W_k = 0 makes
    the drafted keys zero (score 0).  The query of step k sits at position
    P = p + k - 1, so its score against the prefilled key (as stored) is
    a_k (cos P k0[0] + sin P k0[d/2]) / sqrt(d) = a_k A cos(k) / sqrt(d) up to
    the key's float32 rounding (a_k the query's pre-rotation length), and
    the attention output is the logistic mix of the prefilled value and the
    drafted values.  A query at p + k instead (off by one) scores
    a_k A cos(k + 1) / sqrt(d): for k = 1, +4.3 turns into -3.3 and the mix
    flips from the prefilled value to the step's own."""
    cfg = _f32_cfg(paged=False)
    W = _weights64(cfg)
    H, d, n_q, n_kv = cfg.H, cfg.head_dim, cfg.n_q, cfg.n_kv
    half = d // 2
    group = n_q // n_kv
    W.w_eh = np.concatenate([np.eye(H), np.zeros((H, H))], axis=1)
    W.w_q = np.zeros_like(W.w_q)
    W.w_q[np.arange(n_q) * d, 0] = A / math.sqrt(H)          # q_h = (A / 16) n_0 e_0
    W.w_k = np.zeros_like(W.w_k)
    rng = np.random.default_rng(7)
    W.w_v = np.zeros_like(W.w_v)
    W.w_v[:, 0] = rng.standard_normal(cfg.kv_dim)
    W.w_o = np.eye(H)
    W.w_down = np.zeros_like(W.w_down)
    kv = _kv(cfg, 1, extra=8)
    k0 = np.zeros((n_kv, d))
    k0[:, 0] = A * math.cos(p - 1)
    k0[:, half] = A * math.sin(p - 1)
    v0 = rng.standard_normal((n_kv, d))
    kv.k_pool[0, :, 0, :] = k0
    kv.v_pool[0, :, 0, :] = v0
    v0 = v0.astype(np.float32).astype(np.float64)
    k0s = k0.astype(np.float32).astype(np.float64)             # as the float32 cache holds it
    h = np.zeros((1, H))
    h[0, 0] = 3.0
    tok = np.array([5])
    res = O.draft(W, h, W.embed_rows(tok), np.array([p]), kv, K)
    # replay the step's inputs with pinned primitives, then the closed form
    h_prev, e_prev = h, W.embed_rows(tok)
    drafted = []
    for k in range(1, K + 1):
        x_k = O.eh_proj(h_prev, e_prev, W)
        n0 = O.rmsnorm(x_k, W.w_norm_in, W.eps)[0, 0]
        a_k = A / math.sqrt(H) * n0                            # |q| before rotation
        drafted.append((W.w_v[:, 0] * n0).astype(np.float32).astype(np.float64).reshape(n_kv, d))
        P = p + k - 1                                          # the query's position
        s0 = a_k * (math.cos(P) * k0s[0, 0] + math.sin(P) * k0s[0, half]) / math.sqrt(d)
        wts = np.array([math.exp(s0)] + [1.0] * k)
        vals = np.concatenate([v0[None], np.stack(drafted)], axis=0)      # [1 + k, n_kv, d]
        mix = np.tensordot(wts / wts.sum(), vals, axes=1)                   # [n_kv, d]
        expect = mix[np.arange(n_q) // group].reshape(-1)
        kv_k = _kv(cfg, 1, extra=8)
        kv_k.k_pool[0, :, 0, :] = k0
        kv_k.v_pool[0, :, 0, :] = v0
        r_k = O.draft(W, h, W.embed_rows(tok), np.array([p]), kv_k, k)
        np.testing.assert_allclose((r_k.hidden_out - x_k)[0], expect, rtol=1e-9, atol=1e-12)
        h_prev, e_prev = r_k.hidden_out, W.embed_rows(r_k.ids[:, k - 1])
    np.testing.assert_array_equal(res.hidden_out, h_prev)
    return res


def test_draft_rotary_position_is_position_plus_step_minus_one():
    _position_pin(3)


def test_position_pin_fails_when_rotation_is_one_position_late(monkeypatch):
    real = OM.rope
    monkeypatch.setattr(OM, "rope", lambda x, pos, theta: real(x, pos + 1, theta))
    with pytest.raises(AssertionError):
        _position_pin(3)


def test_position_pin_fails_when_rotation_is_one_position_early(monkeypatch):
    real = OM.rope
    monkeypatch.setattr(OM, "rope", lambda x, pos, theta: real(x, pos - 1, theta))
    with pytest.raises(AssertionError):
        _position_pin(3)


# ------------------------------------------- (c) naive softmax attention

def _naive_attention(q, k, v):
    """softmax(Q K^T / sqrt(d)) V, with the kv heads repeated so that query
    head h meets kv head h // (n_q / n_kv); the softmax is exp / sum without
    any shift (the inputs are small)."""
    n_q, d = q.shape
    T, n_kv, _ = k.shape
    kr = np.repeat(k, n_q // n_kv, axis=1)          # [T, n_q, d]
    vr = np.repeat(v, n_q // n_kv, axis=1)
    s = np.einsum("hd,thd->ht", q, kr) / math.sqrt(d)
    p = np.exp(s)
    p = p / p.sum(axis=1, keepdims=True)
    return np.einsum("ht,thd->hd", p, vr)


@pytest.mark.parametrize("n_q,n_kv,d,T", [(1, 1, 4, 1), (4, 2, 8, 7), (8, 1, 16, 33), (16, 2, 64, 130),
                                          (6, 3, 32, 2), (32, 8, 128, 50)])
def test_attention_matches_naive_softmax_on_random_inputs(n_q, n_kv, d, T):
    rng = np.random.default_rng(n_q * 1000 + T)
    q = rng.standard_normal((n_q, d))
    k = rng.standard_normal((T, n_kv, d))
    v = rng.standard_normal((T, n_kv, d))
    np.testing.assert_allclose(O.attention(q, k, v), _naive_attention(q, k, v), rtol=1e-12, atol=1e-13)


def test_naive_softmax_check_catches_a_wrong_group_map_and_a_missing_scale():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((8, 16))
    k = rng.standard_normal((9, 2, 16))
    v = rng.standard_normal((9, 2, 16))
    naive = _naive_attention(q, k, v)
    interleaved = np.stack([O.attention(q[h:h + 1], k[:, [h % 2]], v[:, [h % 2]])[0] for h in range(8)])
    assert not np.allclose(interleaved, naive, rtol=1e-6)
    assert not np.allclose(O.attention(q * math.sqrt(16), k, v), naive, rtol=1e-6)


# ---------------------------------------------- (d) whole-step restatement

def _restated_draft(w, H, n_q, n_kv, d, eps, theta, hidden, embeds, positions, prefix_k, prefix_v, K,
                    chain=None):
    """A second float64 statement of draft steps a1..a7 for one request,
    written without the oracle: RMSNorm as x * (||x||^2 / H + eps)^-1/2,
    the concatenation as the two halves of W_eh applied separately, rotation
    as multiplication of the complex numbers x_i + i x_{i+d/2} by
    exp(i pos theta^(-2i/d)), attention as one masked softmax over the whole
    logical sequence (prefix, then drafted entries) with the query heads
    grouped by reshaping, the appended entries rounded to float32 (the
    cache's dtype in the fp32 head), and the tied LM head.  ``chain`` [K-1],
    when given, replaces the recursive draft ids as the next steps' tokens.
    Returns logits [K, V], ids [K], the last hidden [H] and the appended
    (k, v) [K, n_kv, d]."""
    f = lambda name: np.asarray(w[name], dtype=np.float64)
    E = f("embed")
    V = E.shape[0]
    G = n_q // n_kv

    def norm(x, wt):
        return x * (np.dot(x, x) / x.size + eps) ** -0.5 * wt

    def rotate(x, pos):                       # x [heads, d]
        z = x[:, :d // 2] + 1j * x[:, d // 2:]
        z = z * np.exp(1j * pos * theta ** (-np.arange(d // 2) * 2.0 / d))
        return np.concatenate([z.real, z.imag], axis=1)

    Lp = prefix_k.shape[0]
    keys = np.zeros((Lp + K, n_kv, d))
    vals = np.zeros((Lp + K, n_kv, d))
    keys[:Lp], vals[:Lp] = prefix_k, prefix_v
    h, e = np.asarray(hidden, np.float64), np.asarray(embeds, np.float64)
    logits, ids = np.zeros((K, V)), np.zeros(K, dtype=np.int64)
    for step in range(K):
        pos = int(positions) + step
        x = f("w_eh")[:, :H] @ norm(h, f("w_norm_h")) + f("w_eh")[:, H:] @ norm(e, f("w_norm_e"))
        n = norm(x, f("w_norm_in"))
        q = rotate((f("w_q") @ n).reshape(n_q, d), pos)
        keys[Lp + step] = rotate((f("w_k") @ n).reshape(n_kv, d), pos).astype(np.float32)
        vals[Lp + step] = (f("w_v") @ n).reshape(n_kv, d).astype(np.float32)
        T = Lp + K
        visible = np.arange(T) <= Lp + step
        s = np.einsum("cgd,tcd->cgt", q.reshape(n_kv, G, d), keys) / math.sqrt(d)
        s = np.where(visible, s, -np.inf)
        s = s - s.max(axis=-1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=-1, keepdims=True)
        o = np.einsum("cgt,tcd->cgd", p, vals).reshape(-1)
        h1 = x + f("w_o") @ o
        n2 = norm(h1, f("w_norm_post"))
        g, u = f("w_gate") @ n2, f("w_up") @ n2
        h2 = h1 + f("w_down") @ (g / (1.0 + np.exp(-g)) * u)
        z = E @ norm(h2, f("w_norm_f"))
        logits[step] = z
        ids[step] = int(np.flatnonzero(z == z.max())[0])
        h = h2
        e = E[ids[step] if chain is None else int(chain[step])] if step + 1 < K else e
    return logits, ids, h, keys[Lp:], vals[Lp:]


def _whole_step_pin(cfg=synth.TINY_F32, norm="random"):
    """The tiny fp32 workload's shape (H=256, 4 q / 2 kv heads, d=64,
    F=1024, V=4096, 128 committed entries, K=3) with N(1, 0.1) norm weights:
    the oracle and the restatement agree to 1e-5 (normwise, per step) on the
    logits, the last hidden state and the appended entries, and exactly on
    the draft ids."""
    w = synth.make_weights(cfg, norm=norm)
    lens = synth.context_lengths(cfg)
    kv = synth.make_kv(cfg, lens, extra_slots=cfg.K + 2)
    di = synth.make_draft_inputs(cfg, w, lens)
    L = int(lens[0])
    prefix_k, prefix_v = _stored(kv, L, "k"), _stored(kv, L, "v")
    W = O.MTPWeights64.from_stored(w, cfg.dtype, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    res = O.draft(W, O.widen(di.hidden, cfg.dtype), O.widen(di.embeds, cfg.dtype), di.positions, kv, cfg.K)
    z, ids, h, ak, av = _restated_draft(w, cfg.H, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta,
                                        O.widen(di.hidden, cfg.dtype)[0], O.widen(di.embeds, cfg.dtype)[0],
                                        di.positions[0], prefix_k, prefix_v, cfg.K)
    rel = lambda a, b: float(np.max(np.abs(a - b)) / np.max(np.abs(b)))
    for k in range(cfg.K):
        assert rel(res.logits[0, k], z[k]) <= 1e-5, k
    np.testing.assert_array_equal(res.ids[0], ids)
    assert rel(res.hidden_out[0], h) <= 1e-5
    got_k, got_v = _stored(kv, L + cfg.K, "k")[L:], _stored(kv, L + cfg.K, "v")[L:]
    for k in range(cfg.K):
        assert rel(got_k[k], ak[k]) <= 1e-5 and rel(got_v[k], av[k]) <= 1e-5, k


def test_whole_draft_step_matches_independent_restatement():
    _whole_step_pin()


def test_whole_step_restatement_agrees_bf16_shape():
    """The same restatement on a small bf16 head with a shuffled paged cache
    (30 committed entries, K = 4: the drafted slots cross a 16-slot block
    boundary) and a given token chain.  The oracle's cache rounds appended
    entries to bf16 and the restatement to float32, so the bound is the
    bf16 one: 1e-2 normwise per step."""
    cfg = synth.MTPShape("pin_bf16", H=128, n_q=4, n_kv=2, head_dim=32, ffn=256, vocab=1024, batch=1, K=4,
                         dtype="bf16", ctx_lo=30, ctx_hi=30, paged_shuffle=True, seed_index=61)
    w = synth.make_weights(cfg, norm="random")
    lens = synth.context_lengths(cfg)
    kv = synth.make_kv(cfg, lens, extra_slots=cfg.K + 2)
    di = synth.make_draft_inputs(cfg, w, lens)
    L = int(lens[0])
    rows = lambda pool: O.widen(np.stack([pool[int(kv.block_table[0, s // 16]), :, s % 16] for s in range(L)]),
                                "bf16")
    pk, pv = rows(kv.k_pool), rows(kv.v_pool)
    W = O.MTPWeights64.from_stored(w, "bf16", cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    hid, emb = O.widen(di.hidden, "bf16"), O.widen(di.embeds, "bf16")
    chain = np.array([3, 900, 511])
    res = O.draft(W, hid, emb, di.positions, kv, cfg.K, chain_ids=chain[None])
    wf = {k: O.widen(v, "bf16") for k, v in w.items()}
    z, _, _, _, _ = _restated_draft(wf, cfg.H, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta,
                                    hid[0], emb[0], di.positions[0], pk, pv, cfg.K, chain=chain)
    for k in range(cfg.K):
        assert np.max(np.abs(res.logits[0, k] - z[k])) <= 1e-2 * np.max(np.abs(z[k])), k


_MUTATIONS = {
    "concat order swapped": ("eh_proj", lambda real: (lambda h, e, W: real(e, h, W))),
    "rotation one position late": ("rope", lambda real: (lambda x, pos, th: real(x, pos + 1, th))),
    "attention without 1/sqrt(d)": ("attention", lambda real: (lambda q, k, v: real(q * math.sqrt(q.shape[1]), k, v))),
    "gate and up swapped": ("swiglu_mlp", lambda real: (lambda n, g, u, dn: real(n, u, g, dn))),
    "norm weight dropped": ("rmsnorm", lambda real: (lambda x, w, eps: real(x, np.ones_like(w), eps))),
    "span one slot too long": ("kv_read_slots", lambda real: (lambda kv, b, n, dt: real(kv, b, n + 1, dt))),
    "keys read as values": ("kv_read_slots", lambda real: (lambda kv, b, n, dt: (real(kv, b, n, dt)[0],) * 2)),
}


@pytest.mark.parametrize("name", sorted(_MUTATIONS))
def test_whole_step_pin_fails_on_planted_mistake(monkeypatch, name):
    attr, make = _MUTATIONS[name]
    monkeypatch.setattr(OM, attr, make(getattr(OM, attr)))
    with pytest.raises(AssertionError):
        _whole_step_pin()
