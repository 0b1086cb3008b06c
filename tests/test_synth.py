"""The seeded input generator: published SplitMix64 outputs, determinism,
sub-range regeneration, and the recipes' distributions.  CPU only."""
import numpy as np

import synth


def test_splitmix64_published_sequence():
    # SplitMix64 from state 1234567 (reference outputs of Vigna's splitmix64.c)
    np.testing.assert_array_equal(
        synth.splitmix64_seq(1234567, 5),
        np.array([6457827717110365317, 3203168211198807973, 9817491932198370423,
                  4593380528125082431, 16408922859458223821], dtype=np.uint64))


def test_counter_subranges_match_full_draw():
    full = synth.normal(3, 7, (10000,), dtype="bf16")
    part = synth.normal(3, 7, (100,), dtype="bf16", offset=5000)
    np.testing.assert_array_equal(full[5000:5100], part)
    assert not np.array_equal(full, synth.normal(3, 8, (10000,), dtype="bf16"))


def test_normal_moments_and_bf16_rounding():
    x = synth.normal(5, 1, (400000,), 0.0, 0.02, dtype="f32").astype(np.float64)
    assert abs(x.mean()) < 3 * 0.02 / np.sqrt(len(x)) * 2
    assert abs(x.std() / 0.02 - 1) < 0.01
    b = synth.bf16_to_f32(synth.normal(5, 1, (400000,), 0.0, 0.02, dtype="bf16")).astype(np.float64)
    assert np.max(np.abs(b - x) / np.abs(x)) <= 2.0 ** -8


def test_uniform_int_range():
    u = synth.uniform_int(1, 2, (200000,), 512, 8193)
    assert u.min() >= 512 and u.max() <= 8192
    assert abs(u.mean() - (512 + 8192) / 2) < 30


def test_paged_kv_layout_roundtrip():
    cfg = synth.shrink(synth.QWEN3_8B_CB32, H=64, n_q=4, n_kv=2, head_dim=8, ffn=32, vocab=128, batch=5)
    lens = np.array([1, 16, 17, 40, 0])
    kv = synth.make_kv(cfg, lens, extra_slots=3)
    # every request's entries come back in slot order through the block table
    for b, L in enumerate(lens):
        want = synth.normal(cfg.seed, synth.stream_id("k_pool"), (int(L), 2, 8), dtype="bf16",
                            offset=(b << 24) * 16)
        got = np.stack([kv.k_pool[kv.block_table[b, s // 16], :, s % 16] for s in range(L)]) if L else want
        np.testing.assert_array_equal(got, want)
    # blocks are distinct across requests
    used = kv.block_table[kv.block_table >= 0]
    assert len(np.unique(used)) == len(used)
