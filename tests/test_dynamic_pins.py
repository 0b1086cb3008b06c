"""Pins of the dynamic draft length ("Speculative Decoding" (OpenVINO GenAI),
"Fast Draft", "Backend Differences"): the draft confidence against closed
forms, the leading-run rule, the adaptive count on hand-worked sequences, and
the C ABI's host-side count against the oracle's.  CPU only."""
import math

import numpy as np

from oracle import dynamic as D


def test_confidence_closed_forms():
    V = 1000
    # uniform logits: 1 / V
    assert abs(D.draft_confidence(np.zeros((1, V)))[0] - 1.0 / V) < 1e-15
    # one logit L above the rest: e^L / (e^L + V - 1)
    for L in (0.5, 3.0, 20.0):
        z = np.zeros(V)
        z[7] = L
        assert abs(D.draft_confidence(z) - math.exp(L) / (math.exp(L) + V - 1)) < 1e-12
    # two logits tied at the top: at most 1/2
    z = np.zeros(V)
    z[1] = z[2] = 10.0
    assert abs(D.draft_confidence(z) - math.exp(10) / (2 * math.exp(10) + V - 2)) < 1e-12
    # invariant under a common shift, and a softmax probability in (0, 1]
    rng = np.random.default_rng(1)
    z = rng.standard_normal((4, V)) * 3
    np.testing.assert_allclose(D.draft_confidence(z), D.draft_confidence(z + 123.0), rtol=1e-12)
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(D.draft_confidence(z), p.max(axis=1), rtol=1e-12)


def test_leading_run_rule():
    conf = np.array([[0.9, 0.8, 0.3, 0.95],
                     [0.2, 0.99, 0.99, 0.99],
                     [0.5, 0.5, 0.5, 0.5],
                     [0.51, 0.52, 0.53, 0.54]])
    np.testing.assert_array_equal(D.num_drafts_from_confidence(conf, 0.5), [2, 0, 0, 4])
    # the threshold is strict: a step exactly at it is not proposed
    np.testing.assert_array_equal(D.num_drafts_from_confidence(np.array([[0.4, 0.7]]), 0.4), [0])


def test_adaptive_count_hand_sequence():
    K, seq = 5, []
    # all accepted twice, then a rejection, then nothing drafted, then all
    for acc, drafted in ((5, 5), (7, 7), (2, 8), (0, 0), (7, 7)):
        K = D.next_k(K, acc, drafted, 1, 8)
        seq.append(K)
    assert seq == [7, 8, 7, 6, 8]
    assert D.next_k(1, 0, 1, 1, 8) == 1          # never below k_min


def test_c_abi_adapt_k_matches_oracle():
    import ctypes, os
    lib = ctypes.CDLL(os.path.join(os.path.dirname(os.path.dirname(__file__)),
                                   "mtp_self_speculative_gb300", "libmtp.so"))
    f = lib.mtp_adapt_k
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 5
    rng = np.random.default_rng(2)
    for _ in range(500):
        K = int(rng.integers(1, 9))
        drafted = int(rng.integers(0, K + 1))
        acc = int(rng.integers(0, drafted + 1))
        assert f(K, acc, drafted, 1, 8) == D.next_k(K, acc, drafted, 1, 8)
