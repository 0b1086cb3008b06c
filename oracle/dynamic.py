"""Dynamic draft length for the oracle: the confidence stop and the
acceptance-driven draft count.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources (page title, section):
  [P3] "Speculative Decoding" (OpenVINO GenAI), "Fast Draft", "Configuration
       and Usage": with assistant_confidence_threshold the drafter keeps
       proposing while the candidate token's probability exceeds the
       threshold; "Backend Differences": the number of assistant tokens is
       adapted per step from recent acceptance.
  [P2] "MTP 深度解析", section 7.3: adapting the MTP depth to the live
       acceptance rate.

Readings (listed in the design notes):
  D1  the candidate's probability is the softmax probability of the draft
      token (the argmax) under the draft step's logits;
  D2  a request proposes the leading run of draft steps whose probability
      exceeds the threshold (a step at or below it, and every later step, is
      not proposed); the draft steps themselves still run;
  D3  the pages give no adaptation rule; the plainest is the usual
      heuristic: after a step whose drafts were all accepted the next draft
      count grows by 2, otherwise it shrinks by 1, within [k_min, k_max].
"""
import numpy as np


def draft_confidence(logits: np.ndarray) -> np.ndarray:
    """[..., V] logits -> probability of the argmax token: exp(z_max) / sum exp(z)
    = 1 / sum_v exp(z_v - z_max), in float64."""
    z = np.asarray(logits, dtype=np.float64)
    m = z.max(axis=-1, keepdims=True)
    return 1.0 / np.exp(z - m).sum(axis=-1)


def num_drafts_from_confidence(conf: np.ndarray, tau: float) -> np.ndarray:
    """[B, K] probabilities -> [B] length of the leading run with conf > tau."""
    conf = np.asarray(conf)
    out = np.zeros(conf.shape[0], dtype=np.int32)
    for b in range(conf.shape[0]):
        n = 0
        while n < conf.shape[1] and conf[b, n] > tau:
            n += 1
        out[b] = n
    return out


def next_k(K: int, accepted: int, drafted: int, k_min: int, k_max: int) -> int:
    """D3: the next step's draft count after `accepted` of `drafted` drafts
    were accepted with draft count K."""
    if drafted > 0 and accepted == drafted:
        return min(K + 2, k_max)
    return max(K - 1, k_min)
