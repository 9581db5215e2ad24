"""Accounting formulas the pages state: acceptance length, cycle latency,
speedup, fusion-projection memory and context-layer selection.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  The product's benchmark
computes its own numbers; these functions exist to be pinned against the
pages' printed values and to check the benchmark's arithmetic in tests.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np


def tau_from_accepts(accepted: Sequence[int]) -> float:
    """Acceptance length per cycle, tau = E[A + 1]: the bonus token counts
    ("DFlash: Why a Diffusion Drafter Can Accelerate an Autoregressive Model"
    §2.3 eq. 2; the digest's Paper vs code, "Acceptance length counts the
    bonus token")."""
    a = np.asarray(accepted, dtype=np.float64)
    return float(np.mean(a + 1.0))


def tau_tail_sum(accepted: Sequence[int], m: int) -> float:
    """Tail-sum form of eq. 2: 1 + sum_{k=1..m} P(A >= k)."""
    a = np.asarray(accepted)
    return 1.0 + sum(float(np.mean(a >= k)) for k in range(1, m + 1))


def tau_geometric(a: float, m: int) -> float:
    """Eq. 3 of the review: tau = (1 - a^(m+1)) / (1 - a) for a constant
    per-token survival probability a != 1 and m = B - 1 proposals."""
    return (1.0 - a ** (m + 1)) / (1.0 - a)


def cycle_latency(t_draft: float, t_verify: float, tau: float, t_other: float = 0.0) -> float:
    """Per-token latency L = (T_draft + T_verify [+ T_other]) / tau
    (the digest's eq. 1; the review's eq. 4 adds the orchestration term)."""
    return (t_draft + t_verify + t_other) / tau


def speedup(tau: float, r_draft: float, r_verify: float, r_other: float = 0.0) -> float:
    """Review eq. 4 with costs normalised by the AR per-token time:
    S = tau / (r_d + r_v + r_o); S > 1 iff tau > r_d + r_v + r_o (eq. 5)."""
    return tau / (r_draft + r_verify + r_other)


def effective_tokens_per_s(batch: int, tau: float, t_draft_ms: float, t_verify_ms: float) -> float:
    """Tokens emitted per second by a batch of independent sequences: each
    round emits tau tokens per sequence in (t_draft + t_verify)."""
    return batch * tau / ((t_draft_ms + t_verify_ms) * 1e-3)


def fusion_param_bytes(width: int, n_features: int, bytes_per: int = 2) -> int:
    """Parameters of the fusion map W_c [width, n_features * width] in bytes
    (review §5.3 eq. 11)."""
    return n_features * width * width * bytes_per


def fusion_io_bytes(width: int, n_features: int, rows: int, bytes_per: int = 2):
    """(concatenated input bytes, projected output bytes) for ``rows`` positions."""
    return rows * n_features * width * bytes_per, rows * width * bytes_per


def draft_cache_bytes(batch: int, draft_layers: int, ctx_len: int, kv_width: int, bytes_per: int) -> int:
    """Rough draft context cache size 2 * b * d * L * d_kv * s (review §5.3)."""
    return 2 * batch * draft_layers * ctx_len * kv_width * bytes_per


def context_layer_ids(n_target_layers: int, n_features: int) -> list:
    """Evenly spaced target layers from index 1 to index L-3 (the digest's
    Paper vs code, "Context layers match the text").  Returns 0-based layer
    indices; the hidden-states list read by the code is offset by one because
    its entry 0 is the embedding output."""
    start, end = 1, n_target_layers - 3
    if n_features == 1:
        return [start]
    return [int(round(start + i * (end - start) / (n_features - 1))) for i in range(n_features)]
