"""Training forward of the block drafter: the position-weighted loss value.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

Follows "DFlash: Block Diffusion for Flash Speculative Decoding" (Training,
§4.2: features from the clean sequence, anchor-based blocks, packed blocks
with a sparse mask, loss weighting, frozen embeddings and head) and "DFlash:
Why a Diffusion Drafter Can Accelerate an Autoregressive Model" §6 (eq. 12,
Algorithm 2):

    L = mean over anchors a of  sum_{k=1}^{B-1} exp(-(k-1)/lambda) * [-log q_k(x_{a+k} | c_a, x_a)]

where q_k is the drafter's softmax at block row k of the block
[x_a, MASK x (B-1)] at positions a .. a+B-1, and c_a is the legal context:
the fused target features of the positions before a.

Readings where the pages leave the step open:
- the frozen target runs once, causally, over the whole clean sequence; its
  selected-layer states at positions < a are the context of the block at a
  (no feature of a token at or after the anchor: the review's "hide target
  features containing future tokens relative to each anchor");
- blocks see their own rows (bidirectionally) and their legal context only,
  never another block (the digest's "attention across blocks is disallowed");
- an anchor a needs 1 <= a and a + B - 1 < N, so the context is non-empty and
  every predicted position has a label;
- the expectation over anchors is the mean over the given anchors; lambda is
  7, 5 and 4 for B = 16, 10 and 8 (the appendix values the review quotes),
  otherwise supplied by the caller;
- the value only: target, embeddings and head are frozen and no gradient is
  taken here.
"""
from __future__ import annotations

import numpy as np

from .model import Model, attention

LAMBDA_FOR_BLOCK = {16: 7.0, 10: 5.0, 8: 4.0}


def position_weights(B: int, lam: float) -> np.ndarray:
    """exp(-(k-1)/lambda) for the predicted positions k = 1 .. B-1 (eq. 12)."""
    k = np.arange(1, B, dtype=np.float64)
    return np.exp(-(k - 1.0) / lam)


def _lam(model: Model, lam):
    if lam is not None:
        return float(lam)
    B = model.cfg.block_size
    if B not in LAMBDA_FOR_BLOCK:
        raise ValueError(f"no lambda for block size {B}; pass one")
    return LAMBDA_FOR_BLOCK[B]


def context_features(model: Model, x) -> np.ndarray:
    """Fused target features of every position of the clean sequence [N, d]."""
    _, sel = model.target_forward(np.asarray(x, dtype=np.int64), model.new_target_cache(), want_logits=False)
    return model.fuse(sel)


def _check_anchors(model: Model, x, anchors):
    B, N = model.cfg.block_size, len(x)
    for a in anchors:
        if not (1 <= a and a + B - 1 < N):
            raise ValueError(f"anchor {a} outside [1, {N - B}]")


def block_logits(model: Model, feats: np.ndarray, x, a: int) -> np.ndarray:
    """Drafter logits [B, V] of the block at anchor a, with context features[:a]."""
    dc = model.new_draft_cache()
    model.append_context(feats[:a], dc)
    return model.draft_forward(int(x[a]), dc)


def block_loss(logits: np.ndarray, x, a: int, lam: float) -> float:
    """sum_k w_k * -log softmax(logits[k])[x[a+k]] over k = 1 .. B-1."""
    B = logits.shape[0]
    z = logits[1:] - logits[1:].max(axis=-1, keepdims=True)
    logp = z - np.log(np.exp(z).sum(axis=-1, keepdims=True))
    labels = np.asarray(x[a + 1: a + B], dtype=np.int64)
    nll = -logp[np.arange(B - 1), labels]
    return float((position_weights(B, lam) * nll).sum())


def training_loss(model: Model, x, anchors, lam=None) -> float:
    """eq. 12 with one block per anchor, each block its own drafter pass."""
    x = np.asarray(x, dtype=np.int64)
    _check_anchors(model, x, anchors)
    lam = _lam(model, lam)
    feats = context_features(model, x)
    return float(np.mean([block_loss(block_logits(model, feats, x, int(a)), x, int(a), lam) for a in anchors]))


def packed_block_logits(model: Model, feats: np.ndarray, x, anchors) -> np.ndarray:
    """All blocks in one drafter pass (the digest's packed training forward): the
    context K/V of every position are projected once, the m blocks' rows are
    concatenated, and the attention mask lets a row of block i see the context
    positions before a_i and the rows of block i only.  Returns [m, B, V]."""
    c = model.cfg
    B, m, N = c.block_size, len(anchors), feats.shape[0]
    ctx = model.new_draft_cache()
    model.append_context(feats, ctx)                    # positions 0 .. N-1
    anchors = np.asarray(anchors, dtype=np.int64)
    tokens = np.concatenate([[int(x[a])] + [c.mask_token] * (B - 1) for a in anchors]).astype(np.int64)
    pos = np.concatenate([np.arange(a, a + B) for a in anchors])
    blk = np.repeat(np.arange(m), B)
    visible = np.zeros((m * B, N + m * B), dtype=bool)
    visible[:, :N] = np.arange(N)[None, :] < anchors[blk][:, None]
    visible[:, N:] = blk[:, None] == blk[None, :]
    h = model.w("embed")[tokens].copy()
    for l in range(c.draft_layers):
        p = f"d{l}"
        q, kb, vb = model._qkv(p, h, pos, True)
        K = np.concatenate([ctx.k[l], kb], axis=0)
        V = np.concatenate([ctx.v[l], vb], axis=0)
        h = model._attn_out_mlp(p, h, attention(q, K, V, visible))
    return model.logits(h, "draft_norm").reshape(m, B, -1)


def packed_training_loss(model: Model, x, anchors, lam=None) -> float:
    x = np.asarray(x, dtype=np.int64)
    _check_anchors(model, x, anchors)
    lam = _lam(model, lam)
    lg = packed_block_logits(model, context_features(model, x), x, anchors)
    return float(np.mean([block_loss(lg[i], x, int(a), lam) for i, a in enumerate(anchors)]))
