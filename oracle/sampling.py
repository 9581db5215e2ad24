"""Draft-and-verify rounds at temperature T > 0: speculative rejection sampling.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

Follows "DFlash: Why a Diffusion Drafter Can Accelerate an Autoregressive
Model" §4.2 (eq. 6-8) and Algorithm 1 (steps 2-3, 7-8 and 10), and the
sampling rule of "DFlash: Block Diffusion for Flash Speculative Decoding"
(Paper vs code, "Sampling rule": speculative rejection sampling with residual
resampling above temperature 0).  At one position with proposal law q and
target law p, a proposal y ~ q is accepted with probability min(1, p(y)/q(y))
(eq. 6); on rejection the emitted token is drawn from the residual
r = [p - q]_+ / Z, Z = sum_z [p(z) - q(z)]_+ (eq. 7), so that the emitted
token has law p (eq. 8).

Readings where the pages leave the step open:
- laws: q_j = softmax(draft logits of block row j / T) for the mask rows
  j = 1..B-1; p_j = softmax(verify logits of block row j / T), the target's
  law for the token after block row j (so proposal j, block row j + 1, is
  accepted or rejected under p_j);
- top-k / top-p ("Paper vs code", "Sampling rule": they apply to both the
  draft and the target distributions): one setting (k, p) filters every law
  q_j and p_j after the temperature.  Tokens are ranked by probability,
  highest first, equal probabilities (equal logits) in increasing token id;
  top-k keeps the first min(k, V) of them (k = 0: all); top-p then keeps,
  under the top-k law renormalised, each token whose mass ranked strictly
  before it is below p (the smallest ranked prefix whose mass reaches p;
  p = 1: all); the kept tokens' probabilities are renormalised.  Eq. 6-8
  then hold for the filtered laws, so the emitted token has the filtered
  target law;
- every draw is an inverse-CDF lookup with a caller-supplied uniform
  u in [0, 1): the lowest index z whose cumulative weight exceeds u times the
  total weight (the method's random numbers are inputs, so both sides of a
  comparison use the same ones);
- per round the caller supplies B-1 draft uniforms (one per mask row),
  B-1 acceptance uniforms (proposal j is accepted while u_acc[j] < p/q) and
  one emission uniform (residual at the first rejection, else the bonus
  token from p_{B-1});
- Z = 0 at a rejection (possible only through rounding) draws from p;
- the prompt's first token stays the target's argmax (prefill is outside the
  sampled round).
"""
from __future__ import annotations

import numpy as np

from .model import Model, argmax_lowest
from .spec import Round, SeqState


def softmax_t(logits: np.ndarray, T: float) -> np.ndarray:
    """softmax(logits / T) along the last axis, in fp64."""
    z = np.asarray(logits, dtype=np.float64) / T
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def rank_order(logits: np.ndarray) -> np.ndarray:
    """Token ids by decreasing logit (= decreasing probability at any T > 0),
    equal logits in increasing id."""
    l = np.asarray(logits, dtype=np.float64)
    return np.lexsort((np.arange(l.shape[-1]), -l))


def filter_law(logits: np.ndarray, T: float, top_k: int = 0, top_p: float = 1.0) -> np.ndarray:
    """softmax(logits / T) of one row, restricted to its top-k tokens, then to
    the top-p prefix of that renormalised law, and renormalised."""
    pi = softmax_t(logits, T)
    V = pi.shape[-1]
    order = rank_order(logits)
    kept = order[: top_k] if 0 < top_k < V else order
    if top_p < 1.0:
        w = pi[kept] / pi[kept].sum()
        before = np.cumsum(w) - w                     # mass ranked strictly before each token
        kept = kept[before < top_p]
    out = np.zeros(V)
    out[kept] = pi[kept]
    return out / out.sum()


def filter_laws(logits: np.ndarray, T: float, top_k: int = 0, top_p: float = 1.0) -> np.ndarray:
    """filter_law of every row of a [rows, V] array."""
    lg = np.atleast_2d(logits)
    return np.stack([filter_law(r, T, top_k, top_p) for r in lg])


def sample_inverse_cdf(weights: np.ndarray, u: float) -> int:
    """Lowest index z with cumsum(weights)[z] > u * sum(weights)."""
    c = np.cumsum(np.asarray(weights, dtype=np.float64))
    z = int(np.searchsorted(c, u * c[-1], side="right"))
    return min(z, len(c) - 1)


def accept_probability(p_y: float, q_y: float) -> float:
    """eq. 6: min(1, p(y) / q(y))."""
    return 1.0 if q_y <= 0.0 else min(1.0, p_y / q_y)


def residual(p: np.ndarray, q: np.ndarray):
    """eq. 7: unnormalised residual [p - q]_+ and its mass Z."""
    r = np.maximum(np.asarray(p, np.float64) - np.asarray(q, np.float64), 0.0)
    return r, float(r.sum())


def speculative_step(p: np.ndarray, q: np.ndarray, u_draft: float, u_acc: float, u_emit: float):
    """One position: draw y ~ q, accept it with eq. 6, else draw from eq. 7.

    Returns (token, accepted)."""
    y = sample_inverse_cdf(q, u_draft)
    if u_acc < accept_probability(p[y], q[y]):
        return y, True
    r, Z = residual(p, q)
    return (sample_inverse_cdf(r, u_emit) if Z > 0.0 else sample_inverse_cdf(p, u_emit)), False


def draft_sampled(model: Model, st: SeqState, T: float, u_draft: np.ndarray, top_k: int = 0,
                  top_p: float = 1.0):
    """Algorithm 1 steps 2-3: the drafter's laws q_1..q_{B-1} (filtered by
    top-k / top-p) and the proposals drawn from them.
    Returns (proposals [B-1], q [B-1, V], draft logits [B, V])."""
    lg = model.draft_forward(st.anchor, st.dcache)
    q = filter_laws(lg[1:], T, top_k, top_p) if lg.shape[0] > 1 else softmax_t(lg[1:], T)
    y = np.array([sample_inverse_cdf(q[j], float(u_draft[j])) for j in range(q.shape[0])], dtype=np.int64)
    return y, q, lg


def verify_sampled(model: Model, st: SeqState, proposal, q: np.ndarray, T: float, u_acc: np.ndarray,
                   u_emit: float, keep_logits: bool = False, top_k: int = 0, top_p: float = 1.0) -> Round:
    """Algorithm 1 steps 4-10 with eq. 6-8: scan proposals left to right under
    the surviving prefix; at the first rejection emit a residual draw, else the
    bonus draw from p_{B-1}.  The target laws p_j are filtered by top-k /
    top-p like the drafter's.  Caches keep the anchor and accepted rows."""
    c = model.cfg
    n0 = st.committed
    proposal = np.asarray(proposal, dtype=np.int64)
    assert proposal.shape == (c.block_size - 1,)
    block = np.concatenate([[st.anchor], proposal])
    lg, sel = model.target_forward(block, st.tcache)
    p = filter_laws(lg, T, top_k, top_p)
    a = 0
    for j in range(c.block_size - 1):
        y = int(proposal[j])
        if u_acc[j] < accept_probability(p[j][y], q[j][y]):
            a += 1
        else:
            break
    if a < c.block_size - 1:
        r, Z = residual(p[a], q[a])
        emit = sample_inverse_cdf(r, u_emit) if Z > 0.0 else sample_inverse_cdf(p[a], u_emit)
    else:
        emit = sample_inverse_cdf(p[a], u_emit)
    st.tcache.truncate(n0 + a + 1)
    model.append_context(model.fuse(sel[: a + 1]), st.dcache)
    rd = Round(n_before=n0, anchor=st.anchor, drafts=proposal, proposal=proposal, posterior=argmax_lowest(lg),
               accepted=a, bonus=int(emit), verify_logits=lg if keep_logits else None)
    st.generated += [int(t) for t in proposal[:a]] + [int(emit)]
    st.anchor = int(emit)
    st.rounds.append(rd)
    return rd
