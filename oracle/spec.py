"""The greedy draft-and-verify loop, step by step, and plain AR greedy decoding.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

The loop follows the greedy decoding round given in "DFlash: Block Diffusion
for Flash Speculative Decoding" (Method, the greedy dflash_decode pseudocode
and the draft-layer pseudocode) and the verification rule of "DFlash: Why a
Diffusion Drafter Can Accelerate an Autoregressive Model" (§4.1 and
Algorithm 1):

1. prefill the prompt; the target's argmax on the last row is the first
   token and the first anchor; the prompt's selected-layer states become the
   context;
2. draft: one parallel pass over [anchor, MASK x (B-1)], argmax of the head
   on the mask rows;
3. verify: one causal target pass over [anchor, d_1 .. d_{B-1}];
4. accept the longest prefix of drafts equal to the target's argmax at the
   preceding position, emit it plus the target's token after it (the bonus);
5. keep target cache entries and context features only for the anchor and the
   accepted drafts; the bonus becomes the next anchor;
6. stop once max_new_tokens are produced and cut the output to that length.

A round may run with a smaller block than the drafter was trained with
(``at_block_size``): the "DFlash" wiki (Ablations, block size) and the paper
digest's Pitfalls (on §5.5.4 and tab. 8) report that a drafter trained at 16
still drafts at 8, and suggest a smaller block when verification is
compute-bound.  Reading: the same weights, B' rows [anchor, MASK x (B'-1)] at
positions n .. n+B'-1; nothing else changes.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, List, Optional

import numpy as np

from .model import KV, Model, argmax_lowest


def count_leading_matches(drafts, posterior) -> int:
    """Number of leading positions j with drafts[j] == posterior[j]."""
    a = 0
    for d, p in zip(drafts, posterior):
        if int(d) != int(p):
            break
        a += 1
    return a


def top2_margin(logits: np.ndarray) -> np.ndarray:
    """Gap between the largest and second-largest logit of each row."""
    part = np.partition(logits, -2, axis=-1)
    return part[..., -1] - part[..., -2]


@dataclass
class Round:
    n_before: int                 # committed length (target KV = draft context) at round start
    anchor: int
    drafts: np.ndarray            # the drafter's own B-1 proposals
    proposal: np.ndarray          # what was verified (== drafts unless a proposer overrides)
    posterior: np.ndarray         # target argmax at the B block positions
    accepted: int
    bonus: int
    draft_logits: Optional[np.ndarray] = None     # [B, V]
    verify_logits: Optional[np.ndarray] = None    # [B, V]


@dataclass
class SeqState:
    prompt: np.ndarray
    tcache: KV
    dcache: KV
    anchor: int
    generated: List[int] = field(default_factory=list)
    first_logits: Optional[np.ndarray] = None
    prefill_sel: Optional[np.ndarray] = None
    rounds: List[Round] = field(default_factory=list)

    @property
    def committed(self) -> int:
        return self.tcache.length


def prefill(model: Model, prompt) -> SeqState:
    prompt = np.asarray(prompt, dtype=np.int64)
    tc, dc = model.new_target_cache(), model.new_draft_cache()
    lg, sel = model.target_forward(prompt, tc)
    first = int(argmax_lowest(lg[-1:])[0])
    model.append_context(model.fuse(sel), dc)
    st = SeqState(prompt=prompt, tcache=tc, dcache=dc, anchor=first, generated=[first])
    st.first_logits = lg[-1]
    st.prefill_sel = sel
    return st


def at_block_size(model: Model, B: int) -> Model:
    """The same target and drafter with an inference block of B rows, 1 <= B <=
    the configured (training) block size; the weights are shared, not copied."""
    if not 1 <= B <= model.cfg.block_size:
        raise ValueError(f"block size {B} outside [1, {model.cfg.block_size}]")
    return Model(model.cfg.with_(block_size=B), weights=model.w, act_round=model.act_round)


def draft(model: Model, st: SeqState):
    """Returns (drafts [B-1], logits [B, V])."""
    lg = model.draft_forward(st.anchor, st.dcache)
    return argmax_lowest(lg[1:]), lg


def verify(model: Model, st: SeqState, proposal, drafts=None, draft_logits=None, keep_logits=False) -> Round:
    c = model.cfg
    n0 = st.committed
    proposal = np.asarray(proposal, dtype=np.int64)
    assert proposal.shape == (c.block_size - 1,)
    block = np.concatenate([[st.anchor], proposal])
    lg, sel = model.target_forward(block, st.tcache)
    post = argmax_lowest(lg)
    a = count_leading_matches(proposal, post[:-1])
    bonus = int(post[a])
    st.tcache.truncate(n0 + a + 1)
    model.append_context(model.fuse(sel[: a + 1]), st.dcache)
    rd = Round(n_before=n0, anchor=st.anchor, drafts=proposal if drafts is None else drafts,
               proposal=proposal, posterior=post, accepted=a, bonus=bonus,
               draft_logits=draft_logits if keep_logits else None, verify_logits=lg if keep_logits else None)
    st.generated += [int(t) for t in proposal[:a]] + [bonus]
    st.anchor = bonus
    st.rounds.append(rd)
    return rd


Proposer = Callable[[SeqState, np.ndarray], np.ndarray]


def generate(model: Model, prompt, max_new_tokens: int, proposer: Optional[Proposer] = None,
             keep_logits: bool = False, max_rounds: Optional[int] = None,
             block_schedule: Optional[List[int]] = None) -> SeqState:
    """Speculative greedy decoding of one sequence.  ``proposer(state, drafts)``
    may replace the drafter's tokens by any proposal of length B-1.
    ``block_schedule``: block size of round r = block_schedule[r % len], each
    at most the configured one (default: the configured block every round)."""
    st = prefill(model, prompt)
    while len(st.generated) < max_new_tokens:
        if max_rounds is not None and len(st.rounds) >= max_rounds:
            break
        m = model
        if block_schedule:
            m = at_block_size(model, int(block_schedule[len(st.rounds) % len(block_schedule)]))
        d, dl = draft(m, st)
        prop = d if proposer is None else np.asarray(proposer(st, d), dtype=np.int64)
        verify(m, st, prop, drafts=d, draft_logits=dl, keep_logits=keep_logits)
    st.generated = st.generated[:max_new_tokens]
    return st


def ar_generate(model: Model, prompt, max_new_tokens: int, keep_logits: bool = False):
    """Plain greedy decoding: t_0 = argmax f(prompt), t_j = argmax f(prompt, t_<j).

    Returns (tokens, logits per step or None)."""
    prompt = np.asarray(prompt, dtype=np.int64)
    tc = model.new_target_cache()
    lg, _ = model.target_forward(prompt, tc)
    out = [int(argmax_lowest(lg[-1:])[0])]
    logs = [lg[-1]] if keep_logits else None
    while len(out) < max_new_tokens:
        lg, _ = model.target_forward([out[-1]], tc)
        out.append(int(argmax_lowest(lg)[0]))
        if keep_logits:
            logs.append(lg[0])
    return np.array(out[:max_new_tokens], dtype=np.int64), (np.stack(logs) if keep_logits else None)


def planted_proposer(stream: np.ndarray, tau_seq, vocab: int) -> Proposer:
    """Proposals built from a known greedy stream so that the round accepts a
    chosen number of drafts: the next (tau-1) true tokens, then a wrong one.

    ``stream`` is the target's greedy continuation (first token first);
    ``tau_seq`` gives the intended tokens per round (accepted + 1), cycled."""
    taus = list(tau_seq)

    def prop(st: SeqState, drafts: np.ndarray) -> np.ndarray:
        B1 = drafts.shape[0]
        g = len(st.generated)             # stream[g] is the token after the anchor
        t = taus[len(st.rounds) % len(taus)]
        a = max(0, min(int(t) - 1, B1))
        out = np.empty(B1, dtype=np.int64)
        for j in range(B1):
            idx = g + j
            true = int(stream[idx]) if idx < len(stream) else 0
            out[j] = true if j < a else (true + 1) % vocab
        return out

    return prop
