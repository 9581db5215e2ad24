"""CPU oracle for the greedy DFlash draft-and-verify round.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import, call or execute
anything in this package.  The CUDA library never does, and nothing here
imports the library: the two share only the seeded inputs from ``synth``.

Contents
--------
model    fp64 target decoder, context fusion, KV injection, block drafter.
spec     prefill / draft / verify / accept loop, plain AR greedy decode,
         planted proposals that fix the number of accepted drafts.
metrics  acceptance length, cycle latency, speedup, memory accounting,
         context-layer selection.
sampling rounds at temperature T > 0: draft laws (optionally filtered by
         top-k / top-p, the same setting for both laws), proposals drawn by
         inverse CDF from caller-supplied uniforms, acceptance min(1, p/q),
         residual resampling, bonus draw.
training the drafter's training forward (loss value): features of the clean
         sequence, anchor blocks with their legal context, the packed
         block-sparse pass, position-weighted cross-entropy (eq. 12).

Pins (checked by ``tests/test_oracle_*.py`` against the pages and the
mathematics, not against this code):

* speculative greedy output == plain AR greedy output (losslessness),
  for several block sizes, batch shapes and proposers, including block 1,
  and with the block size changed between rounds (``spec.at_block_size``:
  planted proposals accept exactly min(tau, B') - 1 drafts);
* the drafter's incremental context cache == a from-scratch recomputation of
  every context feature and key/value from the committed sequence;
* the verify pass with cache rollback == a fresh causal forward of the
  committed sequence;
* brute-force attention (scalar loops) for the causal and the bidirectional
  masks; closed forms of RMSNorm, RoPE and SiLU;
* acceptance against its characterisation, exhaustively on tiny inputs;
  planted proposals accept exactly the planted count;
* printed worked values of the review's eq. 3, eq. 4/5 and eq. 11 and the
  context-layer lists of the workloads;
* sampling: the inverse-CDF draw's law by exact quadrature, eq. 6 acceptance
  frequencies, eq. 7's two forms of the residual mass and the review's worked
  totals, eq. 8 (the emitted token has the target's law) by seeded Monte
  Carlo, which also rejects resampling from the target on rejection, and the
  T -> 0 limit equal to the greedy round;
* top-k / top-p: closed forms on hand-made laws (temperature first, top-p on
  the renormalised top-k law, the strict "mass before < p" rule, ties in
  increasing id), the kept sets by brute force over subsets, a filtered
  residual known in closed form, top-k = 1 equal to the greedy round, and the
  whole round emitting the filtered target law (seeded Monte Carlo);
* training: the packed block-sparse pass equals one pass per anchor, a block
  equals the inference draft pass with the same context and anchor token, no
  block sees a token at or after its anchor (or another block), the review's
  lambda table and final weight, and the closed-form loss of a uniform drafter;
* the drafter's block pass, by hand-made drafters with closed-form outputs:
  the drafts are the shared head's argmax on the B-1 mask rows (the anchor
  row dropped, rows embedded with the target's table); the block's queries
  are RMS-normalised per head (scaling W_q changes nothing); the block sits
  at positions n .. n+B-1 right after the n context entries (each row picks
  the context key whose RoPE angle matches its own position).

What no pin can fix here is what a trained drafter proposes (its acceptance
length): no trained weights exist, so only the structure and arithmetic of
the drafter's pass are pinned, not its quality.
"""
from . import metrics, model, sampling, spec, training  # noqa: F401
