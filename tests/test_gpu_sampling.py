"""GPU rounds at temperature T > 0 (speculative rejection sampling) through the
C ABI against the fp64 oracle ("DFlash: Why a Diffusion Drafter Can
Accelerate an Autoregressive Model" §4.2 eq. 6-8, Algorithm 1).

Both sides receive the same uniforms.  fp32 workloads: logits within 1e-3,
and every draw (proposal, residual, bonus) and every acceptance decision
equal to the oracle's unless the oracle's fp64 value lies within 1e-4 of the
decision boundary (then the two streams may part, and the sequence stops being
compared).  The GPU's proposals are what both sides verify, as in any verify.
bf16: at T -> 0 the sampled round is the greedy round.

With a top-k / top-p filter ("DFlash: Block Diffusion for Flash Speculative
Decoding", Paper vs code "Sampling rule": both laws are filtered) the same
comparison runs on the filtered laws.  Where the GPU's logit error could move
a filter cut (tokens within twice that error of the top-k cut, or whose
preceding mass lies within the implied mass error of p), a differing decision
is allowed if it involves such a token or lies within the boundary margin
widened by their mass; it ends the comparison of its sequence.  Vocabularies of 40000 and 70001 tokens
split each row over a cluster of 5 and 8 CTAs (the latter with a ragged last
chunk and rows that are not 16-byte aligned)."""
import numpy as np
import pytest

import synth
from synth import configs
from oracle import model as om, sampling as sp, spec

pytestmark = pytest.mark.gpu

LOGIT_TOL = 1e-3
EDGE = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_speculative_ctx_gb300 import build
    build.build()


def _draw_margin(weights, u):
    """Distance of u * total from the boundaries of the bin it falls in, relative to the total."""
    c = np.cumsum(np.asarray(weights, np.float64))
    c = c / c[-1]
    z = min(int(np.searchsorted(c, u, side="right")), len(c) - 1)
    lo = c[z - 1] if z > 0 else 0.0
    return min(u - lo, c[z] - u)


def _uncertain(l, dl, T, top_k, top_p):
    """Tokens whose place inside or outside the oracle's filtered law of logit row l a
    logit error dl could change, and their share of that law's mass (with the
    mass of the token the cut would move in)."""
    l = np.asarray(l, np.float64)
    V = l.shape[-1]
    order = sp.rank_order(l)
    eps = 2.0 * dl + 1e-6
    unsure = np.zeros(V, bool)
    kept = order
    if 0 < top_k < V:
        cut = 0.5 * (l[order[top_k - 1]] + l[order[top_k]])
        unsure |= np.abs(l - cut) < eps
        kept = order[:top_k]
    if top_p < 1.0:
        pi = sp.softmax_t(l[kept], T)
        before = np.cumsum(pi) - pi
        unsure[kept[np.abs(before - top_p) < 4.0 * eps / T + 1e-6]] = True
    pi_all = sp.softmax_t(l, T)
    law = sp.filter_law(l, T, top_k, top_p)
    mass = pi_all[unsure].sum() / pi_all[law > 0].sum()
    return unsure, mass


def run_sampled(name, T, rounds, seed=0, top_k=0, top_p=1.0, **wkw):
    from block_diffusion_speculative_ctx_gb300 import Session
    w = configs.get(name)
    if wkw:
        w = w.with_(**wkw)
    filtered = top_k > 0 or top_p < 1.0
    B, B1 = w.block_size, w.block_size - 1
    m = om.Model(w)
    prompts = synth.prompts(w)
    states = [spec.prefill(m, p) for p in prompts]
    b = len(states)
    alive = [True] * b
    rng = np.random.default_rng(1000 + seed)
    compared = 0
    sess = Session(w, keep_logits=True, max_seq_len=max(w.prompt_lens) + (rounds + 2) * B + 8)
    try:
        if filtered:
            sess.set_sampling_filter(top_k, top_p)
        first = sess.prefill(prompts)
        for s, st in enumerate(states):
            assert int(first[s]) == st.anchor
        for r in range(rounds):
            ud = rng.random((b, max(B1, 1))).astype(np.float32)
            uv = rng.random((b, B)).astype(np.float32)
            drafts = sess.draft_block_sampled(T, ud)
            dlog = sess.logits("draft")
            laws = []
            for s, st in enumerate(states):
                if not alive[s]:
                    laws.append(None)
                    continue
                y, q, odl = sp.draft_sampled(m, st, T, ud[s, :B1].astype(np.float64), top_k=top_k, top_p=top_p)
                if B1 > 0:   # (block size 1 runs no draft head)
                    assert np.abs(dlog[s] - odl).max() <= LOGIT_TOL, f"round {r} seq {s} draft logits"
                unsure = [_uncertain(odl[j + 1], np.abs(dlog[s][j + 1] - odl[j + 1]).max(), T, top_k, top_p)
                          if filtered else (np.zeros(w.vocab, bool), 0.0) for j in range(B1)]
                for j in range(B1):     # (both sides verify the GPU's proposals: a differing draw ends nothing)
                    if int(drafts[s, j]) != int(y[j]) and not (unsure[j][0][int(drafts[s, j])] or
                                                              unsure[j][0][int(y[j])]):
                        assert _draw_margin(q[j], float(ud[s, j])) < EDGE + unsure[j][1], f"round {r} seq {s} draw {j}"
                laws.append((q, unsure))
            acc, emit = sess.verify_sampled(T, drafts, uv)
            vlog = sess.logits("verify")
            lens = sess.lengths()
            for s, st in enumerate(states):
                if not alive[s]:
                    continue
                q, unsure_q = laws[s]
                rd = sp.verify_sampled(m, st, drafts[s, :B1].astype(np.int64), q, T, uv[s, :B1].astype(np.float64),
                                       float(uv[s, B1]), keep_logits=True, top_k=top_k, top_p=top_p)
                assert np.abs(vlog[s] - rd.verify_logits).max() <= LOGIT_TOL, f"round {r} seq {s} verify logits"
                unsure_p = [_uncertain(rd.verify_logits[j], np.abs(vlog[s][j] - rd.verify_logits[j]).max(), T, top_k,
                                       top_p) if filtered else (np.zeros(w.vocab, bool), 0.0) for j in range(B)]
                p = sp.filter_laws(rd.verify_logits, T, top_k, top_p)
                a_o, a_g = rd.accepted, int(acc[s])
                if a_g != a_o:
                    j = min(a_g, a_o)                       # the first decision taken differently
                    y = int(drafts[s, j])
                    if not (unsure_p[j][0][y] or unsure_q[j][0][y]):
                        ratio = sp.accept_probability(p[j][y], q[j][y])
                        tol = EDGE + 2 * (unsure_p[j][1] + unsure_q[j][1])
                        assert abs(float(uv[s, j]) - ratio) < tol, f"round {r} seq {s}: accepted {a_g} vs {a_o}"
                    alive[s] = False
                    continue
                if int(emit[s]) != rd.bonus:
                    e, o = int(emit[s]), rd.bonus
                    near_cut = unsure_p[a_o][0][e] or unsure_p[a_o][0][o] or (
                        a_o < B1 and (unsure_q[a_o][0][e] or unsure_q[a_o][0][o]))
                    if not near_cut:
                        if a_o < B1:
                            wts, Z = sp.residual(p[a_o], q[a_o])
                            wts = wts if Z > 0 else p[a_o]
                            tol = EDGE + 2 * (unsure_p[a_o][1] + unsure_q[a_o][1])
                        else:
                            wts = p[a_o]
                            tol = EDGE + 2 * unsure_p[a_o][1]
                        assert _draw_margin(wts, float(uv[s, B1])) < tol, f"round {r} seq {s}: emitted"
                    alive[s] = False
                    continue
                assert lens[s] == st.committed
                compared += 1
        return compared
    finally:
        sess.close()


@pytest.mark.parametrize("T", [0.7, 1.0, 1.6])
def test_tiny_f32_sampled_rounds(T):
    assert run_sampled("tiny_f32", T, rounds=8) >= 6


def test_tiny_f32_ragged_batch_sampled():
    assert run_sampled("tiny_f32_b3", 1.0, rounds=6, seed=3) >= 15      # of 3 x 6


def test_small_f32_hd128_block16_sampled():
    assert run_sampled("small_f32", 1.0, rounds=4, seed=5) >= 6         # of 2 x 4


def test_block_size_one_sampling_is_plain_sampling():
    # B = 1: no proposals; every round emits one draw from the target's law
    assert run_sampled("tiny_f32_b3", 0.9, rounds=5, seed=7, block_size=1) >= 12


@pytest.mark.parametrize("T,top_k,top_p", [(1.0, 5, 1.0), (0.8, 0, 0.9), (1.3, 20, 0.7)])
def test_tiny_f32_filtered_sampled_rounds(T, top_k, top_p):
    assert run_sampled("tiny_f32", T, rounds=8, seed=11, top_k=top_k, top_p=top_p) >= 6


def test_tiny_f32_ragged_batch_filtered():
    assert run_sampled("tiny_f32_b3", 1.1, rounds=5, seed=13, top_k=40, top_p=0.8) >= 10     # of 3 x 5


@pytest.mark.parametrize("vocab,top_k,top_p", [(40000, 50, 0.9), (70001, 0, 0.95), (70001, 300, 1.0)])
def test_large_vocab_filtered_sampled_rounds(vocab, top_k, top_p):
    """Rows split over 5 and 8 CTAs (ragged last chunk, rows not 16-byte aligned
    at 70001); top-p alone keeps tens of thousands of tokens here."""
    assert run_sampled("tiny_f32", 1.0, rounds=4, seed=17, top_k=top_k, top_p=top_p, vocab=vocab) >= 3


def test_top_k_one_sampled_round_is_the_greedy_round():
    """top-k = 1: every law is one-hot at the lowest-index argmax, so at any T and
    for any uniforms the sampled round makes the greedy round's choices, exactly
    (fp32, no near-ties in this workload)."""
    from block_diffusion_speculative_ctx_gb300 import Session
    w = configs.get("tiny_f32_b3")
    prompts = synth.prompts(w)
    b, B = len(prompts), w.block_size
    rng = np.random.default_rng(23)
    with Session(w, max_seq_len=max(w.prompt_lens) + 8 * B) as sg, Session(w, max_seq_len=max(w.prompt_lens) + 8 * B) as ss:
        ss.set_sampling_filter(1, 1.0)
        assert np.array_equal(sg.prefill(prompts), ss.prefill(prompts))
        for _ in range(5):
            d = sg.draft_block()
            acc, bonus = sg.verify(d)
            ds = ss.draft_block_sampled(1.5, rng.random((b, B - 1)).astype(np.float32))
            assert np.array_equal(ds, d)
            acc_s, emit = ss.verify_sampled(1.5, ds, rng.random((b, B)).astype(np.float32))
            assert np.array_equal(acc_s, acc) and np.array_equal(emit, bonus)
        assert np.array_equal(ss.lengths(), sg.lengths())


def test_sampled_round_at_small_temperature_is_the_greedy_round_bf16():
    """T -> 0: the laws are one-hot at the argmax, so proposals, acceptance and
    the emitted token are the greedy round's (checked against the oracle's
    greedy round; positions whose top-2 margin is below the bf16 tolerance are
    excluded)."""
    from block_diffusion_speculative_ctx_gb300 import Session
    w = configs.get("small_bf16")
    m = om.Model(w)
    prompts = synth.prompts(w)
    states = [spec.prefill(m, p) for p in prompts]
    b, B = len(states), w.block_size
    rng = np.random.default_rng(11)
    with Session(w, keep_logits=True, max_seq_len=max(w.prompt_lens) + 8 * B) as sess:
        sess.prefill(prompts)
        alive = [True] * b
        for r in range(3):
            drafts = sess.draft_block_sampled(1e-4, rng.random((b, B - 1)).astype(np.float32))
            acc, emit = sess.verify_sampled(1e-4, drafts, rng.random((b, B)).astype(np.float32))
            for s, st in enumerate(states):
                if not alive[s]:
                    continue
                d, dl = spec.draft(m, st)
                if spec.top2_margin(dl[1:]).min() < 5e-2:
                    alive[s] = False
                    continue
                assert np.array_equal(drafts[s], d)
                rd = spec.verify(m, st, d, keep_logits=True)
                if spec.top2_margin(rd.verify_logits).min() < 5e-2:
                    alive[s] = False
                    continue
                assert (int(acc[s]), int(emit[s])) == (rd.accepted, rd.bonus)


def test_sampling_errors():
    from block_diffusion_speculative_ctx_gb300 import Session, DFlashError
    w = configs.get("tiny_f32")
    with Session(w, max_seq_len=256) as sess:
        sess.prefill(synth.prompts(w))
        B = w.block_size
        u = np.full((1, B - 1), 0.5, np.float32)
        with pytest.raises(DFlashError, match="temperature"):
            sess.draft_block_sampled(0.0, u)
        with pytest.raises(DFlashError, match="uniform"):
            sess.draft_block_sampled(1.0, np.full((1, B - 1), 1.0, np.float32))
        with pytest.raises(DFlashError, match="top_p"):
            sess.set_sampling_filter(0, 0.0)
        with pytest.raises(DFlashError, match="top_k"):
            sess.set_sampling_filter(-1, 1.0)
        sess.set_sampling_filter(3, 0.5)
        d = sess.draft_block_sampled(1.0, u)
        with pytest.raises(DFlashError, match="between a draft and its verify"):
            sess.set_sampling_filter(0, 1.0)
        sess.verify_sampled(1.0, d, np.full((1, B), 0.5, np.float32))
        sess.set_sampling_filter(0, 1.0)
        d = sess.draft_block()                          # a greedy draft keeps no laws
        with pytest.raises(DFlashError, match="draft_block_sampled"):
            sess.verify_sampled(1.0, d, np.full((1, B), 0.5, np.float32))
        sess.verify(d)                                  # the greedy verify still works
        d = sess.draft_block_sampled(1.0, u)
        acc, emit = sess.verify_sampled(1.0, d, np.full((1, B), 0.5, np.float32))
        assert 0 <= acc[0] <= B - 1 and 0 <= emit[0] < w.vocab
