"""GPU rounds at temperature T > 0 (speculative rejection sampling) through the
C ABI against the fp64 oracle ("DFlash: Why a Diffusion Drafter Can
Accelerate an Autoregressive Model" §4.2 eq. 6-8, Algorithm 1).

Both sides receive the same uniforms.  fp32 workloads: logits within 1e-3,
and every draw (proposal, residual, bonus) and every acceptance decision
equal to the oracle's unless the oracle's fp64 value lies within 1e-4 of the
decision boundary (then the two streams may part, and the sequence stops being
compared).  The GPU's proposals are what both sides verify, as in any verify.
bf16: at T -> 0 the sampled round is the greedy round."""
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


def run_sampled(name, T, rounds, seed=0, **wkw):
    from block_diffusion_speculative_ctx_gb300 import Session
    w = configs.get(name)
    if wkw:
        w = w.with_(**wkw)
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
                y, q, odl = sp.draft_sampled(m, st, T, ud[s, :B1].astype(np.float64))
                if B1 > 0:   # (block size 1 runs no draft head)
                    assert np.abs(dlog[s] - odl).max() <= LOGIT_TOL, f"round {r} seq {s} draft logits"
                for j in range(B1):
                    if int(drafts[s, j]) != int(y[j]):
                        assert _draw_margin(q[j], float(ud[s, j])) < EDGE, f"round {r} seq {s} draw {j}"
                laws.append(q)
            acc, emit = sess.verify_sampled(T, drafts, uv)
            vlog = sess.logits("verify")
            lens = sess.lengths()
            for s, st in enumerate(states):
                if not alive[s]:
                    continue
                q = laws[s]
                rd = sp.verify_sampled(m, st, drafts[s, :B1].astype(np.int64), q, T, uv[s, :B1].astype(np.float64),
                                       float(uv[s, B1]), keep_logits=True)
                assert np.abs(vlog[s] - rd.verify_logits).max() <= LOGIT_TOL, f"round {r} seq {s} verify logits"
                p = sp.softmax_t(rd.verify_logits, T)
                a_o, a_g = rd.accepted, int(acc[s])
                if a_g != a_o:
                    j = min(a_g, a_o)                       # the first decision taken differently
                    y = int(drafts[s, j])
                    ratio = sp.accept_probability(p[j][y], q[j][y])
                    assert abs(float(uv[s, j]) - ratio) < EDGE, f"round {r} seq {s}: accepted {a_g} vs {a_o}"
                    alive[s] = False
                    continue
                if int(emit[s]) != rd.bonus:
                    if a_o < B1:
                        wts, Z = sp.residual(p[a_o], q[a_o])
                        wts = wts if Z > 0 else p[a_o]
                    else:
                        wts = p[a_o]
                    assert _draw_margin(wts, float(uv[s, B1])) < EDGE, f"round {r} seq {s}: emitted"
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
        d = sess.draft_block()                          # a greedy draft keeps no laws
        with pytest.raises(DFlashError, match="draft_block_sampled"):
            sess.verify_sampled(1.0, d, np.full((1, B), 0.5, np.float32))
        sess.verify(d)                                  # the greedy verify still works
        d = sess.draft_block_sampled(1.0, u)
        acc, emit = sess.verify_sampled(1.0, d, np.full((1, B), 0.5, np.float32))
        assert 0 <= acc[0] <= B - 1 and 0 <= emit[0] < w.vocab
