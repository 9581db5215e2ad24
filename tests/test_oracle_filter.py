"""Pins of the oracle's top-k / top-p filter of the sampled round ("DFlash:
Block Diffusion for Flash Speculative Decoding", Paper vs code "Sampling
rule": top-p and top-k apply to both the draft and the target distributions;
"DFlash: Why a Diffusion Drafter Can Accelerate an Autoregressive Model" §4.2
eq. 6-8 on the filtered laws).

Closed forms on hand-made laws fix the order of the steps (temperature, then
top-k, then top-p on the renormalised top-k law), the strict "mass before <
p" rule and the tie order; a brute force over subsets fixes the kept sets
independently of the ranking code; top-k = 1 reduces the sampled round to the
greedy round; a seeded Monte Carlo checks that the whole round emits the
filtered target law.  Each pin is also run against planted mistakes."""
import copy
import itertools

import numpy as np
import pytest

import synth
from synth import configs
from oracle import model as om, sampling as sp, spec


def _lg(probs):
    return np.log(np.asarray(probs, np.float64))


# ------------------------------------------------------------------ pins, parameterised by the filter under test
def _pin_closed_forms(f):
    l = _lg([0.1, 0.4, 0.2, 0.3])
    # top-p 0.65: ranked 1 (0.4), 3 (0.3), 2 (0.2), 0 (0.1); masses before 0, 0.4, 0.7 -> {1, 3}
    np.testing.assert_allclose(f(l, 1.0, 0, 0.65), [0, 4 / 7, 0, 3 / 7], atol=1e-12)
    np.testing.assert_allclose(f(l, 1.0, 2, 1.0), [0, 4 / 7, 0, 3 / 7], atol=1e-12)
    # top-p on the renormalised top-3 law: masses before 0, 0.4/0.9 = 0.444 >= 0.42 -> {1} only,
    # while top-p 0.42 on the whole law keeps {1, 3} (0.4 < 0.42)
    np.testing.assert_allclose(f(l, 1.0, 3, 0.42), [0, 1, 0, 0], atol=1e-12)
    np.testing.assert_allclose(f(l, 1.0, 0, 0.42), [0, 4 / 7, 0, 3 / 7], atol=1e-12)
    # switched off: k = 0, k >= V, p = 1
    for k in (0, 4, 9):
        np.testing.assert_allclose(f(l, 1.0, k, 1.0), [0.1, 0.4, 0.2, 0.3], atol=1e-12)
    # a tiny p keeps the most probable token only
    np.testing.assert_allclose(f(l, 1.0, 0, 1e-9), [0, 1, 0, 0], atol=1e-12)


def _pin_temperature_first(f):
    l = _lg([0.4, 0.3, 0.2, 0.1])
    # T = 1: masses before 0, 0.4, 0.7 -> {0, 1}; T = 2 flattens the law (proportional to
    # sqrt(p)): masses before 0, 0.325, 0.607 < 0.65 -> {0, 1, 2}
    np.testing.assert_allclose(f(l, 1.0, 0, 0.65), [4 / 7, 3 / 7, 0, 0], atol=1e-12)
    r = np.sqrt([0.4, 0.3, 0.2])
    np.testing.assert_allclose(f(l, 2.0, 0, 0.65), np.append(r / r.sum(), 0), atol=1e-12)


def _pin_ties_and_strict_rule(f):
    # equal logits rank in increasing id: top-2 of [1, 3, 3, 3, 0] is {1, 2}
    np.testing.assert_allclose(f(np.array([1.0, 3, 3, 3, 0]), 1.0, 2, 1.0), [0, 0.5, 0.5, 0, 0], atol=1e-12)
    # four equal probabilities: masses before 0, 1/4, 1/2, 3/4 (exact); p = 1/2 keeps a token only
    # while the mass before it is strictly below 1/2 -> {0, 1}
    np.testing.assert_allclose(f(np.zeros(4), 1.0, 0, 0.5), [0.5, 0.5, 0, 0], atol=1e-12)


def _pin_brute_force(f):
    """Kept sets from their definitions, by enumeration: top-k = the k-token set of
    largest mass; top-p = among subsets of it holding at least p of its mass, the
    fewest tokens, and among those the largest mass."""
    rng = np.random.default_rng(17)
    V = 7
    for trial in range(30):
        pi = rng.gamma(0.8, size=V)
        pi /= pi.sum()
        T = float(rng.choice([0.5, 1.0, 1.7]))
        l = np.log(pi) * T                    # softmax(l / T) == pi
        k = int(rng.integers(0, V + 2))
        p = float(rng.choice([1.0, rng.uniform(0.05, 0.99)]))
        K = set(range(V))
        if 0 < k < V:
            K = set(max(itertools.combinations(range(V), k), key=lambda c: pi[list(c)].sum()))
        S = K
        if p < 1.0:
            mk = pi[list(K)].sum()
            ok = [set(c) for r in range(1, len(K) + 1) for c in itertools.combinations(sorted(K), r)
                  if pi[list(c)].sum() >= p * mk]
            n = min(len(c) for c in ok)
            S = max((c for c in ok if len(c) == n), key=lambda c: pi[list(c)].sum())
        want = np.zeros(V)
        want[list(S)] = pi[list(S)]
        np.testing.assert_allclose(f(l, T, k, p), want / want.sum(), atol=1e-12,
                                   err_msg=f"trial {trial} k={k} p={p}")


PINS = (_pin_closed_forms, _pin_temperature_first, _pin_ties_and_strict_rule, _pin_brute_force)


@pytest.mark.parametrize("pin", PINS)
def test_filter_pins(pin):
    pin(sp.filter_law)


# ------------------------------------------------------------------ planted mistakes
def _filter_before_temperature(l, T, k=0, p=1.0):
    keep = sp.filter_law(l, 1.0, k, p) > 0
    out = np.where(keep, sp.softmax_t(l, T), 0.0)
    return out / out.sum()


def _top_p_before_top_k(l, T, k=0, p=1.0):
    a = sp.filter_law(l, T, 0, p) > 0
    b = sp.filter_law(l, T, k, 1.0) > 0
    out = np.where(a & b, sp.softmax_t(l, T), 0.0)
    return out / out.sum()


def _top_p_not_strict(l, T, k=0, p=1.0):
    pi = sp.softmax_t(l, T)
    order = sp.rank_order(l)
    kept = order[:k] if 0 < k < len(pi) else order
    if p < 1.0:
        w = pi[kept] / pi[kept].sum()
        kept = kept[np.cumsum(w) - w <= p]
    out = np.zeros(len(pi))
    out[kept] = pi[kept]
    return out / out.sum()


def _top_k_keeps_ties(l, T, k=0, p=1.0):
    pi = sp.softmax_t(l, T)
    if 0 < k < len(pi):
        kth = np.sort(l)[::-1][k - 1]
        pi = np.where(l >= kth, pi, 0.0)
    return sp.filter_law(np.log(np.maximum(pi, 1e-300)) * T, T, 0, p)


@pytest.mark.parametrize("mutant,pin", [(_filter_before_temperature, _pin_temperature_first),
                                        (_top_p_before_top_k, _pin_closed_forms),
                                        (_top_p_not_strict, _pin_ties_and_strict_rule),
                                        (_top_k_keeps_ties, _pin_ties_and_strict_rule)])
def test_planted_filter_mistakes_are_caught(mutant, pin):
    with pytest.raises(AssertionError):
        pin(mutant)


# ------------------------------------------------------------------ eq. 6-8 on filtered laws
def test_filtered_residual_closed_form():
    """Target law (0.5, 0.3, 0.15, 0.05), drafter law (0.3, 0.5, 0.05, 0.15), top-2:
    p' = (5/8, 3/8, 0, 0), q' = (3/8, 5/8, 0, 0); eq. 6 accepts with total
    probability sum min(p', q') = 3/4, and eq. 7's residual is (1/4, 0, 0, 0): every
    rejection is corrected to token 0.  Unfiltered the same pair accepts 0.7 and
    the residual (0.2, 0, 0.1, 0) also reaches token 2."""
    lp, lq = _lg([0.5, 0.3, 0.15, 0.05]), _lg([0.3, 0.5, 0.05, 0.15])
    p, q = sp.filter_law(lp, 1.0, 2), sp.filter_law(lq, 1.0, 2)
    np.testing.assert_allclose(p, [5 / 8, 3 / 8, 0, 0], atol=1e-12)
    np.testing.assert_allclose(q, [3 / 8, 5 / 8, 0, 0], atol=1e-12)
    assert abs(np.minimum(p, q).sum() - 0.75) < 1e-12
    r, Z = sp.residual(p, q)
    assert abs(Z - 0.25) < 1e-12 and np.flatnonzero(r).tolist() == [0]
    assert abs(sp.accept_probability(p[1], q[1]) - 0.6) < 1e-12
    r0, Z0 = sp.residual(sp.softmax_t(lp, 1.0), sp.softmax_t(lq, 1.0))
    assert abs(Z0 - 0.3) < 1e-12 and np.flatnonzero(r0).tolist() == [0, 2]
    # the emitted token's law by exact enumeration over the drafter's law: p'
    emit = np.zeros(4)
    for y in range(4):
        a = sp.accept_probability(p[y], q[y])
        emit[y] += q[y] * a
        emit += q[y] * (1 - a) * r / Z
    np.testing.assert_allclose(emit, p, atol=1e-12)


def test_top_k_one_sampled_round_is_the_greedy_round():
    """top-k = 1 makes every law one-hot at the lowest-index argmax, at any T and for
    any uniforms: the drafter's proposals are its greedy drafts, each is accepted
    exactly when it is the target's argmax, and the emitted token is the greedy
    bonus (filtering only one of the two laws breaks this)."""
    cfg = configs.get("tiny_f32_b3")
    m = om.Model(cfg)
    rng = np.random.default_rng(9)
    B1 = cfg.block_size - 1
    for prompt in synth.prompts(cfg)[:2]:
        st_g = spec.prefill(m, prompt)
        st_s = copy.deepcopy(st_g)
        for _ in range(4):
            d, _ = spec.draft(m, st_g)
            rg = spec.verify(m, st_g, d)
            y, q, _ = sp.draft_sampled(m, st_s, 1.3, rng.random(B1), top_k=1)
            assert np.array_equal(y, d)
            rs = sp.verify_sampled(m, st_s, y, q, 1.3, rng.random(B1), float(rng.random()), top_k=1)
            assert (rs.accepted, rs.bonus) == (rg.accepted, rg.bonus)
            assert st_s.committed == st_g.committed


def test_round_emits_the_filtered_target_law():
    """Whole round with top-k 5 and top-p 0.8 at T = 3 on a 16-token toy model (both
    filters bind: 4 tokens survive): the first emitted token has the filtered
    target law after the anchor (eq. 8 on the filtered laws)."""
    w = configs.get("tiny_f32").with_(name="toy_filter", vocab=16, d_model=32, n_heads=2, n_kv_heads=1,
                                      head_dim=16, ffn=64, target_layers=2, draft_layers=1, ctx_layer_ids=(0, 1),
                                      block_size=4, prompt_lens=(6,), weight_std=0.5)
    m = om.Model(w)
    T, k, p = 3.0, 5, 0.8
    st0 = spec.prefill(m, synth.prompts(w)[0])
    lg, _ = m.target_forward([st0.anchor], st0.tcache.copy())
    p0 = sp.filter_law(lg[0], T, k, p)
    assert np.count_nonzero(p0) == 4 and np.count_nonzero(sp.filter_law(lg[0], T, k)) == k
    rng = np.random.default_rng(22)
    n = 6000
    counts = np.zeros(w.vocab)
    B1 = w.block_size - 1
    for _ in range(n):
        st = copy.deepcopy(st0)
        y, q, _ = sp.draft_sampled(m, st, T, rng.random(B1), top_k=k, top_p=p)
        rd = sp.verify_sampled(m, st, y, q, T, rng.random(B1), float(rng.random()), top_k=k, top_p=p)
        counts[int(y[0]) if rd.accepted >= 1 else rd.bonus] += 1
    assert counts[p0 == 0].sum() == 0
    assert np.abs(counts / n - p0).max() < 5 * np.sqrt(0.25 / n)


@pytest.mark.parametrize("side", ["draft_sampled", "verify_sampled"])
def test_filtering_one_law_only_is_caught(monkeypatch, side):
    """The filter applies to both laws: dropping it from either one breaks the top-k = 1 pin."""
    orig = getattr(sp, side)
    monkeypatch.setattr(sp, side, lambda *a, top_k=0, top_p=1.0, **kw: orig(*a, **kw))
    with pytest.raises(AssertionError):
        test_top_k_one_sampled_round_is_the_greedy_round()
