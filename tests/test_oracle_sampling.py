"""Pins of the oracle's temperature-sampling round ("DFlash: Why a Diffusion
Drafter Can Accelerate an Autoregressive Model" §4.2 eq. 6-8, Algorithm 1).

The draws are inverse-CDF lookups of caller-supplied uniforms, so their laws
are checked by exact quadrature over a grid of uniforms; the composed
position (eq. 8: the emitted token has the target's law) by a seeded Monte
Carlo with a bound of several standard errors; the T -> 0 limit against the
greedy round."""
import copy
import json
import os

import numpy as np
import pytest

import synth
from synth import configs
from oracle import model as om, sampling as sp, spec

with open(os.path.join(os.path.dirname(__file__), "golden", "pages_values.json")) as _f:
    GOLD = json.load(_f)


def _grid(n):
    return (np.arange(n) + 0.5) / n


def _laws(seed, V=6):
    rng = np.random.default_rng(seed)
    p = rng.gamma(0.7, size=V)
    q = rng.gamma(0.7, size=V)
    return p / p.sum(), q / q.sum()


def test_inverse_cdf_draws_have_the_weights_law():
    w = np.array([0.0, 2.0, 0.5, 0.0, 1.5, 1.0])
    N = 20000
    f = np.bincount([sp.sample_inverse_cdf(w, u) for u in _grid(N)], minlength=len(w)) / N
    np.testing.assert_allclose(f, w / w.sum(), atol=1.0 / N)
    assert f[0] == 0 and f[3] == 0                       # zero weight is never drawn
    assert sp.sample_inverse_cdf(w, 0.0) == 1            # lowest index with positive mass
    assert sp.sample_inverse_cdf(w, 1.0 - 1e-15) == 5


def test_eq6_acceptance_frequency():
    N = 10000
    for p_y, q_y in ((0.2, 0.4), (0.4, 0.2), (0.3, 0.3), (0.0, 0.5)):
        f = np.mean([u < sp.accept_probability(p_y, q_y) for u in _grid(N)])
        assert abs(f - min(1.0, p_y / q_y)) <= 1.0 / N


def test_eq7_residual_mass_two_forms_and_the_worked_totals():
    for seed in range(5):
        p, q = _laws(seed)
        r, Z = sp.residual(p, q)
        assert abs(Z - (1.0 - np.minimum(p, q).sum())) < 1e-12
        assert np.all(r >= 0) and np.all(r[p <= q] == 0)
    g = GOLD["speculative_sampling_example"]
    # a two-law pair with the review's totals: accepted mass 0.7, the whole residual on "A"
    p = np.array([0.5, 0.3, 0.2])   # tokens A, B, C
    q = np.array([0.2, 0.4, 0.4])
    r, Z = sp.residual(p, q)
    assert abs(np.minimum(p, q).sum() - g["accept_total"]) < 1e-12
    assert abs(Z - g["residual_mass"]) < 1e-12
    assert np.flatnonzero(r).tolist() == [0]          # every rejection is corrected to A
    assert all(sp.sample_inverse_cdf(r, u) == 0 for u in _grid(100))


def _emitted_law(step, p, q, n, seed):
    rng = np.random.default_rng(seed)
    u = rng.random((n, 3))
    out = np.bincount([step(p, q, *u[i])[0] for i in range(n)], minlength=len(p))
    return out / n


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_eq8_emitted_token_has_the_target_law(seed):
    p, q = _laws(seed)
    n = 60000
    f = _emitted_law(sp.speculative_step, p, q, n, 100 + seed)
    assert np.abs(f - p).max() < 5 * np.sqrt(0.25 / n)


def test_eq8_catches_resampling_from_the_target_on_rejection():
    """The mistake the review names: on rejection, drawing from p instead of
    the residual gives the wrong mixture."""
    def wrong(p, q, ud, ua, ue):
        y = sp.sample_inverse_cdf(q, ud)
        if ua < sp.accept_probability(p[y], q[y]):
            return y, True
        return sp.sample_inverse_cdf(p, ue), False

    p, q = _laws(0)
    n = 60000
    assert np.abs(_emitted_law(wrong, p, q, n, 7) - p).max() > 10 * np.sqrt(0.25 / n)


def test_identical_laws_accept_every_proposal():
    p, _ = _laws(3)
    rng = np.random.default_rng(4)
    for _ in range(200):
        ud, ua, ue = rng.random(3)
        y, acc = sp.speculative_step(p, p, ud, ua, ue)
        assert acc and y == sp.sample_inverse_cdf(p, ud)


def test_zero_temperature_limit_is_the_greedy_round():
    """At T -> 0 the laws are one-hot at the argmax: the sampled round makes the
    greedy round's choices (no near-ties in this fixture)."""
    cfg = configs.get("tiny_f32_b3")
    m = om.Model(cfg)
    p = synth.prompts(cfg)[0]
    st_g = spec.prefill(m, p)
    st_s = copy.deepcopy(st_g)
    rng = np.random.default_rng(5)
    B1 = cfg.block_size - 1
    for _ in range(4):
        d, dl = spec.draft(m, st_g)
        rg = spec.verify(m, st_g, d)
        y, q, _ = sp.draft_sampled(m, st_s, 1e-9, rng.random(B1))
        assert np.array_equal(y, d)
        rs = sp.verify_sampled(m, st_s, y, q, 1e-9, rng.random(B1), float(rng.random()))
        assert (rs.accepted, rs.bonus) == (rg.accepted, rg.bonus)
        assert st_s.committed == st_g.committed


def test_round_emits_its_first_token_with_the_target_law():
    """Whole round (draft, acceptance, residual): on a toy model the first token
    a sampled round emits has the target's law after the anchor (eq. 8 applied
    to the round), whatever the drafter proposes."""
    w = configs.get("tiny_f32").with_(name="toy_sampling", vocab=16, d_model=32, n_heads=2, n_kv_heads=1,
                                      head_dim=16, ffn=64, target_layers=2, draft_layers=1, ctx_layer_ids=(0, 1),
                                      block_size=4, prompt_lens=(6,), weight_std=0.5)
    m = om.Model(w)
    T = 1.0
    st0 = spec.prefill(m, synth.prompts(w)[0])
    # the target's law of the token after the anchor
    lg, _ = m.target_forward([st0.anchor], st0.tcache.copy())
    p0 = sp.softmax_t(lg[0], T)
    rng = np.random.default_rng(21)
    n = 6000
    counts = np.zeros(w.vocab)
    B1 = w.block_size - 1
    for _ in range(n):
        st = copy.deepcopy(st0)
        y, q, _ = sp.draft_sampled(m, st, T, rng.random(B1))
        rd = sp.verify_sampled(m, st, y, q, T, rng.random(B1), float(rng.random()))
        first = int(y[0]) if rd.accepted >= 1 else rd.bonus
        counts[first] += 1
    assert np.abs(counts / n - p0).max() < 5 * np.sqrt(0.25 / n)


def test_round_pin_catches_resampling_from_the_target(monkeypatch):
    """The same whole-round check fails when a rejection draws from p instead of the residual."""
    monkeypatch.setattr(sp, "residual", lambda p, q: (np.asarray(p, np.float64), 1.0))
    with pytest.raises(AssertionError):
        test_round_emits_its_first_token_with_the_target_law()


def test_all_accepted_emits_the_bonus_from_the_last_block_row():
    """Algorithm 1's last step: when every proposal survives (acceptance uniforms of 0
    accept any token the target gives positive mass), the emitted token is the draw
    from the target's law at the last block row, p_{B-1} -- the law after the last
    proposal, not after the anchor or an earlier proposal."""
    w = configs.get("tiny_f32").with_(name="toy_bonus", vocab=16, d_model=32, n_heads=2, n_kv_heads=1,
                                      head_dim=16, ffn=64, target_layers=2, draft_layers=1, ctx_layer_ids=(0, 1),
                                      block_size=4, prompt_lens=(6,), weight_std=0.5)
    m = om.Model(w)
    T, B1 = 0.7, w.block_size - 1
    st0 = spec.prefill(m, synth.prompts(w)[0])
    rng = np.random.default_rng(5)
    seen_rows = set()
    for u_emit in _grid(40):
        st = copy.deepcopy(st0)
        y, q, _ = sp.draft_sampled(m, st, T, rng.random(B1))
        lg, _ = m.target_forward(np.concatenate([[st0.anchor], y]), st0.tcache.copy())
        rd = sp.verify_sampled(m, st, y, q, T, np.zeros(B1), float(u_emit))
        assert rd.accepted == B1
        laws = [sp.softmax_t(lg[j], T) for j in range(w.block_size)]
        draws = [sp.sample_inverse_cdf(pj, float(u_emit)) for pj in laws]
        assert rd.bonus == draws[B1]
        seen_rows.update(j for j in range(B1) if draws[j] != draws[B1])
    assert seen_rows == set(range(B1))   # every other row's law would have given a different token somewhere
