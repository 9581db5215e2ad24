"""Planted mistakes in the oracle (CPU only) must be caught by its pins.

Each case patches one plausible error into the oracle and checks that the pin
meant to guard that step fails."""
import numpy as np
import pytest

import synth
from synth import configs
from oracle import model as om, spec


def _lossless(m, cfg, n=30, taus=(3, 1, 4)):
    p = synth.prompts(cfg)[0]
    ar, _ = spec.ar_generate(om.Model(cfg, weights=m.w), p, n)      # reference from the unpatched pieces
    st = spec.generate(m, p, n, proposer=spec.planted_proposer(ar, list(taus), cfg.vocab))
    return np.array_equal(np.array(st.generated), ar)


def test_rollback_off_by_one_is_caught(monkeypatch):
    cfg = configs.get("tiny_f32_b3")
    m = om.Model(cfg)
    assert _lossless(m, cfg)
    orig = spec.verify

    def bad_verify(model, st, proposal, **kw):
        rd = orig(model, st, proposal, **kw)
        st.tcache.truncate(st.tcache.length - 1)      # keeps a rows instead of a + 1
        return rd

    monkeypatch.setattr(spec, "verify", bad_verify)
    try:
        ok = _lossless(m, cfg)
    except Exception:
        ok = False
    assert not ok


def test_acceptance_shift_is_caught(monkeypatch):
    cfg = configs.get("tiny_f32_b3")
    m = om.Model(cfg)

    def shifted(d, p):                                  # compares d[j] with the posterior one step late
        a = 0
        p = list(p) + [-1]
        for j, x in enumerate(d):
            if int(x) != int(p[j + 1]):
                break
            a += 1
        return a

    monkeypatch.setattr(spec, "count_leading_matches", shifted)
    # Under-acceptance still emits true tokens, so losslessness alone cannot see
    # this mistake; the planted-count pin does.
    p = synth.prompts(cfg)[0]
    ar, _ = spec.ar_generate(m, p, 30)
    st = spec.generate(m, p, 30, proposer=spec.planted_proposer(ar, [4], cfg.vocab))
    assert [r.accepted for r in st.rounds] != [3] * len(st.rounds)


def test_context_append_dropping_bonus_row_is_caught(monkeypatch):
    """Appending features for a rows (dropping the anchor's) breaks the
    incremental == recompute pin."""
    cfg = configs.get("tiny_f32_b3")
    m = om.Model(cfg)
    orig_fuse = m.fuse
    calls = {"n": 0}

    def fuse_skip_first_row(sel):
        calls["n"] += 1
        return orig_fuse(sel) if calls["n"] == 1 else orig_fuse(sel)[1:]

    monkeypatch.setattr(m, "fuse", fuse_skip_first_row)
    p = synth.prompts(cfg)[1]
    ar, _ = spec.ar_generate(om.Model(cfg, weights=m.w), p, 20)
    st = spec.generate(m, p, 20, proposer=spec.planted_proposer(ar, [3, 2], cfg.vocab))
    assert st.dcache.length != st.tcache.length


def test_rope_sign_error_is_caught():
    x = np.random.default_rng(1).standard_normal((3, 2, 8))
    pos = np.array([1, 2, 3])

    def bad_rope(x, pos, theta):
        return om.rope(x, -pos, theta)

    from tests.test_oracle_primitives import _rope_complex
    assert not np.allclose(bad_rope(x, pos, 1e4), _rope_complex(x, pos, 1e4))


def test_attention_without_scale_is_caught():
    rng = np.random.default_rng(2)
    q, k, v = rng.standard_normal((3, 2, 8)), rng.standard_normal((5, 1, 8)), rng.standard_normal((5, 1, 8))
    vis = np.ones((3, 5), bool)
    from tests.test_oracle_primitives import _attention_loops
    bad = om.attention(q * np.sqrt(8), k, v, vis)          # i.e. scores not divided by sqrt(hd)
    assert not np.allclose(bad, _attention_loops(q, k, v, vis))
