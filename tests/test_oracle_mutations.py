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


# ------------------------------------------------ the drafter's block pass
def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def test_draft_of_the_wrong_rows_is_caught(monkeypatch):
    """Argmax over rows 0..B-2 (keeping the anchor row, dropping the last mask row)."""
    from tests import test_oracle_drafter as pins

    def bad_draft(model, st):
        lg = model.draft_forward(st.anchor, st.dcache)
        return om.argmax_lowest(lg[:-1]), lg

    monkeypatch.setattr(spec, "draft", bad_draft)
    assert _fails(pins.test_drafts_are_the_mask_rows_argmax_through_the_shared_head, 4)


def test_missing_query_norm_in_the_drafter_is_caught(monkeypatch):
    """Block queries without the per-head RMSNorm (keys still normalised)."""
    from tests import test_oracle_drafter as pins
    orig = om.Model._qkv

    def qkv_without_qnorm(self, p, x, pos, qk_norm):
        if not p.startswith("d"):
            return orig(self, p, x, pos, qk_norm)
        c, w = self.cfg, self.w
        n = x.shape[0]
        xn = self.r(om.rms_norm(x, w(f"{p}.attn_norm"), c.rms_eps))
        q = (xn @ w(f"{p}.wq").T).reshape(n, c.n_heads, c.head_dim)
        k = (xn @ w(f"{p}.wk").T).reshape(n, c.n_kv_heads, c.head_dim)
        v = (xn @ w(f"{p}.wv").T).reshape(n, c.n_kv_heads, c.head_dim)
        k = om.rms_norm(k, w(f"{p}.k_norm"), c.rms_eps)
        return (self.r(om.rope(q, pos, c.rope_theta)), self.r(om.rope(k, pos, c.rope_theta)), self.r(v))

    monkeypatch.setattr(om.Model, "_qkv", qkv_without_qnorm)
    assert _fails(pins.test_block_queries_are_rms_normalised, "tiny_f32")
    assert _fails(pins.test_block_queries_are_rms_normalised, "tiny_f32_b3")


def _draft_forward_at(shift_fn):
    """The oracle's draft pass with block positions shift_fn(n0, B) instead of n0 .. n0+B-1."""
    def draft_forward(self, anchor, cache):
        c, w = self.cfg, self.w
        B, n0 = c.block_size, cache.length
        pos = shift_fn(n0, B)
        tokens = np.array([anchor] + [c.mask_token] * (B - 1), dtype=np.int64)
        h = w("embed")[tokens].copy()
        for l in range(c.draft_layers):
            p = f"d{l}"
            q, kb, vb = self._qkv(p, h, pos, True)
            K = np.concatenate([cache.k[l], kb], axis=0)
            V = np.concatenate([cache.v[l], vb], axis=0)
            att = om.attention(q, K, V, np.ones((B, n0 + B), dtype=bool))
            h = self._attn_out_mlp(p, h, att)
        return self.logits(h, "draft_norm")
    return draft_forward


@pytest.mark.parametrize("shift", [lambda n0, B: np.arange(n0 + 1, n0 + B + 1),   # one position late
                                   lambda n0, B: np.arange(n0 - 1, n0 + B - 1),   # one position early
                                   lambda n0, B: np.arange(0, B)])                # positions from 0
def test_block_position_offset_is_caught(monkeypatch, shift):
    from tests import test_oracle_drafter as pins
    monkeypatch.setattr(om.Model, "draft_forward", _draft_forward_at(shift))
    assert _fails(pins.test_block_sits_at_positions_n_to_n_plus_B_minus_1, 9)
