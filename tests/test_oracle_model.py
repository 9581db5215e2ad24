"""Pins of the oracle's context feature ("DFlash: Why a Diffusion Drafter Can
Accelerate an Autoregressive Model" §5.1 eq. 9; "DFlash: Block Diffusion for
Flash Speculative Decoding", Paper vs code "Feature indexing"): the fused
feature is RMSNorm(W_c [h_l1; ...; h_lk]) of the residual stream after each
selected target layer.  Each pin fails for a plausible slip: a dropped norm, a
dropped layer block, or a hidden state taken one layer early."""
import numpy as np
import pytest

import synth
from synth import configs
from oracle import model as om


def _sel(name):
    w = configs.get(name)
    m = om.Model(w)
    x = np.asarray(synth.prompts(w)[0], dtype=np.int64)
    _, sel = m.target_forward(x, m.new_target_cache(), want_logits=False)
    return w, m, x, sel


@pytest.mark.parametrize("name", ["tiny_f32", "tiny_f32_b3"])
def test_feature_rows_are_rms_normalised(name):
    """Divided by its norm scale, every feature row has unit root-mean-square, and the
    feature does not change when the selected states are scaled (RMSNorm after W_c)."""
    w, m, x, sel = _sel(name)
    f = m.fuse(sel)
    g = f / m.w("fc_norm")
    # eps (1e-6) keeps the RMS just below one: sqrt(ms / (ms + eps)) with ms ~ 3e-3 here;
    # without the norm the rows would keep the raw scale of W_c h (RMS ~ 0.07)
    rms = np.sqrt((g ** 2).mean(axis=-1))
    assert np.all(rms <= 1.0) and np.all(rms > 0.99), rms
    np.testing.assert_allclose(m.fuse(3.0 * sel), f, rtol=1e-2, atol=1e-3)


def test_feature_uses_every_selected_layer():
    w, m, x, sel = _sel("tiny_f32")
    d, k = w.d_model, len(w.ctx_layer_ids)
    f = m.fuse(sel)
    for i in range(k):
        s2 = sel.copy()
        s2[:, i * d:(i + 1) * d] *= -1.0
        assert np.abs(m.fuse(s2) - f).max() > 1e-3, f"layer block {i} does not reach the feature"


@pytest.mark.parametrize("layer", [0, 1, 3])
def test_selected_state_is_the_residual_after_the_layer(layer):
    """A model cut after target layer l (same weights) feeds its final norm exactly the
    state the full model selects for layer l: the residual after layer l (0-based)."""
    w = configs.get("tiny_f32").with_(ctx_layer_ids=(0, 1, 3))
    m = om.Model(w)
    x = np.asarray(synth.prompts(w)[0], dtype=np.int64)
    _, sel = m.target_forward(x, m.new_target_cache(), want_logits=False)
    i = w.ctx_layer_ids.index(layer)
    h = sel[:, i * w.d_model:(i + 1) * w.d_model]
    cut = om.Model(w.with_(target_layers=layer + 1, ctx_layer_ids=(layer,)), weights=m.w)
    lg_cut, _ = cut.target_forward(x, cut.new_target_cache())
    np.testing.assert_allclose(m.logits(h, "final_norm"), lg_cut, rtol=1e-9, atol=1e-9)
    if layer > 0:   # the state one layer earlier is a different one
        prev = om.Model(w.with_(target_layers=layer, ctx_layer_ids=(layer - 1,)), weights=m.w)
        lg_prev, _ = prev.target_forward(x, prev.new_target_cache())
        assert np.abs(m.logits(h, "final_norm") - lg_prev).max() > 1e-3


def test_context_values_are_linear_in_the_feature():
    """Context injection (eq. 10): V = W_V f with no norm in between, so doubling the
    feature doubles the stored values; K = RoPE(k_norm(W_K f)) is per-head normalised,
    so it does not change.  An extra RMSNorm of the feature before the projections
    would make V scale-invariant, and a missing k-norm would double K."""
    w, m, x, sel = _sel("tiny_f32_b3")
    f = m.fuse(sel)
    c1, c2 = m.new_draft_cache(), m.new_draft_cache()
    m.append_context(f, c1)
    m.append_context(2.0 * f, c2)
    for l in range(w.draft_layers):
        np.testing.assert_allclose(c2.v[l], 2.0 * c1.v[l], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(c2.k[l], c1.k[l], rtol=1e-3, atol=1e-4)
        assert np.abs(c1.k[l]).max() > 1e-2


def _layer_model(d, gate_scale):
    """A model whose layer t0 has W_o = I, unit norms, W_gate = s I, W_up = I, W_down = I."""
    w = configs.get("tiny_f32").with_(d_model=d, ffn=d, n_heads=1, n_kv_heads=1, head_dim=d)
    eye = np.eye(d)
    mats = {"t0.wo": eye, "t0.mlp_norm": np.ones(d), "t0.w_gate": gate_scale * eye, "t0.w_up": eye,
            "t0.w_down": eye}
    return w, om.Model(w, weights=om.Weights(lambda name: mats[name]), act_round=False)


def test_swiglu_gates_through_silu_of_the_gate_projection():
    """x + W_down (silu(W_gate xn) * W_up xn) with xn = rms_norm(x): with W_gate = g I for a
    large |g|, silu(g z) tends to max(g z, 0), so the update is max(g xn, 0) * xn -- open where
    g xn > 0, closed elsewhere.  Applying the SiLU to the up projection instead, or swapping
    the two projections, gives another update."""
    d, s = 64, 60.0
    x = np.random.default_rng(2).normal(size=(3, d))
    att = np.zeros((3, 1, d))                   # no attention update: only the MLP acts
    for g in (s, -s):
        w, m = _layer_model(d, g)
        xn = om.rms_norm(x, np.ones(d), w.rms_eps)
        want = x + np.maximum(g * xn, 0.0) * xn
        big = np.abs(xn) > 0.2                  # away from the kink: silu(g z) = max(g z, 0) to ~1e-4
        got = m._attn_out_mlp("t0", x, att)
        np.testing.assert_allclose(got[big], want[big], rtol=1e-4, atol=1e-4)
        assert np.abs(got - x)[big].max() > 1.0  # the MLP really acts


def test_one_token_layer_is_pre_norm_with_residuals():
    """A one-token pass through a layer with W_v = W_o = I and a closed MLP gate (W_gate = 0,
    silu(0) = 0): the token attends only to itself, so the residual after the layer is
    e + rms_norm(e) (pre-norm attention input, values of the normalised input, residual
    add), and the logits through an identity head are rms_norm(e + rms_norm(e))."""
    d = 32
    w = configs.get("tiny_f32").with_(d_model=d, ffn=d, n_heads=2, n_kv_heads=2, head_dim=d // 2, vocab=d,
                                      target_layers=1, ctx_layer_ids=(0,), target_qk_norm=False)
    rng = np.random.default_rng(9)
    eye = np.eye(d)
    mats = {"embed": rng.normal(size=(d, d)), "t0.attn_norm": np.ones(d), "t0.wq": rng.normal(size=(d, d)),
            "t0.wk": rng.normal(size=(d, d)), "t0.wv": eye, "t0.wo": eye, "t0.mlp_norm": np.ones(d),
            "t0.w_gate": np.zeros((d, d)), "t0.w_up": eye, "t0.w_down": eye, "final_norm": np.ones(d), "head": eye}
    m = om.Model(w, weights=om.Weights(lambda name: mats[name]), act_round=False)
    tok = 5
    lg, sel = m.target_forward([tok], m.new_target_cache())
    e = mats["embed"][tok]
    after = e + om.rms_norm(e, np.ones(d), w.rms_eps)
    np.testing.assert_allclose(sel[0], after, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lg[0], om.rms_norm(after, np.ones(d), w.rms_eps), rtol=1e-12, atol=1e-12)
