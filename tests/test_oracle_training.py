"""Pins of the oracle's training forward ("DFlash: Why a Diffusion Drafter Can
Accelerate an Autoregressive Model" §6, eq. 12, Algorithm 2; "DFlash: Block
Diffusion for Flash Speculative Decoding", Training §4.2).

The packed block-sparse pass is checked against one drafter pass per anchor,
each block against the inference draft pass with the same context and anchor
token, the mask against leakage of tokens at or after the anchor, the weights
against the review's printed values and the loss against its closed form for
a drafter with uniform output."""
import json
import os

import numpy as np
import pytest

import synth
from synth import configs
from oracle import model as om, spec, training as tr

with open(os.path.join(os.path.dirname(__file__), "golden", "pages_values.json")) as _f:
    GOLD = json.load(_f)


def _setup(name="tiny_f32"):
    w = configs.get(name)
    m = om.Model(w)
    x = synth.prompts(w)[0]
    return w, m, np.asarray(x, dtype=np.int64)


def test_position_weights_printed_values():
    g = GOLD["loss_position_weights"]
    assert tr.LAMBDA_FOR_BLOCK == {int(k): float(v) for k, v in g["lambda"].items()}
    w16 = tr.position_weights(16, tr.LAMBDA_FOR_BLOCK[16])
    assert len(w16) == 15 and w16[0] == g["first_weight"]
    assert abs(w16[-1] - g["last_weight_b16"]) <= g["tol"]
    assert np.all(np.diff(w16) < 0)


def test_packed_pass_equals_one_pass_per_anchor():
    w, m, x = _setup()
    anchors = [1, 5, 6, 17, len(x) - w.block_size]      # overlapping spans included
    feats = tr.context_features(m, x)
    packed = tr.packed_block_logits(m, feats, x, anchors)
    for i, a in enumerate(anchors):
        np.testing.assert_allclose(packed[i], tr.block_logits(m, feats, x, a), rtol=1e-10, atol=1e-12)
    assert abs(tr.packed_training_loss(m, x, anchors, 3.0) - tr.training_loss(m, x, anchors, 3.0)) < 1e-10


def test_blocks_see_no_token_at_or_after_their_anchor_but_their_own():
    w, m, x = _setup()
    anchors = [3, 9, 20]
    base = tr.packed_block_logits(m, tr.context_features(m, x), x, anchors)
    for i, a in enumerate(anchors):
        y = x.copy()
        y[a + 1:] = (y[a + 1:] + 17) % w.vocab          # every token after the anchor changes
        lg = tr.packed_block_logits(m, tr.context_features(m, y), y, anchors)
        np.testing.assert_allclose(lg[i], base[i], rtol=1e-12, atol=1e-12)
        for j in range(i + 1, len(anchors)):              # later blocks do see those tokens
            assert np.abs(lg[j] - base[j]).max() > 1e-6


def test_block_equals_the_inference_draft_with_the_same_context_and_anchor():
    """A training block is the draft pass of a round whose committed prefix is
    x[:a] and whose anchor is x[a] (the review's 'one clean anchor')."""
    w, m, x = _setup()
    feats = tr.context_features(m, x)
    for a in (2, 11, 25):
        st = spec.prefill(m, x[:a])
        np.testing.assert_allclose(m.draft_forward(int(x[a]), st.dcache), tr.block_logits(m, feats, x, a),
                                   rtol=1e-10, atol=1e-12)


def test_a_context_that_includes_the_anchor_feature_is_caught():
    w, m, x = _setup()
    feats = tr.context_features(m, x)
    a = 11
    dc = m.new_draft_cache()
    m.append_context(feats[:a + 1], dc)                   # leaks the anchor's own feature
    st = spec.prefill(m, x[:a])
    assert np.abs(m.draft_forward(int(x[a]), dc) - m.draft_forward(int(x[a]), st.dcache)).max() > 1e-6


def test_loss_of_a_uniform_drafter_is_log_vocab_times_the_weights():
    w = configs.get("tiny_f32")
    base = om.Model(w)

    def get(name, wfn=base.w):
        v = wfn(name)
        return np.zeros_like(v) if name == "head" else v

    m = om.Model(w, weights=om.Weights(get), act_round=False)
    x = np.asarray(synth.prompts(w)[0], dtype=np.int64)
    anchors = [1, 7, 19]
    lam = 2.5
    want = np.log(w.vocab) * tr.position_weights(w.block_size, lam).sum()
    assert abs(tr.training_loss(m, x, anchors, lam) - want) < 1e-10


def test_anchor_range_is_checked():
    w, m, x = _setup()
    with pytest.raises(ValueError):
        tr.training_loss(m, x, [0], 3.0)
    with pytest.raises(ValueError):
        tr.training_loss(m, x, [len(x) - w.block_size + 1], 3.0)


@pytest.mark.parametrize("B,lam", [(16, 7.0), (10, 5.0), (4, 3.0)])
def test_each_position_predicts_the_token_k_after_the_anchor_with_weight_k(B, lam):
    """Closed form of eq. 12 for hand-made logits: every predicted row k = 1..B-1
    puts (practically) all mass on x[a+k] except row k0, which is uniform over V;
    the block loss is then exp(-(k0-1)/lambda) * log V.  A label shifted by one
    position or a weight exponent off by one gives a different value."""
    V, a = 40, 5
    x = np.random.default_rng(7).integers(0, V, size=a + B + 3)
    for k0 in range(1, B):
        lg = np.full((B, V), -1e4)
        for k in range(1, B):
            lg[k, x[a + k]] = 0.0
        lg[k0] = 0.0
        want = np.exp(-(k0 - 1) / lam) * np.log(V)
        assert abs(tr.block_loss(lg, x, a, lam) - want) < 1e-9 * want
