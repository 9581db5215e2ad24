"""Pins of the drafter's own block pass, from hand-made weights whose output
has a closed form.

What they fix ("DFlash: Block Diffusion for Flash Speculative Decoding",
Paper vs code "Drafted tokens match" and "KV injection matches, with extras",
Pitfalls "Positional encoding"):

* the drafted tokens are the argmax of the target's shared head on the B-1
  mask rows; the anchor row (row 0) is dropped, and the block rows are the
  anchor and B-1 mask ids embedded with the target's own table;
* the block's queries pass through the per-head RMSNorm, so scaling the
  query projection changes nothing;
* the block occupies positions n .. n+B-1 right after the n context entries,
  so RoPE places the anchor query at n, one step after the last context key.

Each pin fails under a mistake planted in ``tests/test_oracle_mutations.py``.
"""
import math

import numpy as np
import pytest

import synth
from synth import configs
from oracle import model as om, spec


def _rms(x, eps):
    """x / sqrt(mean(x^2) + eps) with unit scales, row by row."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)


def _mats_model(cfg, mats):
    return om.Model(cfg, weights=om.Weights(lambda name: mats[name]), act_round=False)


# ------------------------------------------------- (i) rows, embedding, head
def _passthrough_drafter(B):
    """One draft layer whose output projection and MLP gate are zero: the block's
    hidden states leave the layer unchanged, so row j's logits are
    rms(embed[token_j]) through an identity head (vocab = width)."""
    d, V = 16, 16
    cfg = configs.get("tiny_f32").with_(d_model=d, vocab=V, n_heads=2, n_kv_heads=1, head_dim=8, ffn=8,
                                        draft_layers=1, block_size=B)
    rng = np.random.default_rng(21)
    embed = 0.1 * rng.standard_normal((V, d))
    anchor = 2
    embed[anchor, 5] = 3.0                     # the anchor's own argmax would be token 5
    embed[cfg.mask_token, 9] = 2.0             # every mask row's argmax is token 9
    mats = {"embed": embed, "head": np.eye(V, d), "draft_norm": np.ones(d),
            "d0.attn_norm": np.ones(d), "d0.mlp_norm": np.ones(d), "d0.q_norm": np.ones(8), "d0.k_norm": np.ones(8),
            "d0.wq": rng.standard_normal((16, d)), "d0.wk": rng.standard_normal((8, d)),
            "d0.wv": rng.standard_normal((8, d)), "d0.wo": np.zeros((d, 16)),
            "d0.w_gate": np.zeros((8, d)), "d0.w_up": rng.standard_normal((8, d)),
            "d0.w_down": rng.standard_normal((d, 8))}
    m = _mats_model(cfg, mats)
    cache = m.new_draft_cache()
    cache.append(0, rng.standard_normal((3, 1, 8)), rng.standard_normal((3, 1, 8)))
    return cfg, m, cache, embed, anchor


@pytest.mark.parametrize("B", [2, 4, 7])
def test_drafts_are_the_mask_rows_argmax_through_the_shared_head(B):
    """With the layer passing the embeddings through, every draft is argmax(rms(embed[MASK])),
    there are exactly B-1 of them, and the anchor row's own argmax is not among them."""
    cfg, m, cache, embed, anchor = _passthrough_drafter(B)
    st = spec.SeqState(prompt=np.zeros(3, np.int64), tcache=m.new_target_cache(), dcache=cache, anchor=anchor)
    drafts, lg = spec.draft(m, st)
    tokens = [anchor] + [cfg.mask_token] * (B - 1)
    np.testing.assert_allclose(lg, _rms(embed[tokens], cfg.rms_eps), rtol=1e-12, atol=1e-12)
    assert drafts.shape == (B - 1,)
    assert list(drafts) == [9] * (B - 1)
    assert int(np.argmax(lg[0])) == 5 and 5 not in list(drafts)


# ------------------------------------------------------ (ii) query RMSNorm
@pytest.mark.parametrize("name", ["tiny_f32", "tiny_f32_b3"])
def test_block_queries_are_rms_normalised(name):
    """Scaling every draft layer's query projection by c > 0 leaves the draft logits
    unchanged (q-norm per head before RoPE); a drafter without it would attend with
    c-times sharper scores."""
    cfg = configs.get(name)
    m = om.Model(cfg)
    st = spec.prefill(m, synth.prompts(cfg)[0])
    base = m.draft_forward(st.anchor, st.dcache)

    def scaled(c):
        def get(n, w=m.w):
            x = w(n)
            return c * x if n.startswith("d") and n.endswith(".wq") else x
        return om.Model(cfg, weights=om.Weights(get), act_round=False)

    for c in (0.25, 3.0):
        # q = W_q x has mean square ~1e-2 or more per head here, so the eps of the norm moves
        # the scaled result by a relative ~1e-4 at most
        np.testing.assert_allclose(scaled(c).draft_forward(st.anchor, st.dcache), base, rtol=1e-3, atol=1e-4)


# ------------------------------------------------------ (iii) block positions
def _angle_drafter(n_ctx, B, C=1000.0):
    """A drafter on a 2-dimensional residual with one head of width 2.  At head width 2
    RoPE rotates a query or key by its position in radians (inverse frequency
    theta^0 = 1).  Both embeddings point along (1, 0) and W_q = I, so the query of the
    block row at position p points at angle p.  The n_ctx context keys are placed by
    hand, C times longer than a normalised key, at angles n_ctx + k pi/2 (k = i mod 4)
    with value vals[k]; each block row then attends (to within exp(-300)) to the context
    key whose angle is nearest its own position, and its residual becomes
    embed + vals[k].  W_o = I, the MLP gate is zero and the head is the identity."""
    d = 2
    cfg = configs.get("tiny_f32").with_(d_model=d, vocab=2, n_heads=1, n_kv_heads=1, head_dim=2, ffn=2,
                                        draft_layers=1, block_size=B, rope_theta=1e4)
    embed = np.array([[2.0, 0.0], [0.5, 0.0]])          # token 0 = the anchor, token 1 = MASK
    rng = np.random.default_rng(5)
    eye = np.eye(2)
    mats = {"embed": embed, "head": eye, "draft_norm": np.ones(d), "d0.attn_norm": np.ones(d),
            "d0.mlp_norm": np.ones(d), "d0.q_norm": np.ones(2), "d0.k_norm": np.ones(2), "d0.wq": eye, "d0.wk": eye,
            "d0.wv": rng.standard_normal((2, 2)), "d0.wo": eye, "d0.w_gate": np.zeros((2, 2)), "d0.w_up": eye,
            "d0.w_down": eye}
    m = _mats_model(cfg, mats)
    vals = np.array([[0.3, 1.7], [-1.1, 0.4], [0.9, -0.6], [-0.2, -1.3]])
    ks = np.arange(n_ctx) % 4
    ang = n_ctx + ks * (math.pi / 2)
    keys = C * np.stack([np.cos(ang), np.sin(ang)], axis=1)
    cache = m.new_draft_cache()
    cache.append(0, keys[:, None, :], vals[ks][:, None, :])
    return cfg, m, cache, embed, vals


def _nearest_quarter_turn(offset):
    """k in 0..3 maximising cos(offset - k pi/2)."""
    return int(np.argmax([math.cos(offset - k * math.pi / 2) for k in range(4)]))


@pytest.mark.parametrize("n_ctx", [4, 9, 13])
def test_block_sits_at_positions_n_to_n_plus_B_minus_1(n_ctx):
    """Row j of the block (position n + j) picks the context value at the quarter turn
    nearest j: the anchor (j = 0) the key at angle n itself, so the anchor query sits one
    position after the last context entry (n - 1).  The logits are rms(embed + that value).
    A block placed one position later, or starting at 0, picks other values."""
    B = 4
    cfg, m, cache, embed, vals = _angle_drafter(n_ctx, B)
    lg = m.draft_forward(0, cache)
    tokens = [0] + [cfg.mask_token] * (B - 1)
    picks = [_nearest_quarter_turn(j) for j in range(B)]
    assert picks == [0, 1, 1, 2]
    want = _rms(embed[tokens] + vals[picks], cfg.rms_eps)
    np.testing.assert_allclose(lg, want, rtol=1e-9, atol=1e-9)
    # the same block one position later would pick these instead
    later = [_nearest_quarter_turn(j + 1) for j in range(B)]
    assert later != picks


def test_block_logits_depend_only_on_relative_position():
    """Shifting the context keys and the block together (n = 4, 9, 13 with the keys at
    n + k pi/2) leaves the block's logits unchanged."""
    out = [_angle_drafter(n, 4)[1].draft_forward(0, _angle_drafter(n, 4)[2]) for n in (4, 9, 13)]
    np.testing.assert_allclose(out[1], out[0], rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(out[2], out[0], rtol=1e-9, atol=1e-9)
