"""Pins of the oracle's draft-and-verify loop.

The whole-path pin is losslessness: greedy speculative output must equal the
target's plain greedy decode ("DFlash: Block Diffusion for Flash Speculative
Decoding", Method step 5 and Pitfalls "Lossless claim"; "DFlash: Why a
Diffusion Drafter Can Accelerate an Autoregressive Model" §4.1).  The cache
logic is pinned against from-scratch recomputation, acceptance against its
characterisation, and the accounting against the pages' worked values.
"""
import itertools
import json
import os

import numpy as np
import pytest

import synth
from synth import configs
from oracle import metrics, model as om, spec

with open(os.path.join(os.path.dirname(__file__), "golden", "pages_values.json")) as _f:
    GOLD = json.load(_f)


def _model(name, **kw):
    cfg = configs.get(name)
    if kw:
        cfg = cfg.with_(**kw)
    return om.Model(cfg), cfg


# ------------------------------------------------------------------ acceptance
def test_acceptance_exhaustive_characterisation():
    """a is the unique count with d[:a] == p[:a] and (a == m or d[a] != p[a])."""
    for m in range(0, 4):
        for d in itertools.product(range(3), repeat=m):
            for p in itertools.product(range(3), repeat=m + 1):
                a = spec.count_leading_matches(d, p[:-1])
                assert 0 <= a <= m
                assert list(d[:a]) == list(p[:a])
                assert a == m or d[a] != p[a]
                # emitted tokens d[:a] + [p[a]] are the target's choices at every emitted position
                emitted = list(d[:a]) + [p[a]]
                assert emitted == list(p[: a + 1])


def test_tau_counts_bonus():
    g = GOLD["tau_counts_bonus"]
    for a, t in zip(g["accepted"], g["tau"]):
        assert metrics.tau_from_accepts([a]) == t


# ------------------------------------------------------------------ lossless
@pytest.mark.parametrize("name", ["tiny_f32", "tiny_f32_b3"])
@pytest.mark.parametrize("block", [1, 2, 4, 7])
def test_lossless_tiny_block_sizes(block, name):
    m, cfg = _model(name, block_size=block)
    p = synth.prompts(cfg)[0]
    ar, _ = spec.ar_generate(m, p, 40)
    st = spec.generate(m, p, 40)
    assert np.array_equal(np.array(st.generated), ar)
    if block == 1:
        assert all(r.accepted == 0 for r in st.rounds) and len(st.rounds) == 39


def test_lossless_ragged_batch_and_planted():
    m, cfg = _model("tiny_f32_b3")
    for p in synth.prompts(cfg):
        ar, _ = spec.ar_generate(m, p, cfg.max_new_tokens)
        assert np.array_equal(np.array(spec.generate(m, p, cfg.max_new_tokens).generated), ar)
        for taus in ([1], [4], [6, 7], [2, 4, 1, 3]):
            st = spec.generate(m, p, cfg.max_new_tokens, proposer=spec.planted_proposer(ar, taus, cfg.vocab))
            assert np.array_equal(np.array(st.generated), ar)
            want = [min(taus[i % len(taus)], cfg.block_size) - 1 for i in range(len(st.rounds))]
            # the final round may run past max_new_tokens but still accepts as planted
            assert [r.accepted for r in st.rounds] == want


@pytest.mark.parametrize("act_round", [False, True])
def test_lossless_small_bf16(act_round):
    m, cfg = _model("small_bf16")
    m.act_round = act_round
    p = synth.prompts(cfg)[0]
    ar, _ = spec.ar_generate(m, p, 24)
    st = spec.generate(m, p, 24, proposer=spec.planted_proposer(ar, [6, 7], cfg.vocab))
    assert np.array_equal(np.array(st.generated), ar)
    assert [r.accepted for r in st.rounds][:3] == [5, 6, 5]


# ------------------------------------------------- runtime block size (B' <= B)
def test_lossless_with_a_runtime_block_schedule():
    """Rounds at blocks 7, 3, 1, 5 of a drafter configured at 7: output equals
    plain greedy, each round accepts at most B'-1 drafts, and planted proposals
    are accepted to min(tau, B') - 1."""
    m, cfg = _model("tiny_f32", block_size=7)
    p = synth.prompts(cfg)[0]
    ar_long, _ = spec.ar_generate(m, p, 48 + 7)    # the last round's proposal may reach past token 48
    ar = ar_long[:48]
    sched = [7, 3, 1, 5]
    st = spec.generate(m, p, 48, block_schedule=sched)
    assert np.array_equal(np.array(st.generated), ar)
    for i, r in enumerate(st.rounds):
        assert len(r.posterior) == sched[i % 4] and 0 <= r.accepted <= sched[i % 4] - 1
    taus = [6, 2, 4, 3, 7]
    st = spec.generate(m, p, 48, proposer=spec.planted_proposer(ar_long, taus, cfg.vocab), block_schedule=sched)
    assert np.array_equal(np.array(st.generated), ar)
    assert [r.accepted for r in st.rounds] == [min(taus[i % 5], sched[i % 4]) - 1 for i in range(len(st.rounds))]


def test_runtime_block_is_the_model_configured_at_that_block():
    """The B' view of a B-configured model drafts exactly like a model whose
    configuration says B' (the synthetic weights do not depend on B), and B'
    outside [1, B] is refused."""
    m, cfg = _model("tiny_f32", block_size=7)
    st = spec.prefill(m, synth.prompts(cfg)[0])
    small = om.Model(cfg.with_(block_size=3))
    np.testing.assert_array_equal(spec.at_block_size(m, 3).draft_forward(st.anchor, st.dcache),
                                  small.draft_forward(st.anchor, st.dcache))
    for bad in (0, 8):
        with pytest.raises(ValueError):
            spec.at_block_size(m, bad)


# ------------------------------------------------------------- cache pins
def _committed_tokens(st):
    seq = np.concatenate([st.prompt, np.array(st.generated, dtype=np.int64)])
    return seq[: st.committed]


@pytest.mark.parametrize("schedule", [None, [4, 2, 1, 3]])
def test_incremental_context_equals_recompute(schedule):
    """Context K/V built round by round from verify passes (a+1 rows each)
    equals the context K/V recomputed from a fresh target pass over the
    committed sequence (also when the block size changes between rounds)."""
    m, cfg = _model("tiny_f32_b3")
    p = synth.prompts(cfg)[1]
    ar, _ = spec.ar_generate(m, p, 30)
    st = spec.generate(m, p, 30, proposer=spec.planted_proposer(ar, [3, 1, 4, 2], cfg.vocab),
                       block_schedule=schedule)
    seq = _committed_tokens(st)
    assert st.dcache.length == st.tcache.length == st.committed == len(p) + sum(r.accepted + 1 for r in st.rounds)
    tc, dc = m.new_target_cache(), m.new_draft_cache()
    _, sel = m.target_forward(seq, tc)
    m.append_context(m.fuse(sel), dc)
    for l in range(cfg.draft_layers):
        np.testing.assert_allclose(st.dcache.k[l], dc.k[l], rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(st.dcache.v[l], dc.v[l], rtol=1e-9, atol=1e-12)
    for l in range(cfg.target_layers):
        np.testing.assert_allclose(st.tcache.k[l], tc.k[l], rtol=1e-9, atol=1e-12)
    # the next draft from the incremental cache equals the draft from the recomputed one
    np.testing.assert_allclose(m.draft_forward(st.anchor, st.dcache), m.draft_forward(st.anchor, dc),
                               rtol=1e-9, atol=1e-12)


def test_verify_posterior_equals_fresh_forward():
    m, cfg = _model("tiny_f32")
    p = synth.prompts(cfg)[0]
    st = spec.prefill(m, p)
    for _ in range(3):
        d, _ = spec.draft(m, st)
        seq = _committed_tokens(st)
        rd = spec.verify(m, st, d, keep_logits=True)
        lg, _ = m.target_forward(np.concatenate([seq, [rd.anchor], d]), m.new_target_cache())
        np.testing.assert_allclose(rd.verify_logits, lg[-cfg.block_size:], rtol=1e-9, atol=1e-12)


def test_draft_pass_leaves_context_unchanged():
    m, cfg = _model("tiny_f32")
    st = spec.prefill(m, synth.prompts(cfg)[0])
    before = st.dcache.copy()
    spec.draft(m, st)
    spec.draft(m, st)
    for l in range(cfg.draft_layers):
        assert np.array_equal(before.k[l], st.dcache.k[l]) and np.array_equal(before.v[l], st.dcache.v[l])


def test_context_really_conditions_the_draft():
    """KV injection is live: perturbing one stored context row changes the block's logits."""
    m, cfg = _model("tiny_f32")
    st = spec.prefill(m, synth.prompts(cfg)[0])
    base = m.draft_forward(st.anchor, st.dcache)
    c2 = st.dcache.copy()
    c2.v[0][3] += 1.0
    assert np.abs(m.draft_forward(st.anchor, c2) - base).max() > 1e-4


def test_draft_block_is_bidirectional():
    """Row 0 (the anchor) sees the mask rows after it: changing the mask token's
    embedding changes the anchor row's output."""
    m, cfg = _model("tiny_f32")
    st = spec.prefill(m, synth.prompts(cfg)[0])
    base = m.draft_forward(st.anchor, st.dcache)

    def get(name, w=m.w):
        x = w(name)
        if name == "embed":
            x = x.copy()
            x[cfg.mask_token] += 0.05
        return x

    alt = om.Model(cfg, weights=om.Weights(get), act_round=False)
    lg = alt.draft_forward(st.anchor, st.dcache)
    assert np.abs(lg[0] - base[0]).max() > 1e-6


# ------------------------------------------------------------- printed values
def test_tau_geometric_printed_values():
    for g in GOLD["tau_geometric"]:
        assert abs(metrics.tau_geometric(g["a"], g["m"]) - g["tau"]) <= g["tol"]


def test_tau_tail_sum_equals_mean():
    a = np.random.default_rng(3).integers(0, 16, 1000)
    assert abs(metrics.tau_tail_sum(a, 15) - metrics.tau_from_accepts(a)) < 1e-12


def test_speedup_printed_values():
    for g in GOLD["speedup"]:
        assert abs(metrics.speedup(g["tau"], g["r_d"], g["r_v"], g["r_o"]) - g["S"]) <= g["tol"]
    # eq. 5: speedup above one iff tau exceeds the summed normalised costs
    assert metrics.speedup(1.5, 0.3, 1.0, 0.1) > 1 and metrics.speedup(1.3, 0.3, 1.0, 0.1) < 1


def test_memory_printed_values():
    g = GOLD["fusion_param_bytes"]
    assert metrics.fusion_param_bytes(g["width"], g["n_features"], g["bytes_per"]) == g["bytes"]
    g = GOLD["fusion_io_mb"]
    i, o = metrics.fusion_io_bytes(g["width"], g["n_features"], g["rows"])
    assert abs(i / 1e6 - g["in_mb"]) / g["in_mb"] <= g["rel_tol"]
    assert abs(o / 1e6 - g["out_mb"]) / g["out_mb"] <= g["rel_tol"]
    g = GOLD["per_round_fusion_input_bytes_below"]
    assert metrics.fusion_io_bytes(g["width"], g["n_features"], g["block"])[0] < g["below_bytes"]


def test_context_layer_ids_printed_lists():
    for g in GOLD["context_layer_ids"]:
        assert metrics.context_layer_ids(g["target_layers"], g["n_features"]) == g["ids"]
    for name in ("qwen3_8b_b1_p512", "llama31_8b_b8_p1024"):
        cfg = configs.get(name)
        assert list(cfg.ctx_layer_ids) == metrics.context_layer_ids(cfg.target_layers, 5)
