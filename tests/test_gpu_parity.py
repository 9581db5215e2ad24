"""GPU path (through the C ABI) against the fp64 CPU oracle on the same seeded
inputs.

fp32 workloads: tokens, acceptance lengths and committed lengths bit-exact;
logits within max-abs 1e-3.  bf16 workloads: logits within max-abs 5e-2 (scaled by
weight std / 0.02 for workloads drawn wider than N(0, 0.02)),
final hidden states within rel-L2 1e-2, tokens identical except where the
oracle's top-2 logit margin is below 5e-2 (after such a position the two
streams may diverge, so the comparison stops there).  The oracle never sees
a GPU result: proposals are built from the oracle's own greedy stream and fed
to both sides.
"""
import numpy as np
import pytest

import synth
from synth import configs
from oracle import model as om, spec

pytestmark = pytest.mark.gpu

F32_LOGIT_TOL = 1e-3
BF16_LOGIT_TOL = 5e-2
BF16_HIDDEN_REL = 1e-2
BF16_MARGIN = 5e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_speculative_ctx_gb300 import build
    build.build()


def _session(w, **kw):
    from block_diffusion_speculative_ctx_gb300 import Session
    return Session(w, **kw)


def _tokens_match(gpu_tok, ora_logits, bf16, near=BF16_MARGIN):
    """Compare argmax tokens; in bf16 return the first index where a mismatch
    sits at a near-tie (-1 if none).  A mismatch at a clear margin fails."""
    ora_tok = np.argmax(ora_logits, axis=-1)
    if not bf16:
        np.testing.assert_array_equal(gpu_tok, ora_tok)
        return -1
    margin = spec.top2_margin(ora_logits)
    bad = np.nonzero(gpu_tok != ora_tok)[0]
    for i in bad:
        assert margin[i] < near, f"token {i}: gpu {gpu_tok[i]} oracle {ora_tok[i]} margin {margin[i]}"
    return int(bad[0]) if len(bad) else -1


def _greedy_stream(m, st, n):
    """The target's plain greedy continuation (first token first) from a prefilled oracle state,
    one single-token causal step at a time on a copy of its cache: the same computation as
    spec.ar_generate without repeating the prefill."""
    cache = st.tcache.copy()
    out = [int(st.anchor)]
    while len(out) < n:
        lg, _ = m.target_forward([out[-1]], cache)
        out.append(int(om.argmax_lowest(lg)[0]))
    return np.array(out, dtype=np.int64)


def _rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def run_stepwise(name, rounds=6, taus=(1, 4, 7, 16, 3, 2), schedule=None, session_kw=None, **wkw):
    """Prefill + `rounds` rounds on both sides; returns the number of
    (sequence, round) pairs compared.  `schedule`: block size of round r =
    schedule[r % len] (dflash_set_block_size on the GPU, the oracle's
    at_block_size view), default the configured block.  A bf16 sequence whose acceptance or bonus
    differs from the oracle's at an exempted near-tie stops being compared (its
    two streams now differ); the other sequences continue."""
    w = configs.get(name)
    if wkw:
        w = w.with_(**wkw)
    bf16 = w.dtype == "bf16"
    # bf16 rounding is relative, so the logit tolerance (stated for N(0, 0.02) weights)
    # scales with the weight std, i.e. with the logit magnitude
    scale = max(1.0, w.weight_std / 0.02)
    ltol = BF16_LOGIT_TOL * scale if bf16 else F32_LOGIT_TOL
    near = BF16_MARGIN * scale
    m = om.Model(w)
    prompts = synth.prompts(w)
    n_ar = 1 + rounds * w.block_size + 1
    states = [spec.prefill(m, p) for p in prompts]
    streams = [_greedy_stream(m, st, n_ar) for st in states]
    props = [spec.planted_proposer(s, taus, w.vocab) for s in streams]
    alive = [True] * len(states)
    sess = _session(w, keep_logits=True, max_seq_len=max(w.prompt_lens) + (rounds + 2) * w.block_size + 8,
                    **(session_kw or {}))
    try:
        first = sess.prefill(prompts)
        plog = sess.logits("prefill")
        for s, st in enumerate(states):
            assert np.abs(plog[s] - st.first_logits).max() <= ltol
            if _tokens_match(first[s:s + 1], st.first_logits[None], bf16, near) >= 0:
                alive[s] = False
        # context K/V after prefill
        for s, st in enumerate(states):
            for l in range(w.draft_layers):
                k = sess.cache("draft", "k", s, l)
                assert k.shape == st.dcache.k[l].shape
                assert _rel_l2(k, st.dcache.k[l]) < (2e-2 if bf16 else 1e-5)
        compared = 0
        for r in range(rounds):
            if not any(alive):
                break
            Bt = schedule[r % len(schedule)] if schedule else w.block_size
            mr = spec.at_block_size(m, Bt) if schedule else m
            if schedule:
                sess.set_block_size(Bt)
                assert sess.B == Bt
            drafts = sess.draft_block()
            dlog = sess.logits("draft") if Bt > 1 else None   # block 1 runs no drafter
            proposals = []
            for s, st in enumerate(states):
                if not alive[s]:
                    proposals.append(np.zeros(Bt - 1, np.int64))
                    continue
                od, odl = spec.draft(mr, st)
                if dlog is not None:
                    assert np.abs(dlog[s] - odl).max() <= ltol, f"round {r} seq {s} draft logits"
                    _tokens_match(drafts[s], odl[1:], bf16, near)      # mismatches only at near-ties
                proposals.append(props[s](st, od))
            prop = np.stack(proposals).astype(np.int32) if Bt > 1 else np.zeros((len(states), 1), np.int32)
            acc, bon = sess.verify(prop)
            vlog = sess.logits("verify")
            post = sess.posterior()
            lens = sess.lengths()
            for s, st in enumerate(states):
                if not alive[s]:
                    continue
                n0 = st.committed
                rd = spec.verify(mr, st, prop[s][: Bt - 1], keep_logits=True)
                assert np.abs(vlog[s] - rd.verify_logits).max() <= ltol, f"round {r} seq {s} verify logits"
                _tokens_match(post[s], rd.verify_logits, bf16, near)
                if acc[s] != rd.accepted or bon[s] != rd.bonus:
                    assert bf16, f"round {r} seq {s}: accepted/bonus differ in fp32"
                    alive[s] = False                             # exempted near-tie changed the stream
                    continue
                assert lens[s] == st.committed == n0 + rd.accepted + 1
                compared += 1
        for s, st in enumerate(states):
            if not alive[s]:
                continue
            for l in (0, w.target_layers - 1):
                k = sess.cache("target", "k", s, l)
                v = sess.cache("target", "v", s, l)
                assert k.shape == st.tcache.k[l].shape
                assert _rel_l2(k, st.tcache.k[l]) < (2e-2 if bf16 else 1e-5)
                assert _rel_l2(v, st.tcache.v[l]) < (2e-2 if bf16 else 1e-5)
        return compared
    finally:
        sess.close()


def test_tiny_f32_stepwise():
    assert run_stepwise("tiny_f32") == 6


def test_tiny_f32_ragged_batch_stepwise():
    assert run_stepwise("tiny_f32_b3") == 3 * 6


def test_small_f32_hd128_block16_stepwise():
    assert run_stepwise("small_f32", rounds=4) == 2 * 4


def test_small_bf16_stepwise():
    assert run_stepwise("small_bf16", rounds=4) >= 4          # of 2 x 4


def test_small_bf16_head_dim_64_stepwise():
    """bf16 with 64-wide heads (16 query heads, 8 per KV head): the separate q/k norm + RoPE +
    store kernel, the 64-wide mma.sync attention for prefill and rounds, and the per-layer
    context K/V GEMMs (the stacked one and the fused epilogues serve 128-wide heads)."""
    assert run_stepwise("small_bf16", rounds=3, taus=(1, 5, 2), head_dim=64, n_heads=16) >= 3


@pytest.mark.parametrize("n_kv", [8, 4, 1])
def test_small_bf16_gqa_ratios_stepwise(n_kv):
    """Query heads per KV head of 1, 2 and 8 (the benchmark models use 4): attention query
    groups of 64 / g vectors per block row, tcgen05 prefill groups of 128 / g rows."""
    assert run_stepwise("small_bf16", rounds=3, taus=(1, 5, 2), n_kv_heads=n_kv) >= 3


def test_small_bf16_llama_ragged_batch_in_a_small_page_pool():
    """Prompts of 64, 5, 130 and 33 tokens in a KV pool of 13 pages, where one run of
    max_seq_len per sequence would take 20: pages are handed out as the sequences grow, so
    each sequence's cache is scattered over the pool (prefill, decode attention, the q/k/v
    store epilogues and the stacked context K/V all follow the page table)."""
    assert run_stepwise("small_bf16_llama", rounds=6, session_kw={"kv_pool_tokens": 13 * 64}) >= 12


def test_page_pool_capacity_errors():
    from block_diffusion_speculative_ctx_gb300 import DFlashError
    w = configs.get("tiny_f32_b3")          # prompts of 32, 7 and 19 tokens
    prompts = synth.prompts(w)
    B = w.block_size
    with _session(w, max_seq_len=256, kv_pool_tokens=2 * 64) as sess:
        with pytest.raises(DFlashError, match="page pool"):
            sess.prefill(prompts)           # three prompts need three pages
    with _session(w, max_seq_len=256, kv_pool_tokens=3 * 64) as sess:
        sess.prefill(prompts)
        wrong = np.zeros((3, B - 1), np.int32)
        with pytest.raises(DFlashError, match="page pool"):
            for _ in range(64):             # one token per round: the 32-token prompt needs a 4th page
                d = sess.draft_block()
                wrong[:] = (d + 1) % w.vocab
                sess.verify(wrong)
        first = sess.prefill(prompts)       # a new batch returns every page to the pool
        m = om.Model(w)
        assert [int(t) for t in first] == [spec.prefill(m, p).anchor for p in prompts]


def test_small_bf16_prompt_longer_than_a_prefill_chunk():
    assert run_stepwise("small_bf16_long", rounds=3) >= 3     # of 2 x 3


def test_small_bf16_llama_batch4_stepwise():
    assert run_stepwise("small_bf16_llama", rounds=4) >= 8    # of 4 x 4


def test_small_bf16_llama_batch12_stepwise():
    # 192 block rows per pass: GEMM tiles of 256 tokens, tokens 128..191 in the tile's second half
    assert run_stepwise("small_bf16_llama_b12", rounds=3) >= 18    # of 12 x 3


def test_small_bf16_long_context_8k_stepwise():
    # 8448 context entries: the draft attention over [context ; block] and the verify attention
    # each walk 133 pages per KV head (8+ key tiles per rank of a 16-CTA cluster); the prefill
    # runs 5 chunks through the tcgen05 causal attention.  Draft and verify logits every round at
    # the stated bf16 tolerances, accepted drafts planted from the oracle's own greedy stream.
    assert run_stepwise("small_bf16_long8k", rounds=3, taus=(1, 3, 2)) >= 3     # of 3 x 3


def test_small_bf16_batch20_persistent_gemm_stepwise():
    # 320 block rows per pass: gate/up (SwiGLU) and the head (argmax, logits kept) run on the
    # persistent kernel with whole tiles, the down projection (residual add, K = 8192) with
    # stream-K pieces summed across CTAs
    assert run_stepwise("small_bf16_b20", rounds=3) >= 20    # of 20 x 3


@pytest.mark.parametrize("block", [8, 10])
def test_small_bf16_block_sizes_8_and_10(block):
    # the LLaMA setup's B = 10 and the smaller block suggested under load
    assert run_stepwise("small_bf16", rounds=3, block_size=block) >= 3        # of 2 x 3


def test_small_bf16_llama_block10_batch4():
    # GQA 4 with 10-row blocks: query groups of 40 vectors
    assert run_stepwise("small_bf16_llama", rounds=3, block_size=10) >= 6     # of 4 x 3


@pytest.mark.parametrize("name", ["tiny_f32_b3", "small_bf16_llama"])
def test_runtime_block_size_schedule(name):
    # a session configured at its drafter's block runs rounds at smaller blocks
    # (16 -> 8 -> 1 -> 12 -> 16 ...; the tiny drafter's 4 -> 2 -> 1 -> 3), sequences ragged
    B = configs.get(name).block_size
    sched = [B, B // 2, 1, 3 * B // 4]
    assert run_stepwise(name, rounds=5, schedule=sched) >= 3 * 5 // 2


def test_runtime_block_size_errors():
    from block_diffusion_speculative_ctx_gb300 import DFlashError
    w = configs.get("tiny_f32")
    with _session(w, max_seq_len=96) as sess:
        with pytest.raises(DFlashError, match="outside"):
            sess.set_block_size(w.block_size + 1)
        with pytest.raises(DFlashError, match="outside"):
            sess.set_block_size(0)
        sess.set_block_size(2)                            # before a prefill
        sess.prefill(synth.prompts(w))
        d = sess.draft_block()
        assert d.shape == (1, 1)
        with pytest.raises(DFlashError, match="between draft_block and verify"):
            sess.set_block_size(3)
        sess.verify(d)
        sess.set_block_size(w.block_size)
        assert sess.draft_block().shape == (1, w.block_size - 1)


def test_block_size_one_is_plain_greedy():
    assert run_stepwise("tiny_f32_b3", rounds=5, block_size=1) == 3 * 5


def test_tiny_f32_generate_equals_oracle_greedy():
    """The full loop through dflash_generate reproduces the oracle's plain
    greedy decode token for token (losslessness on the GPU path)."""
    w = configs.get("tiny_f32")
    m = om.Model(w)
    p = synth.prompts(w)[0]
    ar, _ = spec.ar_generate(m, p, w.max_new_tokens)
    sess = _session(w)
    try:
        out, st = sess.generate([p], w.max_new_tokens)
        np.testing.assert_array_equal(out[0], ar)
        assert st.tokens >= w.max_new_tokens and st.rounds >= 1
        assert st.kernel_launches > 0
    finally:
        sess.close()


def test_ragged_generate_equals_oracle_greedy():
    w = configs.get("tiny_f32_b3")
    m = om.Model(w)
    ps = synth.prompts(w)
    sess = _session(w)
    try:
        out, st = sess.generate(ps, w.max_new_tokens)
        for s, p in enumerate(ps):
            ar, _ = spec.ar_generate(m, p, w.max_new_tokens)
            np.testing.assert_array_equal(out[s], ar)
    finally:
        sess.close()


def test_bf16_hidden_rel_l2_against_pure_fp64():
    """Final residual and logits of a verify block against the oracle without
    any bf16 rounding of activations (plain fp64 on the bf16 weights).  The
    proposal is a fixed synthetic token block, the same on both sides."""
    w = configs.get("small_bf16")
    m = om.Model(w, act_round=False)
    prompts = synth.prompts(w)
    proposal = synth.uniform_ints(123, 0x51, len(prompts) * (w.block_size - 1), w.vocab).reshape(len(prompts), -1)
    sess = _session(w, keep_logits=True)
    try:
        first = sess.prefill(prompts)
        sess.draft_block()
        sess.verify(proposal.astype(np.int32))
        hid = sess.hidden_verify()
        vlog = sess.logits("verify")
        checked = 0
        for s, p in enumerate(prompts):
            st = spec.prefill(m, p)
            if first[s] != st.anchor:
                # the GPU's first token sits at a near-tie of the oracle's logits
                assert spec.top2_margin(st.first_logits[None])[0] < BF16_MARGIN
                continue
            block = np.concatenate([[st.anchor], proposal[s]])
            x = _final_residual(m, p, block)
            lg = m.logits(x, "final_norm")
            assert _rel_l2(hid[s], x) <= BF16_HIDDEN_REL
            assert np.abs(vlog[s] - lg).max() <= BF16_LOGIT_TOL
            checked += 1
        assert checked >= 1
    finally:
        sess.close()


def _final_residual(m, prompt, block):
    """Oracle residual after the last target layer for `block` appended to `prompt`."""
    c = m.cfg
    cache = m.new_target_cache()
    m.target_forward(prompt, cache)
    tokens = np.asarray(block, dtype=np.int64)
    n0, n = cache.length, len(tokens)
    pos = np.arange(n0, n0 + n)
    x = m.w("embed")[tokens].copy()
    for l in range(c.target_layers):
        p = f"t{l}"
        q, k, v = m._qkv(p, x, pos, c.target_qk_norm)
        cache.append(l, k, v)
        visible = np.arange(n0 + n)[None, :] <= pos[:, None]
        x = m._attn_out_mlp(p, x, om.attention(q, cache.k[l], cache.v[l], visible))
    return x


@pytest.mark.parametrize("name", ["small_bf16_llama", "small_bf16_b20"])
def test_graph_replay_matches_eager_launches(name):
    """Rounds replayed from captured CUDA graphs give bit-identical results to
    the same rounds launched kernel by kernel (at batch 20 through the persistent
    stream-K GEMM, whose split tiles are summed in a fixed order)."""
    w = configs.get(name)
    prompts = synth.prompts(w)
    b, B = len(prompts), w.block_size
    props = [synth.uniform_ints(500 + r, 0x33, b * (B - 1), w.vocab).reshape(b, B - 1).astype(np.int32)
             for r in range(5)]
    # plant a few accepted drafts too: reuse the previous round's posterior as the next proposal head
    outs = []
    for graphs in (False, True):
        sess = _session(w, keep_logits=True, graphs=graphs)
        try:
            rec = [sess.prefill(prompts)]
            for r in range(5):
                d = sess.draft_block()
                acc, bon = sess.verify(props[r])
                rec += [d.copy(), acc.copy(), bon.copy(), sess.logits("verify").copy(), sess.lengths().copy()]
            outs.append(rec)
        finally:
            sess.close()
    for a, b_ in zip(*outs):
        np.testing.assert_array_equal(a, b_)


# ------------------------------------------------------------------ errors
def test_state_and_capacity_errors():
    import block_diffusion_speculative_ctx_gb300 as dfl
    w = configs.get("tiny_f32")
    sess = _session(w, max_seq_len=48)
    try:
        with pytest.raises(dfl.DFlashError) as e:
            sess.batch = 1
            sess.draft_block()
        assert e.value.status == dfl.DFLASH_E_STATE
        p = synth.prompts(w)[0]
        sess.prefill([p])
        with pytest.raises(dfl.DFlashError) as e:
            sess.verify(np.zeros((1, 3), np.int32))
        assert e.value.status == dfl.DFLASH_E_STATE
        sess.draft_block()
        with pytest.raises(dfl.DFlashError) as e:
            sess.verify(np.full((1, 3), w.vocab, np.int32))
        assert e.value.status == dfl.DFLASH_E_INVAL
        # after the rejected call the drafted state is intact
        sess.verify(np.zeros((1, 3), np.int32))
        # fill to capacity: 32 + rounds * (a+1) <= 48 - B
        with pytest.raises(dfl.DFlashError) as e:
            for _ in range(20):
                sess.draft_block()
                sess.verify(np.zeros((1, 3), np.int32))
        assert e.value.status == dfl.DFLASH_E_CAPACITY
    finally:
        sess.close()


def test_device_token_check_reports_without_faulting():
    import torch
    import block_diffusion_speculative_ctx_gb300 as dfl
    w = configs.get("tiny_f32")
    sess = _session(w)
    try:
        sess.prefill([synth.prompts(w)[0]])
        sess.draft_block()
        bad = torch.full((1, 3), w.vocab + 5, dtype=torch.int32, device="cuda")
        with pytest.raises(dfl.DFlashError) as e:
            sess.verify(bad, np.zeros(1, np.int32), np.zeros(1, np.int32))
        assert e.value.status == dfl.DFLASH_E_DEVICE_CHECK
        # the context is still usable
        sess.draft_block()
        sess.verify(np.zeros((1, 3), np.int32))
    finally:
        sess.close()
