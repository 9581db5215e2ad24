"""The drafter's training forward on the GPU (dflash_train_forward) against the
fp64 oracle's eq. 12 loss ("DFlash: Why a Diffusion Drafter Can Accelerate an
Autoregressive Model" §6, Algorithm 2) on the same seeded model, sequence and
anchors (overlapping blocks included).  fp32: relative 1e-5; bf16: relative
2e-2 (bf16 storage; the loss averages per-position cross-entropies whose
logits carry the 5e-2 bf16 tolerance)."""
import numpy as np
import pytest

import synth
from synth import configs
from oracle import model as om, training as tr

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_speculative_ctx_gb300 import build
    build.build()


@pytest.mark.parametrize("name,anchors,rel", [
    ("tiny_f32", [1, 5, 6, 17, 28], 1e-5),            # B = 4, 32 tokens
    ("small_bf16", [1, 4, 9, 16, 21], 2e-2),          # B = 16, 37 tokens, head_dim 128
])
def test_train_forward_matches_the_oracle(name, anchors, rel):
    from block_diffusion_speculative_ctx_gb300 import Session
    w = configs.get(name)
    x = np.asarray(synth.prompts(w)[0], dtype=np.int64)
    lam = 3.0
    want = tr.training_loss(om.Model(w), x, anchors, lam)
    with Session(w, max_batch=len(anchors) + 1, max_seq_len=len(x) + 2 * w.block_size) as sess:
        got = sess.train_forward(x, anchors, lam)
        assert abs(got - want) <= rel * abs(want), (got, want)
        # the session is usable again after a prefill
        sess.prefill([x[:10]])
        sess.verify(sess.draft_block())


def test_train_forward_argument_checks():
    from block_diffusion_speculative_ctx_gb300 import Session, DFlashError
    w = configs.get("tiny_f32")
    x = np.asarray(synth.prompts(w)[0], dtype=np.int64)
    with Session(w, max_batch=3, max_seq_len=64) as sess:
        with pytest.raises(DFlashError, match="anchor"):
            sess.train_forward(x, [0], 3.0)
        with pytest.raises(DFlashError, match="anchor"):
            sess.train_forward(x, [len(x) - w.block_size + 1], 3.0)
        with pytest.raises(DFlashError, match="max_batch"):
            sess.train_forward(x, [1, 2, 3], 3.0)
        with pytest.raises(DFlashError, match="lambda"):
            sess.train_forward(x, [1], 0.0)
