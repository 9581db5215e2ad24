"""dflash_head_argmax_noalloc: the shared-head argmax for callers that cannot
allocate device memory (its intermediates live in a fixed device array inside
the library).  Its token ids must agree with the posterior that dflash_verify
computes from the same final hidden states, on consecutive calls, and with
the CPU oracle's head on seeded hidden states.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import synth
from synth import configs

pytestmark = pytest.mark.gpu

# near-tie exemption: a token may differ only where the two largest logits are closer
# than the logit tolerance of the precision (bf16: 5e-2; fp32: tokens exact, with a 1e-4
# guard far below any difference the fp32 kernels produce)
MARGIN = {"bf16": 5e-2, "f32": 1e-4}


def _lib():
    from block_diffusion_speculative_ctx_gb300 import build, load
    build.build()
    lib = load()
    f = lib.dflash_head_argmax_noalloc
    f.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return lib


def _top2(lg):
    part = np.partition(lg, -2, axis=-1)
    return part[..., -1] - part[..., -2]


def _agree(got, want, margin, tol):
    ok = (got == want) | (margin < tol)
    return bool(ok.all()), np.flatnonzero(~ok)


@pytest.mark.parametrize("name", ["small_bf16", "tiny_f32_b3"])
def test_noalloc_head_equals_verify_posterior_on_consecutive_calls(name):
    import torch
    from block_diffusion_speculative_ctx_gb300 import DFLASH_DTYPE_BF16, DFLASH_DTYPE_F32, Session
    from block_diffusion_speculative_ctx_gb300.session import upload_weights

    lib = _lib()
    w = configs.get(name)
    tens = upload_weights(w)
    prompts = synth.prompts(w)
    b, B, d, V = len(prompts), w.block_size, w.d_model, w.vocab
    dtype = DFLASH_DTYPE_BF16 if w.dtype == "bf16" else DFLASH_DTYPE_F32
    stream = torch.cuda.current_stream()
    sess = Session(w, keep_logits=True, tensors=tens)
    try:
        sess.prefill(prompts)
        for call in range(2):
            sess.draft_block()
            proposal = synth.uniform_ints(77 + call, 0x7A, b * (B - 1), V).reshape(b, B - 1).astype(np.int32)
            sess.verify(proposal)
            want = sess.posterior().reshape(-1)          # argmax ids from the existing verify path
            margin = _top2(sess.logits("verify").reshape(b * B, V))
            hid = sess.hidden_verify().reshape(b * B, d)
            x = torch.from_numpy(np.ascontiguousarray(hid)).cuda()
            out = torch.full((b * B,), -2, dtype=torch.int32, device="cuda")
            st = lib.dflash_head_argmax_noalloc(dtype, x.data_ptr(), tens["final_norm"].data_ptr(), w.rms_eps,
                                                tens["head"].data_ptr(), b * B, d, V, out.data_ptr(),
                                                stream.cuda_stream)
            assert st == 0, lib.dflash_last_error(None)
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            assert got.min() >= 0, "the call reported a device-side timeout (-1 ids) or wrote nothing"
            ok, bad = _agree(got, want, margin, MARGIN[w.dtype])
            assert ok, (call, bad, got[bad], want[bad])
    finally:
        sess.close()


@pytest.mark.parametrize("name,rows", [("small_bf16", 24), ("tiny_f32_b3", 40)])
def test_noalloc_head_equals_the_oracle_head_on_seeded_hidden_states(name, rows):
    """Hidden states drawn from the seeded generator (unit normal, the scale of a final
    residual); the oracle's head (RMSNorm with the final scale, bf16 rounding of the
    normalised rows for bf16, then the head, in fp64) decides the expected ids."""
    import torch
    from oracle import model as om
    from block_diffusion_speculative_ctx_gb300 import DFLASH_DTYPE_BF16, DFLASH_DTYPE_F32
    from block_diffusion_speculative_ctx_gb300.session import upload_weights

    lib = _lib()
    w = configs.get(name)
    tens = upload_weights(w)
    d, V = w.d_model, w.vocab
    dtype = DFLASH_DTYPE_BF16 if w.dtype == "bf16" else DFLASH_DTYPE_F32
    m = om.Model(w)
    for call in range(2):
        x = synth.normal_f32(91 + call, 0x4E, rows * d).reshape(rows, d)
        lg = m.logits(x.astype(np.float64), "final_norm")
        want = om.argmax_lowest(lg)
        xd = torch.from_numpy(x).cuda()
        out = torch.full((rows,), -2, dtype=torch.int32, device="cuda")
        st = lib.dflash_head_argmax_noalloc(dtype, xd.data_ptr(), tens["final_norm"].data_ptr(), w.rms_eps,
                                            tens["head"].data_ptr(), rows, d, V, out.data_ptr(), None)
        assert st == 0, lib.dflash_last_error(None)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        ok, bad = _agree(got, want, _top2(lg), MARGIN[w.dtype])
        assert ok, (call, bad, got[bad], want[bad])


def test_noalloc_rejects_requests_above_the_fixed_scratch():
    import torch
    from block_diffusion_speculative_ctx_gb300 import DFLASH_DTYPE_BF16, DFLASH_E_INVAL

    lib = _lib()
    x = torch.zeros((1, 64), dtype=torch.float32, device="cuda")
    w = torch.ones(64, dtype=torch.float32, device="cuda")
    head = torch.zeros((8, 64), dtype=torch.int16, device="cuda")
    out = torch.zeros(64, dtype=torch.int32, device="cuda")
    # 64 rows x 151936 vocab x 4 bytes of logits is far above 16 MiB
    st = lib.dflash_head_argmax_noalloc(DFLASH_DTYPE_BF16, x.data_ptr(), w.data_ptr(), 1e-6, head.data_ptr(), 64, 64,
                                        151936, out.data_ptr(), None)
    assert st == DFLASH_E_INVAL
    assert b"maximum" in lib.dflash_last_error(None)
    st = lib.dflash_head_argmax_noalloc(DFLASH_DTYPE_BF16, None, w.data_ptr(), 1e-6, head.data_ptr(), 1, 64, 8,
                                        out.data_ptr(), None)
    assert st == DFLASH_E_INVAL
    # a head that is not 16-byte aligned is refused before anything is queued
    st = lib.dflash_head_argmax_noalloc(DFLASH_DTYPE_BF16, x.data_ptr(), w.data_ptr(), 1e-6, head.data_ptr() + 2, 1,
                                        64, 8, out.data_ptr(), None)
    assert st == DFLASH_E_INVAL
    assert b"aligned" in lib.dflash_last_error(None)
