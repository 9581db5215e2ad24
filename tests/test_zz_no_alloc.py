"""dflash_head_argmax_noalloc: the shared-head argmax for callers that cannot
allocate device memory (its intermediates live in a fixed device array inside
the library).  Its token ids must equal the posterior that dflash_verify
computes from the same final hidden states, on consecutive calls.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import synth
from synth import configs

pytestmark = pytest.mark.gpu


def _lib():
    from block_diffusion_speculative_ctx_gb300 import build, load
    build.build()
    lib = load()
    f = lib.dflash_head_argmax_noalloc
    f.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return lib


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
            want = sess.posterior()                      # argmax ids from the existing verify path
            hid = sess.hidden_verify().reshape(b * B, d)
            x = torch.from_numpy(np.ascontiguousarray(hid)).cuda()
            out = torch.full((b * B,), -1, dtype=torch.int32, device="cuda")
            st = lib.dflash_head_argmax_noalloc(dtype, x.data_ptr(), tens["final_norm"].data_ptr(), w.rms_eps,
                                                tens["head"].data_ptr(), b * B, d, V, out.data_ptr(),
                                                stream.cuda_stream)
            assert st == 0, lib.dflash_last_error(None)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(out.cpu().numpy().reshape(b, B), want)
    finally:
        sess.close()


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
