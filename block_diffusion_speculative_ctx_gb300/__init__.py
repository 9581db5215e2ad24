"""Python binding of the dflash C ABI (include/dflash.h).

Argument marshalling only: every step of the round runs in the CUDA library
``_build/libdflash.so``.  PyTorch supplies device memory (the library's
allocator callbacks go to torch's caching allocator) and the CUDA stream.
There is no fallback: if the library is missing or no GPU is present, the
calls raise.

The functions carry the C names:

    dflash_init, dflash_prefill, dflash_set_block_size, dflash_block_size, dflash_set_sampling_filter,
    dflash_draft_block, dflash_verify,
    dflash_draft_block_sampled, dflash_verify_sampled, dflash_train_forward,
    dflash_generate, dflash_inspect, dflash_destroy, dflash_last_error

``Session`` wraps them for tests and the benchmark.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build_mod

HERE = os.path.dirname(os.path.abspath(__file__))

# ----------------------------------------------------------------- ABI types
DFLASH_OK, DFLASH_E_INVAL, DFLASH_E_NOMEM, DFLASH_E_CUDA, DFLASH_E_STATE, DFLASH_E_CAPACITY, \
    DFLASH_E_TIMEOUT, DFLASH_E_DEVICE_CHECK = range(8)
STATUS_NAMES = {0: "OK", 1: "E_INVAL", 2: "E_NOMEM", 3: "E_CUDA", 4: "E_STATE", 5: "E_CAPACITY", 6: "E_TIMEOUT",
                7: "E_DEVICE_CHECK"}
DFLASH_DTYPE_F32, DFLASH_DTYPE_BF16 = 0, 1
DFLASH_FLAG_KEEP_LOGITS = 1
DFLASH_FLAG_PROFILE = 2
DFLASH_FLAG_NO_GRAPHS = 4
KERNEL_CLASSES = ("gemm_qkv", "gemm_o", "gemm_gate_up", "gemm_down", "gemm_head", "gemm_fc", "gemm_ctx_kv",
                  "attention", "norm", "rope_store", "swiglu", "argmax", "other", "sampling")
DFLASH_MAX_CTX_LAYERS = 16
(INSPECT_LENGTHS, INSPECT_ANCHORS, INSPECT_POSTERIOR, INSPECT_TARGET_K, INSPECT_TARGET_V, INSPECT_DRAFT_K,
 INSPECT_DRAFT_V, INSPECT_LOGITS_PREFILL, INSPECT_LOGITS_DRAFT, INSPECT_LOGITS_VERIFY, INSPECT_STATS,
 INSPECT_HIDDEN_VERIFY, INSPECT_PROFILE, INSPECT_PROFILE_RESET) = range(1, 15)

ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p)
FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p)


class dflash_config(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("vocab", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("ffn", ctypes.c_int32), ("target_layers", ctypes.c_int32), ("target_qk_norm", ctypes.c_int32),
                ("draft_layers", ctypes.c_int32), ("block_size", ctypes.c_int32), ("n_ctx_layers", ctypes.c_int32),
                ("ctx_layer_ids", ctypes.c_int32 * DFLASH_MAX_CTX_LAYERS), ("mask_token", ctypes.c_int32),
                ("max_batch", ctypes.c_int32), ("max_seq_len", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_double), ("alloc", ALLOC_FN),
                ("free", FREE_FN), ("alloc_user", ctypes.c_void_p), ("kv_pool_tokens", ctypes.c_int64)]


class dflash_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "attn_norm", "mlp_norm", "q_norm", "k_norm")]


class dflash_weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("head", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("target", ctypes.POINTER(dflash_layer_weights)), ("fc", ctypes.c_void_p),
                ("fc_norm", ctypes.c_void_p), ("draft", ctypes.POINTER(dflash_layer_weights)),
                ("draft_norm", ctypes.c_void_p)]


class dflash_stats(ctypes.Structure):
    _fields_ = [("rounds", ctypes.c_int64), ("tokens", ctypes.c_int64), ("accepted", ctypes.c_int64),
                ("prefill_ms", ctypes.c_double), ("draft_ms", ctypes.c_double), ("verify_ms", ctypes.c_double),
                ("kernel_launches", ctypes.c_int64)]


class dflash_profile_entry(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64), ("ms", ctypes.c_double), ("bytes", ctypes.c_double),
                ("flops", ctypes.c_double)]


EXPORTS = ("dflash_init", "dflash_prefill", "dflash_set_block_size", "dflash_block_size", "dflash_draft_block", "dflash_verify", "dflash_draft_block_sampled",
           "dflash_verify_sampled", "dflash_set_sampling_filter", "dflash_train_forward", "dflash_generate",
           "dflash_inspect", "dflash_set_profiling", "dflash_destroy", "dflash_last_error")

_lib = None


def library_path() -> str:
    return _build_mod.LIB


def load(build_if_missing: bool = False):
    """Load libdflash.so.  Raises if it is missing (no silent fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build_mod.LIB):
        if not build_if_missing:
            raise RuntimeError(f"dflash CUDA library not built ({_build_mod.LIB}); run __graft_entry__.build()")
        _build_mod.build()
    lib = ctypes.CDLL(_build_mod.LIB)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.dflash_init.argtypes = [ctypes.POINTER(dflash_config), ctypes.POINTER(dflash_weights), P,
                                ctypes.POINTER(P)]
    lib.dflash_prefill.argtypes = [P, I32, P, P, P]
    lib.dflash_draft_block.argtypes = [P, P]
    lib.dflash_verify.argtypes = [P, P, P, P]
    lib.dflash_draft_block_sampled.argtypes = [P, ctypes.c_float, P, P]
    lib.dflash_verify_sampled.argtypes = [P, ctypes.c_float, P, P, P, P]
    lib.dflash_train_forward.argtypes = [P, I32, P, I32, P, ctypes.c_float, P]
    lib.dflash_generate.argtypes = [P, I32, P, P, I32, P, P, ctypes.POINTER(dflash_stats)]
    lib.dflash_inspect.argtypes = [P, I32, I32, I32, P, SZ, ctypes.POINTER(SZ)]
    lib.dflash_set_profiling.argtypes = [P, I32]
    lib.dflash_set_block_size.argtypes = [P, I32]
    lib.dflash_set_sampling_filter.argtypes = [P, I32, ctypes.c_float]
    lib.dflash_block_size.argtypes = [P]
    lib.dflash_block_size.restype = I32
    lib.dflash_destroy.argtypes = [P]
    lib.dflash_last_error.argtypes = [P]
    lib.dflash_last_error.restype = ctypes.c_char_p
    for f in ("dflash_init", "dflash_prefill", "dflash_draft_block", "dflash_verify", "dflash_draft_block_sampled",
              "dflash_verify_sampled", "dflash_set_sampling_filter", "dflash_train_forward", "dflash_generate",
              "dflash_inspect", "dflash_set_profiling", "dflash_set_block_size"):
        getattr(lib, f).restype = ctypes.c_int
    lib.dflash_destroy.restype = None
    _lib = lib
    return lib


class DFlashError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _ptr(x) -> Optional[int]:
    """Address of a numpy array or torch tensor (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


# ------------------------------------------------------------- thin wrappers
def dflash_last_error(ctx) -> str:
    s = load().dflash_last_error(ctx)
    return s.decode() if s else ""


def _check(ctx, status: int):
    if status != DFLASH_OK:
        raise DFlashError(status, dflash_last_error(ctx))


def dflash_init(cfg: dflash_config, weights: dflash_weights, stream: int):
    ctx = ctypes.c_void_p()
    st = load().dflash_init(ctypes.byref(cfg), ctypes.byref(weights), ctypes.c_void_p(stream), ctypes.byref(ctx))
    if st != DFLASH_OK:
        raise DFlashError(st, dflash_last_error(None))
    return ctx


def dflash_prefill(ctx, prompt_lens: np.ndarray, prompt_tokens: np.ndarray, first_tokens: np.ndarray) -> int:
    return load().dflash_prefill(ctx, len(prompt_lens), _ptr(prompt_lens), _ptr(prompt_tokens), _ptr(first_tokens))


def dflash_draft_block(ctx, draft_tokens) -> int:
    return load().dflash_draft_block(ctx, _ptr(draft_tokens))


def dflash_verify(ctx, draft_tokens, accepted, bonus) -> int:
    return load().dflash_verify(ctx, _ptr(draft_tokens), _ptr(accepted), _ptr(bonus))


def dflash_draft_block_sampled(ctx, temperature, u_draft, draft_tokens) -> int:
    return load().dflash_draft_block_sampled(ctx, float(temperature), _ptr(u_draft), _ptr(draft_tokens))


def dflash_verify_sampled(ctx, temperature, draft_tokens, u_verify, accepted, emitted) -> int:
    return load().dflash_verify_sampled(ctx, float(temperature), _ptr(draft_tokens), _ptr(u_verify), _ptr(accepted),
                                        _ptr(emitted))


def dflash_generate(ctx, prompt_lens, prompt_tokens, max_new_tokens, out_tokens, out_lens, stats=None) -> int:
    return load().dflash_generate(ctx, len(prompt_lens), _ptr(prompt_lens), _ptr(prompt_tokens), max_new_tokens,
                                  _ptr(out_tokens), _ptr(out_lens), ctypes.byref(stats) if stats is not None else None)


def dflash_inspect(ctx, what: int, seq: int, layer: int, dst: np.ndarray) -> int:
    written = ctypes.c_size_t(0)
    st = load().dflash_inspect(ctx, what, seq, layer, _ptr(dst), dst.nbytes, ctypes.byref(written))
    return st


def dflash_set_profiling(ctx, on: bool) -> int:
    return load().dflash_set_profiling(ctx, 1 if on else 0)


def dflash_destroy(ctx):
    load().dflash_destroy(ctx)


from .session import Session, config_from_workload  # noqa: E402,F401
