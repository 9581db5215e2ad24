"""Seeded synthetic inputs shared by the CPU oracle and the CUDA library.

Nothing here computes any step of the decoding method.  The module maps
(seed, stream, index) to numbers with the Philox4x32-10 counter-based
generator (Salmon et al., SC'11) and lays those numbers out as the named
tensors of a workload (``synth.configs``).  A small C library does the bulk
work in parallel; ``philox4x32_10_np`` is an independent numpy statement of
the same generator used to cross-check it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import configs

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the generator with gcc (-fopenmp); returns the library path."""
    src = os.path.join(_HERE, "synth_gen.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, u32, p = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p
            lib.synth_philox4x32_10.argtypes = [p, p, p]
            lib.synth_normal_f32.argtypes = [u64, u32, u64, ctypes.c_double, ctypes.c_double, p]
            lib.synth_uniform_i32.argtypes = [u64, u32, u64, u32, p]
            lib.synth_f32_to_bf16.argtypes = [p, p, u64]
            lib.synth_bf16_to_f32.argtypes = [p, p, u64]
            for f in (lib.synth_philox4x32_10, lib.synth_normal_f32, lib.synth_uniform_i32,
                      lib.synth_f32_to_bf16, lib.synth_bf16_to_f32):
                f.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


# ---------------------------------------------------------------- primitives
def philox4x32_10(ctr, key) -> np.ndarray:
    """One Philox4x32-10 block from the C library."""
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, np.uint32)
    _load().synth_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def philox4x32_10_np(ctr: np.ndarray, key) -> np.ndarray:
    """Vectorised numpy Philox4x32-10 over counters ``ctr`` of shape [n, 4]."""
    c = np.array(ctr, dtype=np.uint64).reshape(-1, 4) & 0xFFFFFFFF
    k0, k1 = np.uint64(key[0]), np.uint64(key[1])
    m0, m1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)
    mask = np.uint64(0xFFFFFFFF)
    for r in range(10):
        if r:
            k0 = (k0 + np.uint64(0x9E3779B9)) & mask
            k1 = (k1 + np.uint64(0xBB67AE85)) & mask
        p0 = c[:, 0] * m0
        p1 = c[:, 2] * m1
        c = np.stack([((p1 >> np.uint64(32)) ^ c[:, 1] ^ k0) & mask, p1 & mask,
                      ((p0 >> np.uint64(32)) ^ c[:, 3] ^ k1) & mask, p0 & mask], axis=1)
    return c.astype(np.uint32)


def normal_f32(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    out = np.empty(int(n), np.float32)
    if n:
        _load().synth_normal_f32(seed, stream, n, mean, std, _ptr(out))
    return out


def uniform_ints(seed: int, stream: int, n: int, high: int) -> np.ndarray:
    out = np.empty(int(n), np.int32)
    if n:
        _load().synth_uniform_i32(seed, stream, n, high, _ptr(out))
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().synth_f32_to_bf16(_ptr(x), _ptr(out), x.size)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    out = np.empty(b.shape, np.float32)
    _load().synth_bf16_to_f32(_ptr(b), _ptr(out), b.size)
    return out


# ------------------------------------------------------------- tensor layout
LAYER_MATS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def weight_specs(cfg: configs.Workload) -> list:
    """Ordered (name, shape, kind) list; a tensor's Philox stream is its index + 1.

    Matrices are stored [out_features, in_features] (y = W x).  ``kind`` is
    "matrix" (N(0, weight_std), held in the workload dtype) or "norm"
    (fp32 scale vector)."""
    d, f, hd = cfg.d_model, cfg.ffn, cfg.head_dim
    qd, kvd = cfg.q_dim, cfg.kv_dim
    shapes = {"wq": (qd, d), "wk": (kvd, d), "wv": (kvd, d), "wo": (d, qd),
              "w_gate": (f, d), "w_up": (f, d), "w_down": (d, f)}
    specs = [("embed", (cfg.vocab, d), "matrix")]

    def layer(prefix, qk_norm):
        for m in LAYER_MATS:
            specs.append((f"{prefix}.{m}", shapes[m], "matrix"))
        specs.append((f"{prefix}.attn_norm", (d,), "norm"))
        specs.append((f"{prefix}.mlp_norm", (d,), "norm"))
        if qk_norm:
            specs.append((f"{prefix}.q_norm", (hd,), "norm"))
            specs.append((f"{prefix}.k_norm", (hd,), "norm"))

    for l in range(cfg.target_layers):
        layer(f"t{l}", cfg.target_qk_norm)
    specs.append(("final_norm", (d,), "norm"))
    specs.append(("head", (cfg.vocab, d), "matrix"))
    specs.append(("fc", (d, cfg.n_ctx_layers * d), "matrix"))
    specs.append(("fc_norm", (d,), "norm"))
    for l in range(cfg.draft_layers):
        layer(f"d{l}", True)
    specs.append(("draft_norm", (d,), "norm"))
    return specs


def _spec_index(cfg):
    return {name: (i, shape, kind) for i, (name, shape, kind) in enumerate(weight_specs(cfg))}


def weight_f32(cfg: configs.Workload, name: str) -> np.ndarray:
    """The tensor as float32 values.  For bf16 workloads matrices are rounded to
    bf16 (round to nearest even) and widened back, so the values are exactly
    those a bf16 buffer holds."""
    i, shape, kind = _spec_index(cfg)[name]
    n = int(np.prod(shape))
    if kind == "norm":
        if cfg.norm_std == 0.0:
            return np.ones(shape, np.float32)
        return normal_f32(cfg.weight_seed, i + 1, n, 1.0, cfg.norm_std).reshape(shape)
    x = normal_f32(cfg.weight_seed, i + 1, n, 0.0, cfg.weight_std).reshape(shape)
    if cfg.dtype == "bf16":
        x = bf16_bits_to_f32(f32_to_bf16_bits(x))
    return x


def weight_bits(cfg: configs.Workload, name: str) -> np.ndarray:
    """The tensor as stored on the device: uint16 bf16 bits for bf16 matrices,
    float32 otherwise (norm scales are always float32)."""
    i, shape, kind = _spec_index(cfg)[name]
    if kind == "matrix" and cfg.dtype == "bf16":
        n = int(np.prod(shape))
        return f32_to_bf16_bits(normal_f32(cfg.weight_seed, i + 1, n, 0.0, cfg.weight_std)).reshape(shape)
    return weight_f32(cfg, name)


def prompts(cfg: configs.Workload) -> list:
    """One int32 array of uniform token ids in [0, vocab) per sequence."""
    return [uniform_ints(cfg.prompt_seed, 0x70000000 + s, n, cfg.vocab) for s, n in enumerate(cfg.prompt_lens)]


__all__ = ["configs", "weight_specs", "weight_f32", "weight_bits", "prompts", "normal_f32", "uniform_ints",
           "f32_to_bf16_bits", "bf16_bits_to_f32", "philox4x32_10", "philox4x32_10_np", "build"]
