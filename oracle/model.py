"""Plain fp64 CPU statement of the target decoder and the block drafter.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import this package.  It shares no
code with the CUDA library; its inputs come from ``synth`` alone.

Sources (page titles; sections and equations as printed on them):

* [digest]  "DFlash: Block Diffusion for Flash Speculative Decoding" (paper digest
  with a "Paper vs code" section on the authors' model.py).
* [review]  "DFlash: Why a Diffusion Drafter Can Accelerate an Autoregressive Model"
  (technical review of the v2 paper).

What the pages fix, and how this file reads them:

* Context feature: hidden states of a fixed set of target layers, concatenated,
  one linear map, then RMS normalisation ([digest] Method, Inference step 1;
  [review] §5.1 eq. 9).
* KV injection: in every draft layer the context feature is projected by that
  layer's key and value maps; queries come from the block only; the context
  rows skip the query/output maps, the attention update and the MLP
  ([digest] Inference step 2 and the draft-layer pseudocode; [review] §5.1 eq. 10).
  The authors' code adds per-head RMS normalisation of q and k and rotary
  position encoding of context keys at their tokens' absolute positions
  ([digest] Paper vs code, "KV injection matches, with extras").
* The block is the anchor plus B-1 mask tokens embedded with the target's
  table; full-attention draft layers are non-causal ([digest] Inference step 3,
  Paper vs code "Attention pattern").
* Drafted tokens are the argmax of the target head on the B-1 mask rows; the
  anchor row is dropped ([digest] Paper vs code "Drafted tokens match").

Readings where the pages are silent (each is listed in the design notes):

* "Hidden state of layer l" is the residual stream after decoder layer l
  (0-based), before any final norm; the code's hidden_states[l+1] offset.
* Decoder form: pre-RMSNorm, GQA softmax attention with scale 1/sqrt(head_dim),
  SwiGLU MLP, no biases, untied head after a final RMSNorm.  Target QK-norm only
  where the workload says so; the drafter always has q/k norm.
* Context keys get k-norm and RoPE; no extra input norm on the context feature.
* RoPE is the half-split form with inv_freq_j = theta^(-2j/head_dim), angles in
  double precision; positions are absolute token positions.
* The drafter has its own final RMSNorm before the shared head.
* Argmax ties go to the lowest token id.

Numerics: every step is fp64.  With ``act_round=True`` (bf16 workloads) the
values that a bf16 model stores are rounded to bf16 at the points where they
are stored: linear-map inputs (norm outputs, attention output, SiLU product,
captured hidden states, context feature), and q/k/v after norm and RoPE.  The
rounding goes through float32 first, as an fp32 accumulator would.
"""
from __future__ import annotations

import math
from typing import Callable, Optional

import numpy as np


# ---------------------------------------------------------------- primitives
def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * w over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotary encoding of x [n, heads, hd] at integer positions pos [n].

    Pair (j, j + hd/2) is rotated by the angle pos * theta^(-2j/hd)."""
    hd = x.shape[-1]
    half = hd // 2
    j = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * j / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, visible: np.ndarray) -> np.ndarray:
    """Softmax attention with grouped KV heads.

    q [nq, H, hd]; k, v [nk, Hkv, hd]; visible [nq, nk] bool.  Query head h
    reads KV head h // (H / Hkv).  Returns [nq, H, hd]."""
    nq, H, hd = q.shape
    Hkv = k.shape[1]
    g = H // Hkv
    out = np.empty_like(q)
    scale = 1.0 / math.sqrt(hd)
    for h in range(H):
        kh = h // g
        s = (q[:, h, :] @ k[:, kh, :].T) * scale
        s = np.where(visible, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, kh, :]
    return out


def argmax_lowest(logits: np.ndarray) -> np.ndarray:
    """Row argmax; np.argmax returns the first (lowest) index among equal maxima."""
    return np.argmax(logits, axis=-1).astype(np.int64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to bfloat16 (nearest even) through float32; returns float64."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


# ------------------------------------------------------------------- weights
class Weights:
    """Named fp64 tensors from a provider ``get(name) -> array``; cached."""

    def __init__(self, get: Callable[[str], np.ndarray], cache: bool = True):
        self._get = get
        self._cache = {} if cache else None

    def __call__(self, name: str) -> np.ndarray:
        if self._cache is not None and name in self._cache:
            return self._cache[name]
        w = np.asarray(self._get(name), dtype=np.float64)
        if self._cache is not None:
            self._cache[name] = w
        return w


def synth_weights(cfg, cache: bool = True) -> Weights:
    import synth
    return Weights(lambda name: synth.weight_f32(cfg, name), cache=cache)


# --------------------------------------------------------------------- model
class KV:
    """Per-layer key/value history of one sequence: rows are positions 0..n-1."""

    def __init__(self, n_layers: int, n_kv: int, hd: int):
        self.k = [np.zeros((0, n_kv, hd)) for _ in range(n_layers)]
        self.v = [np.zeros((0, n_kv, hd)) for _ in range(n_layers)]

    @property
    def length(self) -> int:
        return self.k[0].shape[0]

    def append(self, layer: int, k: np.ndarray, v: np.ndarray):
        self.k[layer] = np.concatenate([self.k[layer], k], axis=0)
        self.v[layer] = np.concatenate([self.v[layer], v], axis=0)

    def truncate(self, n: int):
        self.k = [k[:n] for k in self.k]
        self.v = [v[:n] for v in self.v]

    def copy(self) -> "KV":
        c = KV.__new__(KV)
        c.k = [k.copy() for k in self.k]
        c.v = [v.copy() for v in self.v]
        return c


class Model:
    """Target decoder plus block drafter of one workload (``synth.configs``)."""

    def __init__(self, cfg, weights: Optional[Weights] = None, act_round: Optional[bool] = None):
        self.cfg = cfg
        self.w = weights if weights is not None else synth_weights(cfg)
        self.act_round = (cfg.dtype == "bf16") if act_round is None else act_round

    def r(self, x):
        return round_bf16(x) if self.act_round else x

    # ---- shared decoder pieces
    def _qkv(self, p: str, x: np.ndarray, pos: np.ndarray, qk_norm: bool):
        c, w = self.cfg, self.w
        n = x.shape[0]
        xn = self.r(rms_norm(x, w(f"{p}.attn_norm"), c.rms_eps))
        q = (xn @ w(f"{p}.wq").T).reshape(n, c.n_heads, c.head_dim)
        k = (xn @ w(f"{p}.wk").T).reshape(n, c.n_kv_heads, c.head_dim)
        v = (xn @ w(f"{p}.wv").T).reshape(n, c.n_kv_heads, c.head_dim)
        if qk_norm:
            q = rms_norm(q, w(f"{p}.q_norm"), c.rms_eps)
            k = rms_norm(k, w(f"{p}.k_norm"), c.rms_eps)
        q = self.r(rope(q, pos, c.rope_theta))
        k = self.r(rope(k, pos, c.rope_theta))
        return q, k, self.r(v)

    def _attn_out_mlp(self, p: str, x: np.ndarray, att: np.ndarray) -> np.ndarray:
        c, w = self.cfg, self.w
        n = x.shape[0]
        x = x + self.r(att.reshape(n, -1)) @ w(f"{p}.wo").T
        xn = self.r(rms_norm(x, w(f"{p}.mlp_norm"), c.rms_eps))
        hmid = self.r(silu(xn @ w(f"{p}.w_gate").T) * (xn @ w(f"{p}.w_up").T))
        return x + hmid @ w(f"{p}.w_down").T

    def logits(self, h: np.ndarray, norm_name: str) -> np.ndarray:
        c, w = self.cfg, self.w
        return self.r(rms_norm(h, w(norm_name), c.rms_eps)) @ w("head").T

    # ---- target
    def new_target_cache(self) -> KV:
        c = self.cfg
        return KV(c.target_layers, c.n_kv_heads, c.head_dim)

    def target_forward(self, tokens, cache: KV, want_logits: bool = True):
        """Causal forward of new tokens at positions cache.length .. +n-1.

        Appends their K/V to ``cache``.  Returns (logits [n, V] or None,
        selected hidden [n, k*d]: residual after each context layer, concatenated
        in the listed order)."""
        c, w = self.cfg, self.w
        tokens = np.asarray(tokens, dtype=np.int64)
        n0, n = cache.length, len(tokens)
        pos = np.arange(n0, n0 + n)
        x = w("embed")[tokens].copy()
        keep = {}
        for l in range(c.target_layers):
            p = f"t{l}"
            q, k, v = self._qkv(p, x, pos, c.target_qk_norm)
            cache.append(l, k, v)
            visible = np.arange(n0 + n)[None, :] <= pos[:, None]
            att = attention(q, cache.k[l], cache.v[l], visible)
            x = self._attn_out_mlp(p, x, att)
            if l in c.ctx_layer_ids:
                keep[l] = x.copy()
        sel = np.concatenate([keep[l] for l in c.ctx_layer_ids], axis=1)
        lg = self.logits(x, "final_norm") if want_logits else None
        return lg, sel

    # ---- drafter
    def new_draft_cache(self) -> KV:
        c = self.cfg
        return KV(c.draft_layers, c.n_kv_heads, c.head_dim)

    def fuse(self, sel: np.ndarray) -> np.ndarray:
        """Context feature rms_norm(W_c [h_l1; ...; h_lk])  ([review] §5.1 eq. 9)."""
        c, w = self.cfg, self.w
        return self.r(rms_norm(self.r(sel) @ w("fc").T, w("fc_norm"), c.rms_eps))

    def append_context(self, feat: np.ndarray, cache: KV):
        """Project context features into every draft layer's keys and values and
        store them at positions cache.length .. ([review] §5.1 eq. 10)."""
        c, w = self.cfg, self.w
        n0, n = cache.length, feat.shape[0]
        pos = np.arange(n0, n0 + n)
        for l in range(c.draft_layers):
            p = f"d{l}"
            k = (feat @ w(f"{p}.wk").T).reshape(n, c.n_kv_heads, c.head_dim)
            v = (feat @ w(f"{p}.wv").T).reshape(n, c.n_kv_heads, c.head_dim)
            k = self.r(rope(rms_norm(k, w(f"{p}.k_norm"), c.rms_eps), pos, c.rope_theta))
            cache.append(l, k, self.r(v))

    def draft_forward(self, anchor: int, cache: KV) -> np.ndarray:
        """One parallel pass over [anchor, MASK x (B-1)] at positions n .. n+B-1,
        n = cache.length.  The block attends bidirectionally over [context ; block];
        the cache is not modified.  Returns logits [B, V] (row 0 is the anchor)."""
        c, w = self.cfg, self.w
        B = c.block_size
        n0 = cache.length
        pos = np.arange(n0, n0 + B)
        tokens = np.array([anchor] + [c.mask_token] * (B - 1), dtype=np.int64)
        h = w("embed")[tokens].copy()
        for l in range(c.draft_layers):
            p = f"d{l}"
            q, kb, vb = self._qkv(p, h, pos, True)
            K = np.concatenate([cache.k[l], kb], axis=0)
            V = np.concatenate([cache.v[l], vb], axis=0)
            visible = np.ones((B, n0 + B), dtype=bool)
            att = attention(q, K, V, visible)
            h = self._attn_out_mlp(p, h, att)
        return self.logits(h, "draft_norm")
