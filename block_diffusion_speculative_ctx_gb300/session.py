"""Session helper over the C ABI: builds the config and weight structs from a
synthetic workload, routes library allocations to torch's caching allocator,
and marshals tokens.  No arithmetic of the round happens here."""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np

from . import (ALLOC_FN, DFLASH_DTYPE_BF16, DFLASH_DTYPE_F32, DFLASH_FLAG_KEEP_LOGITS, DFLASH_FLAG_NO_GRAPHS,
               DFLASH_OK, FREE_FN,
               INSPECT_ANCHORS, INSPECT_DRAFT_K, INSPECT_DRAFT_V, INSPECT_HIDDEN_VERIFY, INSPECT_LENGTHS,
               INSPECT_LOGITS_DRAFT, INSPECT_LOGITS_PREFILL, INSPECT_LOGITS_VERIFY, INSPECT_POSTERIOR,
               INSPECT_STATS, INSPECT_TARGET_K, INSPECT_TARGET_V, INSPECT_PROFILE, INSPECT_PROFILE_RESET,
               KERNEL_CLASSES, DFlashError, _check, _ptr, dflash_config, dflash_profile_entry,
               dflash_destroy, dflash_init, dflash_layer_weights, dflash_stats, dflash_weights, load)


def config_from_workload(w, max_batch: int, max_seq_len: int, keep_logits: bool = False) -> dflash_config:
    c = dflash_config()
    c.dtype = DFLASH_DTYPE_BF16 if w.dtype == "bf16" else DFLASH_DTYPE_F32
    c.vocab, c.d_model, c.n_heads, c.n_kv_heads = w.vocab, w.d_model, w.n_heads, w.n_kv_heads
    c.head_dim, c.ffn, c.target_layers = w.head_dim, w.ffn, w.target_layers
    c.target_qk_norm = 1 if w.target_qk_norm else 0
    c.draft_layers, c.block_size, c.n_ctx_layers = w.draft_layers, w.block_size, len(w.ctx_layer_ids)
    for i, l in enumerate(w.ctx_layer_ids):
        c.ctx_layer_ids[i] = l
    c.mask_token = w.mask_token
    c.max_batch, c.max_seq_len = max_batch, max_seq_len
    c.flags = DFLASH_FLAG_KEEP_LOGITS if keep_logits else 0
    c.rms_eps, c.rope_theta = w.rms_eps, w.rope_theta
    return c


class _TorchAllocator:
    """Library allocations served by torch's caching allocator on the current device."""

    def __init__(self):
        import torch
        self.torch = torch
        self.live = {}
        self.alloc_cb = ALLOC_FN(self._alloc)
        self.free_cb = FREE_FN(self._free)

    def _alloc(self, nbytes, user):
        try:
            t = self.torch.empty(int(nbytes) + 256, dtype=self.torch.uint8, device="cuda")
        except Exception:
            return None
        p = t.data_ptr()
        aligned = (p + 255) & ~255
        self.live[aligned] = t
        return aligned

    def _free(self, ptr, user):
        self.live.pop(ptr, None)


def upload_weights(w, device="cuda"):
    """Device tensors of every named weight of a synthetic workload."""
    import torch
    import synth
    out = {}
    for name, shape, kind in synth.weight_specs(w):
        a = synth.weight_bits(w, name)
        if a.dtype == np.uint16:
            t = torch.from_numpy(a.view(np.int16)).to(device)
        else:
            t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)
        out[name] = t
    return out


def weights_struct(w, tens: dict):
    """dflash_weights pointing at ``tens`` (name -> device tensor)."""
    def layer(prefix, qk):
        lw = dflash_layer_weights()
        for m in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "attn_norm", "mlp_norm"):
            setattr(lw, m, tens[f"{prefix}.{m}"].data_ptr())
        if qk:
            lw.q_norm = tens[f"{prefix}.q_norm"].data_ptr()
            lw.k_norm = tens[f"{prefix}.k_norm"].data_ptr()
        return lw

    tl = (dflash_layer_weights * w.target_layers)(*[layer(f"t{l}", w.target_qk_norm) for l in range(w.target_layers)])
    dl = (dflash_layer_weights * w.draft_layers)(*[layer(f"d{l}", True) for l in range(w.draft_layers)])
    ws = dflash_weights()
    ws.embed = tens["embed"].data_ptr()
    ws.head = tens["head"].data_ptr()
    ws.final_norm = tens["final_norm"].data_ptr()
    ws.target = tl
    ws.fc = tens["fc"].data_ptr()
    ws.fc_norm = tens["fc_norm"].data_ptr()
    ws.draft = dl
    ws.draft_norm = tens["draft_norm"].data_ptr()
    return ws, (tl, dl)


class Session:
    """One dflash_ctx on torch's current CUDA stream."""

    def __init__(self, w, max_batch: Optional[int] = None, max_seq_len: Optional[int] = None,
                 keep_logits: bool = False, use_torch_alloc: bool = True, tensors: Optional[dict] = None,
                 graphs: bool = True, kv_pool_tokens: int = 0):
        import torch
        if not torch.cuda.is_available():
            raise RuntimeError("no CUDA device: the dflash library has no CPU path")
        self.lib = load()
        self.w = w
        self.B = w.block_size
        self.max_batch = max_batch or w.batch
        self.max_seq_len = max_seq_len or (max(w.prompt_lens) + w.max_new_tokens + 3 * w.block_size + 8)
        self.cfg = config_from_workload(w, self.max_batch, self.max_seq_len, keep_logits)
        if not graphs:
            self.cfg.flags |= DFLASH_FLAG_NO_GRAPHS
        self.cfg.kv_pool_tokens = int(kv_pool_tokens)  # 0: max_batch * max_seq_len
        self.alloc = _TorchAllocator() if use_torch_alloc else None
        if self.alloc:
            self.cfg.alloc, self.cfg.free = self.alloc.alloc_cb, self.alloc.free_cb
        self.stream = torch.cuda.current_stream()
        tens = tensors if tensors is not None else upload_weights(w)
        ws, keep = weights_struct(w, tens)
        self.ctx = dflash_init(self.cfg, ws, self.stream.cuda_stream)
        del keep
        # the library reads embed, head, fc, wo and w_down in place for the session's lifetime;
        # the other matrices were packed into its own buffers and may go
        packed = {"wq", "wk", "wv", "w_gate", "w_up"}
        self._borrowed = {k: t for k, t in tens.items() if k.rsplit(".", 1)[-1] not in packed}
        self.batch = 0

    # -------------------------------------------------------------- the round
    def prefill(self, prompts: Sequence[np.ndarray]) -> np.ndarray:
        lens = np.array([len(p) for p in prompts], dtype=np.int32)
        toks = np.ascontiguousarray(np.concatenate([np.asarray(p, dtype=np.int32) for p in prompts]))
        first = np.zeros(len(prompts), dtype=np.int32)
        _check(self.ctx, self.lib.dflash_prefill(self.ctx, len(lens), _ptr(lens), _ptr(toks), _ptr(first)))
        self.batch = len(prompts)
        return first

    def set_block_size(self, B: int):
        """Block size of the following rounds, 1 <= B <= the configured one."""
        _check(self.ctx, self.lib.dflash_set_block_size(self.ctx, int(B)))
        self.B = int(self.lib.dflash_block_size(self.ctx))

    def draft_block(self, out=None):
        """Draft tokens [batch, B-1]; ``out`` may be a numpy array or a device tensor."""
        if out is None:
            out = np.zeros((self.batch, max(self.B - 1, 1)), dtype=np.int32)
        _check(self.ctx, self.lib.dflash_draft_block(self.ctx, _ptr(out)))
        return out

    def verify(self, proposal, accepted=None, bonus=None):
        if isinstance(proposal, np.ndarray):
            proposal = np.ascontiguousarray(proposal, dtype=np.int32)
        if accepted is None:
            accepted = np.zeros(self.batch, dtype=np.int32)
        if bonus is None:
            bonus = np.zeros(self.batch, dtype=np.int32)
        _check(self.ctx, self.lib.dflash_verify(self.ctx, _ptr(proposal), _ptr(accepted), _ptr(bonus)))
        return accepted, bonus

    def set_sampling_filter(self, top_k: int = 0, top_p: float = 1.0):
        """Top-k / top-p filter of both laws of the following sampled rounds (0 / 1.0: off)."""
        _check(self.ctx, self.lib.dflash_set_sampling_filter(self.ctx, int(top_k), float(top_p)))

    def draft_block_sampled(self, temperature: float, u_draft, out=None):
        """Proposals [batch, B-1] drawn at temperature T with uniforms u_draft [batch, B-1]."""
        if isinstance(u_draft, np.ndarray):
            u_draft = np.ascontiguousarray(u_draft, dtype=np.float32)
        if out is None:
            out = np.zeros((self.batch, max(self.B - 1, 1)), dtype=np.int32)
        _check(self.ctx, self.lib.dflash_draft_block_sampled(self.ctx, float(temperature), _ptr(u_draft), _ptr(out)))
        return out

    def verify_sampled(self, temperature: float, proposal, u_verify, accepted=None, emitted=None):
        """Speculative rejection sampling of a proposal; u_verify [batch, B] (B-1 acceptance
        uniforms, then the emission uniform).  Returns (accepted, emitted)."""
        if isinstance(proposal, np.ndarray):
            proposal = np.ascontiguousarray(proposal, dtype=np.int32)
        if isinstance(u_verify, np.ndarray):
            u_verify = np.ascontiguousarray(u_verify, dtype=np.float32)
        if accepted is None:
            accepted = np.zeros(self.batch, dtype=np.int32)
        if emitted is None:
            emitted = np.zeros(self.batch, dtype=np.int32)
        _check(self.ctx, self.lib.dflash_verify_sampled(self.ctx, float(temperature), _ptr(proposal), _ptr(u_verify),
                                                        _ptr(accepted), _ptr(emitted)))
        return accepted, emitted

    def train_forward(self, tokens, anchors, lam: float) -> float:
        """The drafter's position-weighted training loss over one clean sequence
        (one block per anchor).  Leaves the session empty."""
        toks = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        anc = np.ascontiguousarray(np.asarray(anchors, dtype=np.int32))
        loss = np.zeros(1, dtype=np.float32)
        _check(self.ctx, self.lib.dflash_train_forward(self.ctx, len(toks), _ptr(toks), len(anc), _ptr(anc),
                                                       float(lam), _ptr(loss)))
        self.batch = 0
        return float(loss[0])

    def generate(self, prompts: Sequence[np.ndarray], max_new_tokens: int):
        lens = np.array([len(p) for p in prompts], dtype=np.int32)
        toks = np.ascontiguousarray(np.concatenate([np.asarray(p, dtype=np.int32) for p in prompts]))
        out = np.zeros((len(prompts), max_new_tokens), dtype=np.int32)
        out_lens = np.zeros(len(prompts), dtype=np.int32)
        st = dflash_stats()
        _check(self.ctx, self.lib.dflash_generate(self.ctx, len(lens), _ptr(lens), _ptr(toks), max_new_tokens,
                                                  _ptr(out), _ptr(out_lens), ctypes.byref(st)))
        self.batch = len(prompts)
        return out, st

    # ------------------------------------------------------------- inspection
    def _inspect(self, what, dst, seq=0, layer=0):
        written = ctypes.c_size_t(0)
        _check(self.ctx, self.lib.dflash_inspect(self.ctx, what, seq, layer, _ptr(dst), dst.nbytes,
                                                 ctypes.byref(written)))
        return dst

    def lengths(self):
        return self._inspect(INSPECT_LENGTHS, np.zeros(self.batch, np.int32))

    def anchors(self):
        return self._inspect(INSPECT_ANCHORS, np.zeros(self.batch, np.int32))

    def posterior(self):
        return self._inspect(INSPECT_POSTERIOR, np.zeros((self.batch, self.B), np.int32))

    def logits(self, which: str):
        V = self.w.vocab
        if which == "prefill":
            return self._inspect(INSPECT_LOGITS_PREFILL, np.zeros((self.batch, V), np.float32))
        item = INSPECT_LOGITS_DRAFT if which == "draft" else INSPECT_LOGITS_VERIFY
        return self._inspect(item, np.zeros((self.batch, self.B, V), np.float32))

    def hidden_verify(self):
        return self._inspect(INSPECT_HIDDEN_VERIFY, np.zeros((self.batch, self.B, self.w.d_model), np.float32))

    def cache(self, which: str, kv: str, seq: int, layer: int) -> np.ndarray:
        """Committed rows of one cache layer as float64 [n, H_kv, hd]."""
        n = int(self.lengths()[seq])
        item = {("target", "k"): INSPECT_TARGET_K, ("target", "v"): INSPECT_TARGET_V,
                ("draft", "k"): INSPECT_DRAFT_K, ("draft", "v"): INSPECT_DRAFT_V}[(which, kv)]
        shape = (n, self.w.n_kv_heads, self.w.head_dim)
        if self.w.dtype == "bf16":
            raw = self._inspect(item, np.zeros(shape, np.uint16), seq, layer)
            return (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        return self._inspect(item, np.zeros(shape, np.float32), seq, layer).astype(np.float64)

    def stats(self) -> dflash_stats:
        st = dflash_stats()
        buf = (ctypes.c_char * ctypes.sizeof(st))()
        written = ctypes.c_size_t(0)
        _check(self.ctx, self.lib.dflash_inspect(self.ctx, INSPECT_STATS, 0, 0, ctypes.addressof(buf),
                                                 ctypes.sizeof(st), ctypes.byref(written)))
        ctypes.memmove(ctypes.addressof(st), buf, ctypes.sizeof(st))
        return st

    def set_profiling(self, on: bool):
        _check(self.ctx, self.lib.dflash_set_profiling(self.ctx, 1 if on else 0))

    def profile(self, reset: bool = False) -> dict:
        """{kernel class: {launches, ms, bytes, flops}} accumulated while profiling was on."""
        arr = (dflash_profile_entry * len(KERNEL_CLASSES))()
        written = ctypes.c_size_t(0)
        _check(self.ctx, self.lib.dflash_inspect(self.ctx, INSPECT_PROFILE, 0, 0, ctypes.addressof(arr),
                                                 ctypes.sizeof(arr), ctypes.byref(written)))
        out = {name: dict(launches=int(e.launches), ms=e.ms, bytes=e.bytes, flops=e.flops)
               for name, e in zip(KERNEL_CLASSES, arr)}
        if reset:
            self.profile_reset()
        return out

    def profile_reset(self):
        dummy = np.zeros(1, np.uint8)
        written = ctypes.c_size_t(0)
        _check(self.ctx, self.lib.dflash_inspect(self.ctx, INSPECT_PROFILE_RESET, 0, 0, _ptr(dummy), 1,
                                                 ctypes.byref(written)))

    def close(self):
        if getattr(self, "ctx", None):
            dflash_destroy(self.ctx)
            self.ctx = None
        self._borrowed = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()
