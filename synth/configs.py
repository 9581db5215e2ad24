"""Workload descriptions: model shapes, seeds and prompt recipes.

Pure data.  Each workload names a target decoder, a block drafter and the
synthetic prompts it runs on.  Linear, embedding and head matrices are drawn
N(0, 0.02); norm scales are 1.0 unless ``norm_std`` > 0, in which case they
are 1 + N(0, norm_std) so that a test can tell a norm weight that is used
from one that is ignored.  Prompts are uniform token ids.

The five named workloads follow the draft-and-verify round described in
"DFlash: Block Diffusion for Flash Speculative Decoding" (method, inference
§4.1) on model shapes of Qwen3-8B and LLaMA-3.1-8B; the remaining ones are
small shapes used for parity tests (several tiles, ragged tails).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                 # "f32" or "bf16": storage type of matrices, KV and GEMM operands
    vocab: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    target_layers: int
    target_qk_norm: bool
    rope_theta: float
    draft_layers: int
    block_size: int
    ctx_layer_ids: tuple
    batch: int
    prompt_lens: tuple         # one per sequence
    max_new_tokens: int
    rms_eps: float = 1e-6
    weight_std: float = 0.02
    norm_std: float = 0.0
    weight_seed: int = 0
    prompt_seed: int = 1

    @property
    def mask_token(self) -> int:
        return self.vocab - 1

    @property
    def n_ctx_layers(self) -> int:
        return len(self.ctx_layer_ids)

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _ragged_lengths(seed: int, n: int, lo: int, hi: int) -> tuple:
    from . import uniform_ints
    raw = uniform_ints(seed, 0x6C656E00, n, hi - lo + 1)
    return tuple(int(lo + x) for x in raw)


_QWEN8B = dict(dtype="bf16", vocab=151936, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128,
               ffn=12288, target_layers=36, target_qk_norm=True, rope_theta=1e6, draft_layers=5,
               block_size=16, ctx_layer_ids=(1, 9, 17, 25, 33))

_LLAMA8B = dict(dtype="bf16", vocab=128256, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128,
                ffn=14336, target_layers=32, target_qk_norm=False, rope_theta=5e5, draft_layers=5,
                block_size=16, ctx_layer_ids=(1, 8, 15, 22, 29))


def _build() -> dict:
    w = {}
    # Tiny fp32 model: 4-layer target, 2-layer block-4 drafter, features from layers {1, 3}.
    w["tiny_f32"] = Workload(
        name="tiny_f32", dtype="f32", vocab=1024, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64,
        ffn=704, target_layers=4, target_qk_norm=False, rope_theta=1e4, draft_layers=2, block_size=4,
        ctx_layer_ids=(1, 3), batch=1, prompt_lens=(32,), max_new_tokens=64)
    # Qwen3-8B-shaped target, batch 1, 512-token prompt.
    w["qwen3_8b_b1_p512"] = Workload(name="qwen3_8b_b1_p512", batch=1, prompt_lens=(512,),
                                     max_new_tokens=256, **_QWEN8B)
    # Same model, 8192-token prompt (long injected context).
    w["qwen3_8b_b1_p8192"] = Workload(name="qwen3_8b_b1_p8192", batch=1, prompt_lens=(8192,),
                                      max_new_tokens=256, **_QWEN8B)
    # LLaMA-3.1-8B-shaped target, batch 8, 1024-token prompts.
    w["llama31_8b_b8_p1024"] = Workload(name="llama31_8b_b8_p1024", batch=8, prompt_lens=(1024,) * 8,
                                        max_new_tokens=256, **_LLAMA8B)
    # Qwen3-8B-shaped target at concurrency 32, ragged prompts of length U[256, 2048].
    w["qwen3_8b_c32_ragged"] = Workload(name="qwen3_8b_c32_ragged", batch=32,
                                        prompt_lens=_ragged_lengths(1, 32, 256, 2048),
                                        max_new_tokens=256, **_QWEN8B)
    # --- parity-test shapes (not benchmark workloads) ---
    # fp32, ragged batch of 3, non-unit norm scales; weight std 0.1 so that the
    # greedy streams are diverse (at 0.02 a model this small repeats one token).
    w["tiny_f32_b3"] = w["tiny_f32"].with_(name="tiny_f32_b3", batch=3, prompt_lens=(32, 7, 19),
                                           max_new_tokens=40, norm_std=0.1, weight_std=0.1, weight_seed=5,
                                           prompt_seed=6)
    # bf16, head_dim 128, several 128-wide tiles with ragged tails (vocab 5000, prompt 37/100).
    w["small_bf16"] = Workload(
        name="small_bf16", dtype="bf16", vocab=5000, d_model=1024, n_heads=8, n_kv_heads=2, head_dim=128,
        ffn=2816, target_layers=6, target_qk_norm=True, rope_theta=1e6, draft_layers=2, block_size=16,
        ctx_layer_ids=(1, 3), batch=2, prompt_lens=(37, 100), max_new_tokens=48, norm_std=0.1,
        weight_seed=7, prompt_seed=8)
    # Same model in fp32 storage (exact-token parity with a 128 head_dim and 16-wide blocks).
    w["small_f32"] = w["small_bf16"].with_(name="small_f32", dtype="f32")
    # Prompt longer than one prefill chunk (2048 rows): chunked causal prefill.
    w["small_bf16_long"] = w["small_bf16"].with_(name="small_bf16_long", prompt_lens=(2100, 300),
                                                 prompt_seed=11)
    # Long injected context at small width: prompts of 8200-8448 tokens (4 prefill chunks of 2048
    # rows and a ragged one), so the draft attention walks up to 133 context pages per KV head (8+
    # key tiles per cluster rank) and the verify attention as many, as in the 8K benchmark workload.
    # (three sequences: a bf16 near-tie retires one sequence from the comparison, not the test)
    w["small_bf16_long8k"] = Workload(
        name="small_bf16_long8k", dtype="bf16", vocab=5000, d_model=1024, n_heads=8, n_kv_heads=2, head_dim=128,
        ffn=2816, target_layers=2, target_qk_norm=True, rope_theta=1e6, draft_layers=1, block_size=16,
        ctx_layer_ids=(0, 1), batch=3, prompt_lens=(8448, 8300, 8200), max_new_tokens=48, norm_std=0.1,
        weight_seed=14, prompt_seed=15)
    # Batch 20: 320-row draft and verify passes (two 256-token tiles) with an FFN of 8192 and a
    # vocabulary of 40000, so that the round's gate/up and head GEMMs fill a wave of 128 x 256
    # tiles (the persistent kernel, whole tiles) and its down projection has K = 8192 (the
    # persistent kernel with stream-K pieces summed across CTAs).
    w["small_bf16_b20"] = w["small_bf16"].with_(
        name="small_bf16_b20", batch=20, ffn=8192, vocab=40000,
        prompt_lens=(37, 100, 5, 64, 19, 130, 250, 8, 77, 41, 300, 3, 58, 90, 16, 121, 29, 66, 200, 11),
        prompt_seed=13)
    # LLaMA-style small model without target QK-norm, batch 4.
    w["small_bf16_llama"] = Workload(
        name="small_bf16_llama", dtype="bf16", vocab=3001, d_model=512, n_heads=4, n_kv_heads=1,
        head_dim=128, ffn=1408, target_layers=5, target_qk_norm=False, rope_theta=5e5, draft_layers=3,
        block_size=16, ctx_layer_ids=(1, 2, 3), batch=4, prompt_lens=(64, 5, 130, 33), max_new_tokens=40,
        norm_std=0.1, weight_seed=9, prompt_seed=10)
    # Same shapes at batch 12: draft and verify passes of 192 rows (256-token GEMM tiles);
    # weight std 0.04 keeps most greedy choices clear of bf16 near-ties.
    w["small_bf16_llama_b12"] = w["small_bf16_llama"].with_(
        name="small_bf16_llama_b12", batch=12, prompt_lens=(64, 5, 130, 33, 17, 90, 41, 8, 120, 77, 3, 50),
        weight_std=0.04, prompt_seed=12)
    # --- profiling shapes: Qwen3-8B layers, head and embedding at reduced depth (3 target
    # layers, 1 draft layer, features from all three), a few GB on the device, for detailed
    # profiler captures of the same kernel launches as the full-depth workloads ---
    _q3 = dict(_QWEN8B, target_layers=3, draft_layers=1, ctx_layer_ids=(0, 1, 2))
    w["qwen3_8b_shapes_b1_p512_3l"] = Workload(name="qwen3_8b_shapes_b1_p512_3l", batch=1, prompt_lens=(512,),
                                               max_new_tokens=64, **_q3)
    w["qwen3_8b_shapes_c32_ragged_3l"] = Workload(name="qwen3_8b_shapes_c32_ragged_3l", batch=32,
                                                  prompt_lens=_ragged_lengths(1, 32, 256, 2048),
                                                  max_new_tokens=64, **_q3)
    return w


WORKLOADS = None


def get(name: str) -> Workload:
    global WORKLOADS
    if WORKLOADS is None:
        WORKLOADS = _build()
    return WORKLOADS[name]


def names() -> list:
    get("tiny_f32")
    return list(WORKLOADS.keys())
