"""The seeded input generator: Philox4x32-10 known answers, the C library
against an independent numpy statement, distributions and layouts."""
import numpy as np
import pytest

import synth
from synth import configs

# Known-answer vectors published with the Random123 library for
# philox4x32 with 10 rounds: (counter, key) -> output.
PHILOX_KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", PHILOX_KAT)
def test_philox_known_answers(ctr, key, want):
    assert tuple(int(x) for x in synth.philox4x32_10(ctr, key)) == want
    assert tuple(int(x) for x in synth.philox4x32_10_np(np.array([ctr]), key)[0]) == want


def test_c_normals_match_numpy_statement():
    seed, stream, n = 123456789012345, 77, 4001
    got = synth.normal_f32(seed, stream, n, 0.0, 0.02)
    j = np.arange((n + 1) // 2, dtype=np.uint64)
    ctr = np.stack([j & 0xFFFFFFFF, j >> np.uint64(32), np.full_like(j, stream), np.zeros_like(j)], 1)
    x = synth.philox4x32_10_np(ctr, (seed & 0xFFFFFFFF, seed >> 32)).astype(np.uint64)
    a = (x[:, 0] << np.uint64(32)) | x[:, 1]
    b = (x[:, 2] << np.uint64(32)) | x[:, 3]
    u1 = ((a >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * 2.0 ** -53
    u2 = (b >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.stack([r * np.cos(2 * np.pi * u2), r * np.sin(2 * np.pi * u2)], 1).reshape(-1)[:n]
    want = (0.02 * z).astype(np.float32)
    # libm and numpy may differ in the last bit of a double; after rounding to
    # float32 that shows up as at most one float32 ulp on rare elements.
    np.testing.assert_array_max_ulp(got, want, maxulp=1)


def test_normal_moments_and_determinism():
    x = synth.normal_f32(0, 5, 2_000_000, 0.0, 1.0).astype(np.float64)
    assert abs(x.mean()) < 3e-3 and abs(x.std() - 1.0) < 3e-3
    assert abs(np.mean(x ** 4) - 3.0) < 0.03          # Gaussian kurtosis
    assert np.array_equal(synth.normal_f32(0, 5, 1000), synth.normal_f32(0, 5, 1000))
    assert not np.array_equal(synth.normal_f32(0, 5, 1000), synth.normal_f32(0, 6, 1000))


def test_uniform_ints_range_and_spread():
    v = synth.uniform_ints(1, 9, 400_000, 1000)
    assert v.min() >= 0 and v.max() < 1000
    counts = np.bincount(v, minlength=1000)
    assert counts.min() > 300 and counts.max() < 520


def test_bf16_round_trip():
    x = np.array([1.0, 1.00390625, 1.005859375, -3.14159, 1e-8, 65504.0, 0.0], np.float32)
    b = synth.f32_to_bf16_bits(x)
    y = synth.bf16_bits_to_f32(b)
    # exactly representable values survive; ties go to even
    assert y[0] == 1.0 and y[1] == 1.0 and y[2] == 1.0078125
    assert np.all(np.abs(y - x) <= np.abs(x) * 2.0 ** -8)
    assert np.array_equal(synth.f32_to_bf16_bits(y), b)


def test_weight_layout_and_values():
    cfg = configs.get("small_bf16")
    specs = synth.weight_specs(cfg)
    names = [s[0] for s in specs]
    assert len(set(names)) == len(names)
    assert names[0] == "embed" and "head" in names and "fc" in names
    shapes = dict((s[0], s[1]) for s in specs)
    assert shapes["fc"] == (cfg.d_model, cfg.n_ctx_layers * cfg.d_model)
    assert shapes["t0.wq"] == (cfg.q_dim, cfg.d_model)
    w = synth.weight_f32(cfg, "t0.wq")
    bits = synth.weight_bits(cfg, "t0.wq")
    assert bits.dtype == np.uint16 and np.array_equal(synth.bf16_bits_to_f32(bits), w)
    assert abs(float(w.std()) - 0.02) < 1e-3
    n = synth.weight_f32(cfg, "t0.attn_norm")
    assert n.dtype == np.float32 and abs(float(n.mean()) - 1.0) < 0.02 and n.std() > 0.05
    n1 = synth.weight_f32(configs.get("tiny_f32"), "t0.attn_norm")
    assert np.all(n1 == 1.0)


def test_prompts():
    cfg = configs.get("qwen3_8b_c32_ragged")
    assert all(256 <= n <= 2048 for n in cfg.prompt_lens) and len(cfg.prompt_lens) == 32
    cfg = configs.get("small_bf16")
    ps = synth.prompts(cfg)
    assert [len(p) for p in ps] == list(cfg.prompt_lens)
    assert all(p.min() >= 0 and p.max() < cfg.vocab for p in ps)
