"""Pins of the oracle's building blocks against closed forms, scalar brute
force and library routines (torch CPU, fp64)."""
import math

import numpy as np
import pytest
import torch

from oracle import model as om

rng = np.random.default_rng(0)


def test_rms_norm_matches_library_and_closed_form():
    x = rng.standard_normal((7, 33))
    w = rng.standard_normal(33)
    got = om.rms_norm(x, w, 1e-6)
    want = torch.nn.functional.rms_norm(torch.from_numpy(x), (33,), torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    # constant vector c*1: output sign(c) * w / sqrt(1 + eps / c^2)
    c, eps = -0.3, 1e-2
    got = om.rms_norm(np.full(5, c), np.arange(1.0, 6.0), eps)
    np.testing.assert_allclose(got, -np.arange(1.0, 6.0) / math.sqrt(1 + eps / c ** 2), rtol=1e-14)


def test_silu_library_and_identity():
    x = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(om.silu(x), torch.nn.functional.silu(torch.from_numpy(x)).numpy(), rtol=1e-14,
                               atol=1e-300)
    np.testing.assert_allclose(om.silu(x) - om.silu(-x), x, atol=1e-12)   # x*s(x) + x*s(-x) = x
    assert om.silu(np.array([0.0]))[0] == 0.0


def _rope_complex(x, pos, theta):
    """Rotary encoding as multiplication of (x_j + i x_{j+hd/2}) by exp(i pos w_j)."""
    hd = x.shape[-1]
    half = hd // 2
    out = np.empty_like(x)
    for n in range(x.shape[0]):
        for h in range(x.shape[1]):
            for j in range(half):
                wj = theta ** (-2.0 * j / hd)
                z = complex(x[n, h, j], x[n, h, j + half]) * complex(math.cos(pos[n] * wj), math.sin(pos[n] * wj))
                out[n, h, j], out[n, h, j + half] = z.real, z.imag
    return out


def test_rope_against_complex_rotation():
    x = rng.standard_normal((5, 3, 16))
    pos = np.array([0, 1, 7, 100, 4095])
    np.testing.assert_allclose(om.rope(x, pos, 1e4), _rope_complex(x, pos, 1e4), rtol=1e-12, atol=1e-12)
    # position 0 is the identity; norms are preserved; scores depend on m - n only
    np.testing.assert_array_equal(om.rope(x[:1], np.array([0]), 1e6), x[:1])
    np.testing.assert_allclose(np.linalg.norm(om.rope(x, pos, 1e6), axis=-1), np.linalg.norm(x, axis=-1))
    q, k = rng.standard_normal((1, 1, 16)), rng.standard_normal((1, 1, 16))
    s1 = (om.rope(q, np.array([10]), 1e4) * om.rope(k, np.array([3]), 1e4)).sum()
    s2 = (om.rope(q, np.array([107]), 1e4) * om.rope(k, np.array([100]), 1e4)).sum()
    assert abs(s1 - s2) < 1e-12


def _attention_loops(q, k, v, visible):
    nq, H, hd = q.shape
    Hkv = k.shape[1]
    g = H // Hkv
    out = np.zeros_like(q)
    for i in range(nq):
        for h in range(H):
            kh = h // g
            scores = []
            for j in range(k.shape[0]):
                if visible[i, j]:
                    scores.append((j, sum(q[i, h, t] * k[j, kh, t] for t in range(hd)) / math.sqrt(hd)))
            m = max(s for _, s in scores)
            den = sum(math.exp(s - m) for _, s in scores)
            for j, s in scores:
                out[i, h] += math.exp(s - m) / den * v[j, kh]
    return out


@pytest.mark.parametrize("causal", [True, False])
def test_attention_brute_force_and_library(causal):
    nq, nk, H, Hkv, hd = 4, 9, 4, 2, 8
    q = rng.standard_normal((nq, H, hd))
    k = rng.standard_normal((nk, Hkv, hd))
    v = rng.standard_normal((nk, Hkv, hd))
    pos = np.arange(nk - nq, nk)
    vis = (np.arange(nk)[None, :] <= pos[:, None]) if causal else np.ones((nq, nk), bool)
    got = om.attention(q, k, v, vis)
    np.testing.assert_allclose(got, _attention_loops(q, k, v, vis), rtol=1e-11, atol=1e-12)
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(np.repeat(k, H // Hkv, axis=1)).permute(1, 0, 2)
    tv = torch.from_numpy(np.repeat(v, H // Hkv, axis=1)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(vis))
    np.testing.assert_allclose(got, ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)


def test_attention_special_cases():
    q = rng.standard_normal((2, 2, 4))
    v = rng.standard_normal((3, 1, 4))
    k_same = np.repeat(rng.standard_normal((1, 1, 4)), 3, axis=0)
    out = om.attention(q, k_same, v, np.ones((2, 3), bool))
    np.testing.assert_allclose(out, np.broadcast_to(v.mean(axis=0), out.shape), atol=1e-14)   # equal keys: mean of values
    only_first = np.zeros((2, 3), bool)
    only_first[:, 0] = True
    out = om.attention(q, rng.standard_normal((3, 1, 4)), v, only_first)
    np.testing.assert_allclose(out, np.broadcast_to(v[0], out.shape), atol=1e-14)


def test_argmax_lowest_index_on_ties():
    x = np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0], [0.0, -1.0, 0.5, 0.5]])
    assert list(om.argmax_lowest(x)) == [1, 0, 2]


def test_round_bf16_matches_library():
    x = np.concatenate([rng.standard_normal(10000) * 10.0 ** rng.integers(-6, 6, 10000),
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8)])])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(om.round_bf16(x), want)
