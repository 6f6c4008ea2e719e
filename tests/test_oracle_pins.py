"""Pins for the fp64 oracle: what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: exact
fractions, closed forms, invariants, an independent numpy restatement and
torch's fp64 scaled_dot_product_attention (the interface the "Optimizing LLM
Inference ..." page names in its FlashAttention section).  A plausible slip in
the oracle (a dropped scale, a wrong sign, an off-by-one mask, a transposed
operand, a wrong GQA head map, a wrong log base, reading past ctx_len) fails
at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

from exact_attention_40_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x):
    """fp32 values that are exactly representable in bf16 -> bit patterns."""
    b = synth.f32_to_bf16_bits(np.asarray(x, np.float32))
    assert np.array_equal(synth.bf16_bits_to_f32(b), np.asarray(x, np.float32)), "not bf16-exact"
    return b


def f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------------ (i) rows
def _golden_rows():
    with open(os.path.join(GOLDEN, "softmax_rows.json")) as f:
        data = json.load(f)
    rows = []
    for r in data["rows"]:
        x = np.array([float(v) for v in r["x"]], np.float64) + r["shift"]
        rows.append((x, np.array(r["expect"], np.float64)))
    return rows


@pytest.mark.parametrize("idx", range(7))
def test_softmax_hand_rows(oracle_mod, idx):
    x, expect = _golden_rows()[idx]
    # the shifted inputs themselves carry a rounding error of ulp(|x|)
    atol = 1e-15 + 8 * np.spacing(np.abs(x[np.isfinite(x)]).max())
    np.testing.assert_allclose(oracle_mod.softmax(x), expect, rtol=0, atol=atol)
    np.testing.assert_allclose(oracle_mod.online_softmax(x), expect, rtol=0, atol=atol)


def test_two_pass_equals_running_softmax(oracle_mod):
    rng = np.random.default_rng(7)
    for n in (1, 2, 5, 64, 1000):
        for scale in (1.0, 30.0):
            x = rng.standard_normal(n) * scale
            a = oracle_mod.softmax(x)
            b = oracle_mod.online_softmax(x)
            np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)
            assert abs(a.sum() - 1.0) < 1e-13


# ------------------------------------------------------------------ (ii) identical keys
def _identical_key_inputs(Nq, Nk, d, seed):
    rng = np.random.default_rng(seed)
    q = bf16(np.round(rng.standard_normal((1, 1, Nq, d)) * 4) / 4)
    k0 = np.round(rng.standard_normal(d) * 4) / 4
    k = bf16(np.broadcast_to(k0, (1, 1, Nk, d)).copy())
    v = bf16(np.round(rng.standard_normal((1, 1, Nk, d)) * 8) / 8)
    return q, k, v


def test_identical_keys_mean_of_v(oracle_mod):
    Nq, Nk, d, scale = 5, 37, 16, 0.25
    q, k, v = _identical_key_inputs(Nq, Nk, d, 1)
    out, lse = oracle_mod.attn(q, k, v, scale, causal=False)
    vm = f64(v)[0, 0].mean(axis=0)
    s = scale * f64(q)[0, 0] @ f64(k)[0, 0, 0]
    for i in range(Nq):
        np.testing.assert_allclose(out[0, 0, i], vm, rtol=0, atol=1e-12)
        assert abs(lse[0, 0, i] - (s[i] + math.log(Nk))) < 1e-12


@pytest.mark.parametrize("Nq,Nk", [(37, 37), (5, 37), (40, 37)])
def test_identical_keys_causal_prefix_mean(oracle_mod, Nq, Nk):
    d, scale = 16, 0.25
    q, k, v = _identical_key_inputs(Nq, Nk, d, 2)
    out, lse = oracle_mod.attn(q, k, v, scale, causal=True)
    vv = f64(v)[0, 0]
    s = scale * f64(q)[0, 0] @ f64(k)[0, 0, 0]
    for i in range(Nq):
        n = i + (Nk - Nq) + 1  # bottom-right aligned mask
        if n <= 0:
            assert np.all(out[0, 0, i] == 0.0) and lse[0, 0, i] == -np.inf
            continue
        np.testing.assert_allclose(out[0, 0, i], vv[:n].mean(axis=0), rtol=0, atol=1e-12)
        assert abs(lse[0, 0, i] - (s[i] + math.log(n))) < 1e-12


def test_zero_query_uniform(oracle_mod):
    q = np.zeros((1, 2, 3, 8), np.uint16)  # +0.0 in bf16
    k = synth.normal_bf16(3, 2, (1, 2, 9, 8))
    v = synth.normal_bf16(3, 3, (1, 2, 9, 8))
    out, lse = oracle_mod.attn(q, k, v, 0.5, causal=False)
    np.testing.assert_allclose(out, np.broadcast_to(f64(v).mean(axis=2, keepdims=True), out.shape),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, math.log(9), rtol=0, atol=1e-12)


# ------------------------------------------------------------------ (iii) dominant score
def test_one_dominant_score_selects_its_value_row(oracle_mod):
    d, Nk, jstar = 32, 50, 17
    rng = np.random.default_rng(3)
    q = np.zeros((1, 1, 1, d), np.float32)
    q[0, 0, 0, 5] = 1.0
    k = np.round(rng.uniform(-1, 1, (1, 1, Nk, d)) * 16) / 16
    k[0, 0, jstar] = 0.0
    k[0, 0, jstar, 5] = 64.0
    v = np.round(rng.standard_normal((1, 1, Nk, d)) * 8) / 8
    out, lse = oracle_mod.attn(bf16(q), bf16(k), bf16(v), 1.0, causal=False)
    np.testing.assert_allclose(out[0, 0, 0], v[0, 0, jstar], rtol=0, atol=1e-12)
    assert abs(lse[0, 0, 0] - 64.0) < 1e-12


# ------------------------------------------------------------------ (iv) permutation
def test_noncausal_permutation_invariance(oracle_mod):
    q, k, v = synth.prefill_inputs_shape(11, 1, 2, 2, 9, 33, 16)
    out, lse = oracle_mod.attn(q, k, v, 0.25, causal=False)
    perm = synth.permutation(99, 33)
    out2, lse2 = oracle_mod.attn(q, k[:, :, perm].copy(), v[:, :, perm].copy(), 0.25, causal=False)
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)
    # a permutation of K alone (V fixed) must change the answer
    out3, _ = oracle_mod.attn(q, k[:, :, perm].copy(), v, 0.25, causal=False)
    assert np.abs(out3 - out).max() > 1e-3


# ------------------------------------------------------------------ (v) brute force
def numpy_attention(q, k, v, scale, causal):
    """Independent matrix-form restatement: softmax(scale*Q K^T + mask) V."""
    Q, K, V = f64(q), f64(k), f64(v)
    B, Hq, Nq, d = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, Nq, d))
    lse = np.zeros((B, Hq, Nq))
    allowed = np.ones((Nq, Nk), bool)
    if causal:
        allowed = np.arange(Nk)[None, :] <= (np.arange(Nq)[:, None] + (Nk - Nq))
    for b in range(B):
        for h in range(Hq):
            S = scale * Q[b, h] @ K[b, h // G].T
            S = np.where(allowed, S, -np.inf)
            m = S.max(axis=1, keepdims=True)
            dead = ~np.isfinite(m[:, 0])
            m[dead] = 0.0
            P = np.exp(S - m)
            den = P.sum(axis=1, keepdims=True)
            with np.errstate(invalid="ignore", divide="ignore"):
                out[b, h] = np.where(dead[:, None], 0.0, (P @ V[b, h // G]) / den)
                lse[b, h] = np.where(dead, -np.inf, m[:, 0] + np.log(den[:, 0]))
    return out, lse


SHAPES = [
    # B, Hq, Hkv, Nq, Nk, d
    (1, 1, 1, 1, 1, 8),
    (2, 4, 2, 7, 11, 8),
    (1, 4, 1, 13, 13, 16),
    (1, 2, 2, 20, 6, 4),
    (2, 8, 4, 33, 65, 32),
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_bruteforce_numpy(oracle_mod, shape, causal):
    B, Hq, Hkv, Nq, Nk, d = shape
    q, k, v = synth.prefill_inputs_shape(5, B, Hq, Hkv, Nq, Nk, d)
    scale = 1.0 / math.sqrt(d)
    out, lse = oracle_mod.attn(q, k, v, scale, causal)
    ref_o, ref_l = numpy_attention(q, k, v, scale, causal)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(ref_l))
    fin = np.isfinite(ref_l)
    np.testing.assert_allclose(lse[fin], ref_l[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_torch_sdpa_fp64(oracle_mod, causal):
    torch = pytest.importorskip("torch")
    B, Hq, Hkv, Nq, Nk, d = 2, 4, 2, 17, 29, 16
    q, k, v = synth.prefill_inputs_shape(6, B, Hq, Hkv, Nq, Nk, d)
    scale = 0.3
    out, _ = oracle_mod.attn(q, k, v, scale, causal)
    G = Hq // Hkv
    tq = torch.from_numpy(f64(q))
    tk = torch.from_numpy(f64(k)).repeat_interleave(G, dim=1)
    tv = torch.from_numpy(f64(v)).repeat_interleave(G, dim=1)
    mask = None
    if causal:
        mask = torch.arange(Nk)[None, :] <= (torch.arange(Nq)[:, None] + (Nk - Nq))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)


def test_rows_match_full(oracle_mod):
    B, Hq, Hkv, N, d = 1, 4, 2, 50, 16
    q, k, v = synth.prefill_inputs_shape(8, B, Hq, Hkv, N, N, d)
    out, lse = oracle_mod.attn(q, k, v, 0.25, True)
    rows = synth.sample_rows(8, B, Hq, N, 7)
    o2, l2 = oracle_mod.attn_rows(q, k, v, rows, 0.25, True)
    np.testing.assert_array_equal(o2, out[rows[:, 0], rows[:, 1], rows[:, 2]])
    np.testing.assert_array_equal(l2, lse[rows[:, 0], rows[:, 1], rows[:, 2]])


def test_no_keys_gives_zero_and_minus_inf(oracle_mod):
    q, k, v = synth.prefill_inputs_shape(9, 1, 2, 1, 4, 0, 8)
    out, lse = oracle_mod.attn(q, k, v, 0.25, False)
    assert np.all(out == 0.0) and np.all(lse == -np.inf)


# ------------------------------------------------------------------ (vii) GQA
def test_gqa_equals_repeated_mha(oracle_mod):
    B, Hq, Hkv, N, d = 2, 8, 2, 24, 16
    q, k, v = synth.prefill_inputs_shape(10, B, Hq, Hkv, N, N, d)
    G = Hq // Hkv
    o1, l1 = oracle_mod.attn(q, k, v, 0.25, True)
    o2, l2 = oracle_mod.attn(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1), 0.25, True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # heads hq and hq+1 of one group share K/V but not Q; interleaved map would differ
    o3, _ = oracle_mod.attn(q, np.tile(k, (1, G, 1, 1)), np.tile(v, (1, G, 1, 1)), 0.25, True)
    assert np.abs(o3 - o1).max() > 1e-3


# ------------------------------------------------------------------ (vi) decode
def _decode_case(lens, Hq=4, Hkv=2, d=16, seed=12, extra=0):
    return synth.decode_inputs_lens(seed, np.array(lens, np.int32), Hq, Hkv, d, 16,
                                    nan_tail=True, extra_blocks=extra)


def test_decode_equals_prefill_on_gathered_kv(oracle_mod):
    inp = _decode_case([1, 15, 16, 17, 40])
    scale = 0.25
    out, lse = oracle_mod.decode_paged(inp["q"], inp["k_cache"], inp["v_cache"],
                                       inp["block_table"], inp["ctx_lens"], scale)
    for s, n in enumerate(inp["ctx_lens"]):
        t = np.arange(n)
        phys = inp["block_table"][s, t // 16]
        kk = inp["k_cache"][phys, :, t % 16, :].transpose(1, 0, 2)[None].copy()
        vv = inp["v_cache"][phys, :, t % 16, :].transpose(1, 0, 2)[None].copy()
        o2, l2 = oracle_mod.attn(inp["q"][s][None, :, None, :].copy(), kk, vv, scale, False)
        np.testing.assert_allclose(out[s], o2[0, :, 0], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[s], l2[0, :, 0], rtol=0, atol=1e-15)
    assert np.all(np.isfinite(out))  # NaN tails past ctx_len are never read


def test_decode_numpy_restatement(oracle_mod):
    inp = _decode_case([3, 33, 64], Hq=8, Hkv=2, d=32, seed=13)
    scale = 1.0 / math.sqrt(32)
    out, lse = oracle_mod.decode_paged(inp["q"], inp["k_cache"], inp["v_cache"],
                                       inp["block_table"], inp["ctx_lens"], scale)
    Q, Kc, Vc = f64(inp["q"]), f64(inp["k_cache"]), f64(inp["v_cache"])
    for s, n in enumerate(inp["ctx_lens"]):
        for h in range(8):
            kv = h // 4
            ks = np.stack([Kc[inp["block_table"][s, t // 16], kv, t % 16] for t in range(n)])
            vs = np.stack([Vc[inp["block_table"][s, t // 16], kv, t % 16] for t in range(n)])
            sc = scale * ks @ Q[s, h]
            w = np.exp(sc - sc.max())
            np.testing.assert_allclose(out[s, h], w @ vs / w.sum(), rtol=0, atol=1e-12)
            assert abs(lse[s, h] - (sc.max() + math.log(w.sum()))) < 1e-12


def test_decode_block_permutation_invariance(oracle_mod):
    inp = _decode_case([20, 47, 5], extra=3)
    nb = inp["k_cache"].shape[0]
    perm = synth.permutation(77, nb)
    k2 = np.empty_like(inp["k_cache"])
    v2 = np.empty_like(inp["v_cache"])
    k2[perm] = inp["k_cache"]
    v2[perm] = inp["v_cache"]
    t2 = np.where(inp["block_table"] >= 0, perm[np.maximum(inp["block_table"], 0)], -1).astype(np.int32)
    a = oracle_mod.decode_paged(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                inp["ctx_lens"], 0.25)
    b = oracle_mod.decode_paged(inp["q"], k2, v2, t2, inp["ctx_lens"], 0.25)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_decode_empty_context(oracle_mod):
    inp = _decode_case([0, 5])
    out, lse = oracle_mod.decode_paged(inp["q"], inp["k_cache"], inp["v_cache"],
                                       inp["block_table"], inp["ctx_lens"], 0.25)
    assert np.all(out[0] == 0.0) and np.all(lse[0] == -np.inf)
    assert np.all(np.isfinite(out[1]))


# ------------------------------------------------------------------ (viii) split/combine algebra
def test_lse_combine_of_key_splits_equals_full(oracle_mod):
    """Partial (o_s, lse_s) over disjoint key ranges merge to the full answer:
    L = log sum_s exp(lse_s), o = sum_s exp(lse_s - L) o_s.  This is the
    algebra the split-KV decode relies on; an empty split (lse = -inf) has
    weight zero."""
    B, H, Nq, Nk, d = 1, 2, 3, 100, 16
    q, k, v = synth.prefill_inputs_shape(14, B, H, H, Nq, Nk, d)
    full_o, full_l = oracle_mod.attn(q, k, v, 0.25, False)
    cuts = [0, 30, 30, 64, 100]  # includes an empty split
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        parts.append(oracle_mod.attn(q, k[:, :, a:b].copy(), v[:, :, a:b].copy(), 0.25, False))
    lses = np.stack([p[1] for p in parts])
    L = np.log(np.sum(np.exp(lses - lses.max(0)), axis=0)) + lses.max(0)
    o = sum(np.exp(p[1] - L)[..., None] * p[0] for p in parts)
    np.testing.assert_allclose(o, full_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, full_l, rtol=0, atol=1e-12)
