"""Pins of the oracle's attention backward (dQ, dK, dV from dO) against
what the mathematics fixes, independently of its formulas.

The main pin is the definition of a gradient: central finite differences of
L = <O, dO>, with O from a plain numpy fp64 forward, must match every entry
of dQ, dK and dV on tiny shapes (GQA, both masks, Nq != Nk with rows that
see no key).  Closed forms and invariants cover the rest: identical keys
give dQ = 0 and dV_j = mean_i dO_i; GQA equals MHA with repeated K, V summed
per group; permuting K and V rows permutes dK and dV the same way.  A slip
in the oracle (a dropped D_i term, a missing scale, P^T for P, the group sum
left out, the mask off by one) fails one of them."""
import numpy as np
import pytest

import oracle
from exact_attention_40_gb300 import synth


def f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def np_forward(q, k, v, scale, causal):
    """O of attention in fp64 from fp64 arrays [B,H,N,d] (GQA by head index)."""
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    out = np.zeros_like(q)
    for b in range(B):
        for h in range(Hq):
            s = scale * q[b, h] @ k[b, h // G].T
            if causal:
                i = np.arange(Nq)[:, None]
                j = np.arange(Nk)[None, :]
                s = np.where(j <= i + (Nk - Nq), s, -np.inf)
            for r in range(Nq):
                if np.all(np.isneginf(s[r])):
                    continue
                p = np.exp(s[r] - s[r].max())
                out[b, h, r] = (p / p.sum()) @ v[b, h // G]
    return out


def finite_difference_grads(q, k, v, do, scale, causal, h=1e-6):
    def loss(qq, kk, vv):
        return float(np.sum(np_forward(qq, kk, vv, scale, causal) * do))
    grads = []
    for which in range(3):
        arrs = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(arrs[which])
        for idx in np.ndindex(*g.shape):
            base = arrs[which][idx]
            arrs[which][idx] = base + h
            lp = loss(*arrs)
            arrs[which][idx] = base - h
            lm = loss(*arrs)
            arrs[which][idx] = base
            g[idx] = (lp - lm) / (2 * h)
        grads.append(g)
    return grads


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 2, 1, 5, 7, 4, False),
    (1, 2, 1, 5, 7, 4, True),
    (1, 2, 2, 6, 6, 3, True),
    (2, 1, 1, 7, 4, 2, True),    # Nq > Nk: the first rows see no key
])
def test_gradients_equal_finite_differences(B, Hq, Hkv, Nq, Nk, d, causal):
    q = synth.normal_bf16(70, 0, (B, Hq, Nq, d))
    k = synth.normal_bf16(70, 1, (B, Hkv, Nk, d))
    v = synth.normal_bf16(70, 2, (B, Hkv, Nk, d))
    do = synth.normal_bf16(70, 3, (B, Hq, Nq, d))
    scale = 0.7
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale, causal)
    fq, fk, fv = finite_difference_grads(f64(q), f64(k), f64(v), f64(do), scale, causal)
    for got, want, name in ((dq, fq, "dq"), (dk, fk, "dk"), (dv, fv, "dv")):
        np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-8, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys(causal):
    # all k_j equal: rows of dS sum to zero, so dQ = 0; non-causal P_ij = 1/Nk
    # so dV_j = mean over queries of dO (summed over the group's heads)
    B, Hq, Hkv, N, d = 1, 4, 2, 9, 8
    q = synth.normal_bf16(71, 0, (B, Hq, N, d))
    k = np.tile(synth.normal_bf16(71, 1, (1, 1, 1, d)), (B, Hkv, N, 1))
    v = synth.normal_bf16(71, 2, (B, Hkv, N, d))
    do = synth.normal_bf16(71, 3, (B, Hq, N, d))
    dq, _, dv = oracle.attn_bwd(q, k, v, do, 0.3, causal)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    if not causal:
        g = f64(do).reshape(B, Hkv, Hq // Hkv, N, d).sum(axis=2).sum(axis=2) / N
        np.testing.assert_allclose(dv, np.repeat(g[:, :, None, :], N, axis=2), rtol=1e-12, atol=1e-14)


def test_gqa_is_mha_with_repeated_kv_summed():
    B, Hq, Hkv, N, d = 1, 6, 2, 11, 8
    q = synth.normal_bf16(72, 0, (B, Hq, N, d))
    k = synth.normal_bf16(72, 1, (B, Hkv, N, d))
    v = synth.normal_bf16(72, 2, (B, Hkv, N, d))
    do = synth.normal_bf16(72, 3, (B, Hq, N, d))
    G = Hq // Hkv
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.35, True)
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    dq2, dk2, dv2 = oracle.attn_bwd(q, kr, vr, do, 0.35, True)
    np.testing.assert_allclose(dq, dq2, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, G, N, d).sum(axis=2), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, G, N, d).sum(axis=2), rtol=1e-12, atol=1e-14)


def test_key_permutation_equivariance():
    B, H, N, d = 1, 2, 10, 8
    q = synth.normal_bf16(73, 0, (B, H, N, d))
    k = synth.normal_bf16(73, 1, (B, H, N, d))
    v = synth.normal_bf16(73, 2, (B, H, N, d))
    do = synth.normal_bf16(73, 3, (B, H, N, d))
    perm = synth.permutation(73, N)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.4, False)
    dq2, dk2, dv2 = oracle.attn_bwd(q, k[:, :, perm].copy(), v[:, :, perm].copy(), do, 0.4, False)
    np.testing.assert_allclose(dq2, dq, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dk2, dk[:, :, perm], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dv2, dv[:, :, perm], rtol=1e-12, atol=1e-14)


def test_rejects_bad_arguments():
    x = np.zeros((1, 3, 4, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.attn_bwd(x, np.zeros((1, 2, 4, 8), np.uint16), np.zeros((1, 2, 4, 8), np.uint16), x, 0.1, False)
