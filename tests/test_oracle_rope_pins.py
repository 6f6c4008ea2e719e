"""Pins of the oracle's rotary embedding + paged KV-cache write against what
the mathematics fixes.  RoPE rotates pairs (i, i + d/2) of each head vector
by theta_i = pos * base^(-2 i / d); the rotated key and the value go to slot
pos % 16 of physical block block_table[seq][pos / 16].

A plausible slip in the oracle fails one of these: the pairs taken
interleaved instead of split in halves, a wrong sign of the sine, the
frequency exponent off by a factor, the position not applied, the block
or slot index transposed."""
import math

import numpy as np
import pytest

import oracle
from exact_attention_40_gb300 import synth

BASE = 500000.0


def bf16(vals):
    return synth.f32_to_bf16_bits(np.asarray(vals, np.float32))


def f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def rope(q, k, pos, base=BASE):
    T = q.shape[0]
    table = np.arange(T, dtype=np.int32).reshape(T, 1)
    n_blocks = T
    return oracle.rope_cache_write(q, k, np.arange(T), np.asarray(pos, np.int32), table, n_blocks, base)


def unit(d, idx, T=1, H=1):
    x = np.zeros((T, H, d), np.uint16)
    x[..., idx] = bf16([1.0])[0]
    return x


def test_position_zero_is_identity():
    q = synth.normal_bf16(1, 0, (3, 4, 64))
    k = synth.normal_bf16(1, 1, (3, 2, 64))
    qo, ko, _ = rope(q, k, [0, 0, 0])
    assert np.array_equal(qo, f64(q)) and np.array_equal(ko, f64(k))


def test_pair_norms_are_kept():
    q = synth.normal_bf16(2, 0, (5, 3, 128))
    k = synth.normal_bf16(2, 1, (5, 1, 128))
    qo, _, _ = rope(q, k, [1, 7, 100, 4095, 32767])
    x = f64(q)
    n_in = x[..., :64] ** 2 + x[..., 64:] ** 2
    n_out = qo[..., :64] ** 2 + qo[..., 64:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12, atol=1e-300)


def test_first_pair_turns_by_the_position():
    # i = 0 has frequency 1: e_0 -> (cos pos) e_0 + (sin pos) e_(d/2)
    d = 128
    for pos in (1, 5, 1234):
        qo, _, _ = rope(unit(d, 0), unit(d, 0), [pos])
        want = np.zeros(d)
        want[0], want[d // 2] = math.cos(pos), math.sin(pos)
        np.testing.assert_allclose(qo[0, 0], want, rtol=0, atol=1e-13)


def test_second_half_partner_and_sign():
    # e_(d/2) -> -(sin pos) e_0 + (cos pos) e_(d/2): halves are partners, and
    # the first component gets minus the sine
    d, pos = 64, 3
    qo, _, _ = rope(unit(d, d // 2), unit(d, d // 2), [pos])
    want = np.zeros(d)
    want[0], want[d // 2] = -math.sin(pos), math.cos(pos)
    np.testing.assert_allclose(qo[0, 0], want, rtol=0, atol=1e-13)


def test_slowest_pair_frequency():
    # i = d/2 - 1 turns by pos * base^(-(d-2)/d)
    d, pos = 128, 30000
    qo, _, _ = rope(unit(d, d // 2 - 1), unit(d, d // 2 - 1), [pos])
    ang = pos * BASE ** (-(d - 2) / d)
    assert abs(qo[0, 0, d // 2 - 1] - math.cos(ang)) < 1e-13
    assert abs(qo[0, 0, d - 1] - math.sin(ang)) < 1e-13


def test_scores_depend_on_relative_position_only():
    # <R_m q, R_n k> = <R_(m+s) q, R_(n+s) k>: the property RoPE is built for
    d = 128
    q = synth.normal_bf16(3, 0, (1, 1, d))
    k = synth.normal_bf16(3, 1, (1, 1, d))
    for m, n, s in [(5, 2, 100), (0, 17, 4000), (300, 300, 7)]:
        q1, _, _ = rope(q, k, [m])
        _, k1, _ = rope(q, k, [n])
        q2, _, _ = rope(q, k, [m + s])
        _, k2, _ = rope(q, k, [n + s])
        a = float(q1[0, 0] @ k1[0, 0])
        b = float(q2[0, 0] @ k2[0, 0])
        assert abs(a - b) < 1e-9 * max(1.0, abs(a)), (m, n, s, a, b)
    # and it does change with the offset m - n
    qa, _, _ = rope(q, k, [5])
    _, ka, _ = rope(q, k, [2])
    _, kb, _ = rope(q, k, [3])
    assert abs(float(qa[0, 0] @ ka[0, 0]) - float(qa[0, 0] @ kb[0, 0])) > 1e-6


def test_slots_follow_the_block_table():
    # the logical order of a sequence read back through its table is the
    # order of positions, whatever the physical block ids
    n_seq, per_seq, d = 3, 40, 8
    tokens = [(s, p) for s in range(n_seq) for p in range(per_seq)]
    T = len(tokens)
    max_blocks = 3
    phys = synth.permutation(9, n_seq * max_blocks).astype(np.int32).reshape(n_seq, max_blocks)
    q = synth.normal_bf16(4, 0, (T, 1, d))
    k = synth.normal_bf16(4, 1, (T, 1, d))
    _, _, slot = oracle.rope_cache_write(q, k, [s for s, _ in tokens], [p for _, p in tokens], phys,
                                         n_seq * max_blocks, BASE)
    assert len(set(slot.tolist())) == T and slot.min() >= 0
    tag = np.full(n_seq * max_blocks * 16, -1, np.int64)
    tag[slot] = np.arange(T)
    for s in range(n_seq):
        logical = np.concatenate([tag[b * 16:(b + 1) * 16] for b in phys[s]])[:per_seq]
        assert np.array_equal(logical, np.array([i for i, (ss, _) in enumerate(tokens) if ss == s]))


def test_outside_the_table_or_cache_is_not_stored():
    q = synth.normal_bf16(5, 0, (4, 1, 8))
    k = synth.normal_bf16(5, 1, (4, 1, 8))
    table = np.array([[0, 5], [1, -1]], np.int32)
    _, _, slot = oracle.rope_cache_write(q, k, [0, 0, 1, 1], [3, 40, 20, 2], table, 4, BASE)
    # pos 40 -> logical block 2 (past the table); pos 20 -> entry -1; block 5 >= 4 unused here
    assert slot.tolist() == [3, -1, -1, 1 * 16 + 2]
    _, _, slot = oracle.rope_cache_write(q, k, [0, 0, 0, 0], [16, 17, 0, 1], table, 4, BASE)
    assert slot.tolist() == [-1, -1, 0, 1]   # block 5 lies outside a 4-block cache


def test_written_cache_feeds_the_decode_oracle():
    # a sequence written token by token through the slots, then read by the
    # decode oracle, equals attention over the rotated keys in order
    d, Hq, Hkv, n = 64, 4, 2, 37
    max_blocks = 4
    table = np.array([[6, 1, 4, 0]], np.int32)
    num_blocks = 8
    q = synth.normal_bf16(6, 0, (n, Hq, d))
    k = synth.normal_bf16(6, 1, (n, Hkv, d))
    v = synth.normal_bf16(6, 2, (n, Hkv, d))
    _, ko, slot = oracle.rope_cache_write(q, k, np.zeros(n), np.arange(n), table, num_blocks, BASE)
    kb = bf16(ko)                                    # the cache holds bf16
    kc = np.zeros((num_blocks * 16, Hkv, d), np.uint16)
    vc = np.zeros((num_blocks * 16, Hkv, d), np.uint16)
    kc[slot], vc[slot] = kb, v
    kc = kc.reshape(num_blocks, 16, Hkv, d).transpose(0, 2, 1, 3).copy()
    vc = vc.reshape(num_blocks, 16, Hkv, d).transpose(0, 2, 1, 3).copy()
    qd = q[n - 1:n]                                  # the last token's query
    out_d, lse_d = oracle.decode_paged(qd, kc, vc, table, np.array([n], np.int32), 0.125)
    kk = kb.transpose(1, 0, 2)[None].copy()          # [1, Hkv, n, d]
    vv = v.transpose(1, 0, 2)[None].copy()
    out_p, lse_p = oracle.attn(qd.transpose(1, 0, 2)[None].copy(), kk, vv, 0.125, False)
    np.testing.assert_allclose(out_d[0], out_p[0, :, 0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse_d[0], lse_p[0, :, 0], rtol=1e-12, atol=1e-14)


def test_rejects_bad_arguments():
    q = np.zeros((1, 1, 7), np.uint16)
    with pytest.raises(ValueError):
        oracle.rope_cache_write(q, q, [0], [0], np.zeros((1, 1), np.int32), 1, BASE)
    q = np.zeros((1, 1, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.rope_cache_write(q, q, [0], [0], np.zeros((1, 1), np.int32), 1, -1.0)
