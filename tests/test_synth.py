"""The seeded input generator: published SplitMix64 values, bf16 rounding,
distribution, paged-layout structure and stored digests."""
import hashlib
import json
import os

import numpy as np

from exact_attention_40_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_values():
    # first outputs of SplitMix64 from state 0 (Steele, Lea & Flood's generator)
    z = synth.splitmix64(0, 3)
    assert [int(x) for x in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_stream_offsets_agree():
    a = synth.splitmix64(123, 100)
    b = synth.splitmix64(123, 60, 40)
    assert np.array_equal(a[40:], b)


def test_bf16_round_to_nearest_even():
    bits = np.array([0x3F800000, 0x3F808000, 0x3F818000, 0xBF808000, 0x3F808001, 0x7F000000],
                    np.uint32)
    got = synth.f32_to_bf16_bits(bits.view(np.float32))
    # 1.00390625 is a tie between 0x3F80 and 0x3F81 -> even 0x3F80;
    # 1.01171875 is a tie between 0x3F81 and 0x3F82 -> even 0x3F82; one ulp
    # above the first tie rounds up
    assert list(got[:5]) == [0x3F80, 0x3F80, 0x3F82, 0xBF80, 0x3F81]
    assert np.isfinite(synth.bf16_bits_to_f32(got[5:]))[0]


def test_normal_moments():
    x = synth.bf16_bits_to_f32(synth.normal_bf16(9, 1, (1 << 20,))).astype(np.float64)
    assert abs(x.mean()) < 0.01
    assert abs(x.std() - 1.0) < 0.01
    assert abs(np.mean(np.abs(x) > 1.96) - 0.05) < 0.005


def test_ctx_lengths_and_block_table():
    lens = synth.ctx_lengths(5, 64, 512, 8192)
    assert lens.min() >= 512 and lens.max() <= 8192
    table, nb = synth.paged_layout(lens, 16, 5)
    nblk = (lens + 15) // 16
    used = np.concatenate([table[s, :n] for s, n in enumerate(nblk)])
    assert np.array_equal(np.sort(used), np.arange(nb))  # each physical block exactly once
    for s, n in enumerate(nblk):
        assert np.all(table[s, n:] == -1)
    assert not np.array_equal(used, np.arange(nb))  # actually permuted


def test_sample_rows_distinct_and_in_range():
    rows = synth.sample_rows(4, 1, 3, 500, 20)
    assert rows.shape == (60, 3)
    for h in range(3):
        r = rows[rows[:, 1] == h, 2]
        assert len(set(r.tolist())) == 20 and r.min() >= 0 and r.max() < 500


def test_stored_digests():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(GOLDEN, "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(GOLDEN, "synth_sha256.json")) as f:
        stored = json.load(f)
    assert mod.digests() == stored


def test_stability_variant_is_exact_times_8():
    cfg = synth.PREFILL["tiny"]
    q, _, _ = synth.prefill_inputs(cfg)
    q8 = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(q) * np.float32(8))
    assert np.array_equal(synth.bf16_bits_to_f32(q8), synth.bf16_bits_to_f32(q) * 8)
