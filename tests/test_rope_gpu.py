"""RoPE + paged KV-cache write parity: the CUDA kernel (through the C ABI)
against the fp64 oracle on the same seeded inputs.

Bar, derived from the arithmetic: angles are reduced in fp64, cos/sin and
the rotation run in fp32 and each output is rounded once to bf16, so an
output element is within half a bf16 step of the exact value (2^-8
relative) plus fp32 error relative to its pair's size:
|y - ref| <= 4e-3 |ref| + 2e-5 (|x_i| + |x_(i+d/2)|).  Values are copied
to the cache bit for bit, and every cache slot no token maps to keeps its
bits."""
import numpy as np
import pytest

from exact_attention_40_gb300 import synth
from helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(oracle_mod):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_40_gb300 import build
    build.build()
    from exact_attention_40_gb300 import exattn
    return torch, exattn, oracle_mod, torch.device("cuda:0")


def bits(t):
    import torch
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def close(got_bits, ref, x_bits, label):
    got = synth.bf16_bits_to_f32(got_bits).astype(np.float64)
    x = synth.bf16_bits_to_f32(x_bits).astype(np.float64)
    h = x.shape[-1] // 2
    pair = np.abs(x[..., :h]) + np.abs(x[..., h:])
    pair = np.concatenate([pair, pair], axis=-1)
    err = np.abs(got - ref)
    bad = err > 4e-3 * np.abs(ref) + 2e-5 * pair
    assert np.all(np.isfinite(got)), label
    assert not bad.any(), "%s: %d elements off, worst %.3e" % (label, int(bad.sum()), float(err.max()))


def run_case(env, inp, Hkv, d, base, expect_status=0, random_cache=True):
    torch, ex, oracle, dev = env
    nb = inp["num_blocks"]
    if random_cache:
        kc0 = synth.normal_bf16(77, 0, (nb, Hkv, 16, d))
        vc0 = synth.normal_bf16(77, 1, (nb, Hkv, 16, d))
    else:
        kc0 = np.zeros((nb, Hkv, 16, d), np.uint16)
        vc0 = np.zeros((nb, Hkv, 16, d), np.uint16)
    qd = to_dev(inp["q"], dev)
    kcd, vcd = to_dev(kc0, dev), to_dev(vc0, dev)
    ex.attn_rope_cache_write(qd, to_dev(inp["k"], dev), to_dev(inp["v"], dev),
                             to_dev(inp["seq_ids"], dev), to_dev(inp["positions"], dev),
                             to_dev(inp["block_table"], dev), kcd, vcd, base=base)
    torch.cuda.synchronize()
    assert ex.attn_get_device_status() == expect_status
    q_ref, k_ref, slot = oracle.rope_cache_write(inp["q"], inp["k"], inp["seq_ids"], inp["positions"],
                                                 inp["block_table"], nb, base)
    close(bits(qd), q_ref, inp["q"], "q")
    kc, vc = bits(kcd), bits(vcd)
    ok = slot >= 0
    blk, off = slot[ok] // 16, slot[ok] % 16
    close(kc[blk, :, off, :], k_ref[ok], inp["k"][ok], "cached k")
    assert np.array_equal(vc[blk, :, off, :], inp["v"][ok]), "cached v"
    # every other slot keeps its bits
    kc[blk, :, off, :] = kc0[blk, :, off, :]
    vc[blk, :, off, :] = vc0[blk, :, off, :]
    assert np.array_equal(kc, kc0) and np.array_equal(vc, vc0), "a slot no token maps to changed"
    return slot


def test_decode_step_small(env):
    # one new token per sequence at ctx_len - 1; first, middle and last slots
    inp = synth.rope_inputs_lens(50, [1, 16, 17, 300, 1000, 4097], 1, 8, 2, 128)
    run_case(env, inp, 2, 128, 500000.0)


def test_prefill_chunk_ragged(env):
    # several tokens per sequence crossing block boundaries, d = 64
    inp = synth.rope_inputs_lens(51, [40, 3, 70, 33], 40, 4, 4, 64)
    run_case(env, inp, 4, 64, 10000.0)


@pytest.mark.parametrize("d", [16, 96, 256])
def test_head_sizes(env, d):
    inp = synth.rope_inputs_lens(52, [20, 35], 20, 2, 1, d)
    run_case(env, inp, 1, d, 10000.0)


@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (128, 16)])
def test_many_heads(env, Hq, Hkv):
    # 704 and 1408 items per token at d = 128: four and eight per thread, the
    # kernel variants with the deepest per-thread staging
    inp = synth.rope_inputs_lens(56, [40, 300], 20, Hq, Hkv, 128)
    run_case(env, inp, Hkv, 128, 500000.0)


def test_long_positions(env):
    # positions up to 32767: the angles reach ~3e4 radians
    inp = synth.rope_inputs_lens(53, [32768, 20000], 8, 4, 2, 128)
    run_case(env, inp, 2, 128, 500000.0)
    run_case(env, inp, 2, 128, 10000.0)


def test_positions_near_2_pow_20(env):
    # angles up to ~1e6 radians, where the reduction modulo 2 pi is hardest;
    # zeroed caches keep the 65,000-block cache copies cheap
    inp = synth.rope_inputs_lens(55, [1 << 20, 3000], 4, 2, 1, 64)
    run_case(env, inp, 1, 64, 500000.0, random_cache=False)
    run_case(env, inp, 1, 64, 10000.0, random_cache=False)


def test_decode_config(env):
    # the decode step of the paged-decode workload (64 sequences, 18101
    # blocks): all of q and every written slot against the oracle
    cfg = synth.ROPE["rope_decode_step"]
    inp = synth.rope_inputs(cfg)
    run_case(env, inp, cfg.Hkv, cfg.d, cfg.base, random_cache=False)


def test_outside_the_table_is_flagged(env):
    inp = synth.rope_inputs_lens(54, [20, 20], 20, 2, 1, 64)
    inp["seq_ids"] = inp["seq_ids"].copy()
    inp["positions"] = inp["positions"].copy()
    inp["seq_ids"][3] = 7            # no such sequence
    inp["positions"][5] = 10 ** 6    # past the table
    inp["block_table"] = inp["block_table"].copy()
    inp["block_table"][1, 0] = -1    # unmapped block for sequence 1's first 16 positions
    slot = run_case(env, inp, 1, 64, 10000.0, expect_status=2)
    assert (slot < 0).sum() == 2 + 16


def test_no_tokens_and_rejected(env):
    torch, ex, _, dev = env
    z = torch.zeros((0, 2, 64), device=dev, dtype=torch.bfloat16)
    zk = torch.zeros((0, 1, 64), device=dev, dtype=torch.bfloat16)
    i0 = torch.zeros((0,), device=dev, dtype=torch.int32)
    tbl = torch.zeros((1, 1), device=dev, dtype=torch.int32)
    kc = torch.zeros((1, 1, 16, 64), device=dev, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    ex.attn_rope_cache_write(z, zk, zk, i0, i0, tbl, kc, vc)
    one = torch.zeros((1, 2, 64), device=dev, dtype=torch.bfloat16)
    onek = torch.zeros((1, 1, 64), device=dev, dtype=torch.bfloat16)
    i1 = torch.zeros((1,), device=dev, dtype=torch.int32)
    with pytest.raises(ex.ExattnError):   # both caches in one buffer
        ex.attn_rope_cache_write(one, onek, onek, i1, i1, tbl, kc, kc)
    with pytest.raises(ex.ExattnError):   # odd head size
        bad = torch.zeros((1, 2, 24), device=dev, dtype=torch.bfloat16)
        badk = torch.zeros((1, 1, 24), device=dev, dtype=torch.bfloat16)
        ex.attn_rope_cache_write(bad, badk, badk, i1, i1, tbl,
                                 torch.zeros((1, 1, 16, 24), device=dev, dtype=torch.bfloat16),
                                 torch.zeros((1, 1, 16, 24), device=dev, dtype=torch.bfloat16))
    torch.cuda.synchronize()
    assert ex.attn_get_device_status() == 0
