"""Prefill parity: the CUDA kernel (through the C ABI) against the fp64
oracle on the same seeded inputs.

Small and mid-size cases are compared element by element; the large
workloads run at full size, in the launch configuration the benchmark times,
and are checked on seeded samples of query rows that the oracle computes one
by one."""
import math

import numpy as np
import pytest

from exact_attention_40_gb300 import synth
from helpers import assert_parity, metrics, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(oracle_mod):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_40_gb300 import build
    build.build()
    from exact_attention_40_gb300 import exattn
    dev = torch.device("cuda:0")
    return torch, exattn, oracle_mod, dev


def run(env, q, k, v, causal, scale=None):
    torch, ex, _, dev = env
    out, lse = ex.attn_fwd(to_dev(q, dev), to_dev(k, dev), to_dev(v, dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ex.attn_get_device_status() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


SHAPES = [
    # B, Hq, Hkv, Nq, Nk, d, causal
    (1, 1, 1, 1, 1, 64, False),
    (1, 1, 1, 1, 1, 128, True),
    (2, 4, 2, 127, 127, 128, True),
    (1, 2, 1, 129, 129, 64, True),
    (1, 8, 8, 300, 300, 128, False),
    (1, 4, 1, 200, 77, 128, False),
    (1, 4, 1, 77, 200, 128, True),   # Nq < Nk: every row sees a prefix plus its diagonal
    (1, 4, 4, 200, 77, 128, True),   # Nq > Nk: the first rows see no key at all
    (3, 2, 2, 257, 513, 64, True),
    (1, 16, 2, 384, 384, 128, True),  # GQA group 8
    (2, 32, 1, 256, 256, 64, True),   # GQA group 32
    (2, 2, 2, 640, 640, 128, False),
    # several items per CTA, some without a tile B (Nq mod 256 <= 128), so
    # one warpgroup stages two O tiles in a row between the other's
    (8, 32, 8, 384, 384, 128, False),
    (8, 32, 8, 384, 128, 128, True),  # and the first item of each head sees no key
    (8, 16, 4, 328, 328, 64, True),
    # Nq - Nk = 150: each head's first item has an empty tile A and a tile B
    # that sees keys; its second has a tile A only
    (8, 32, 8, 300, 150, 128, True),
    # one key, 880 queries: four one-key-tile items per head, the last with
    # a tile A only; causal, only the last row sees the key, so three of
    # each head's items are empty
    (4, 32, 8, 880, 1, 64, False),
    (4, 32, 8, 880, 1, 64, True),
    # one query against 4000 keys: items with a tile A only across 32 key tiles
    (8, 32, 8, 1, 4000, 128, True),
    # d = 64 with several full items per CTA (512 items, causal)
    (4, 32, 8, 1024, 1024, 64, True),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dHq%dHkv%dNq%dNk%dd%d%s" % (
    s[0], s[1], s[2], s[3], s[4], s[5], "c" if s[6] else "n"))
def test_shapes_elementwise(env, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    q, k, v = synth.prefill_inputs_shape(21, B, Hq, Hkv, Nq, Nk, d)
    got_o, got_l = run(env, q, k, v, causal)
    ref_o, ref_l = env[2].attn(q, k, v, 1.0 / math.sqrt(d), causal)
    assert_parity(metrics(got_o, got_l, ref_o, ref_l), str(shape))


def test_tiny_config(env):
    cfg = synth.PREFILL["tiny"]
    q, k, v = synth.prefill_inputs(cfg)
    got_o, got_l = run(env, q, k, v, cfg.causal)
    ref_o, ref_l = env[2].attn(q, k, v, cfg.scale, cfg.causal)
    assert_parity(metrics(got_o, got_l, ref_o, ref_l), "tiny")


def test_llama3_8b_causal_full(env):
    cfg = synth.PREFILL["llama3_8b_causal"]
    q, k, v = synth.prefill_inputs(cfg)
    got_o, got_l = run(env, q, k, v, cfg.causal)
    ref_o, ref_l = env[2].attn(q, k, v, cfg.scale, cfg.causal)
    assert_parity(metrics(got_o, got_l, ref_o, ref_l), "llama3_8b_causal")


def _sampled(env, name, per_head):
    cfg = synth.PREFILL[name]
    q, k, v = synth.prefill_inputs(cfg)
    got_o, got_l = run(env, q, k, v, cfg.causal)
    rows = synth.sample_rows(cfg.seed, cfg.B, cfg.Hq, cfg.N, per_head)
    ref_o, ref_l = env[2].attn_rows(q, k, v, rows, cfg.scale, cfg.causal)
    sel = (rows[:, 0], rows[:, 1], rows[:, 2])
    assert_parity(metrics(got_o[sel], got_l[sel], ref_o, ref_l), name)
    # properties that hold at every row: finite output, LSE finite
    assert np.all(np.isfinite(got_o)) and np.all(np.isfinite(got_l))


@pytest.mark.parametrize("name", ["batched_noncausal", "batched_causal",
                                  "batched_stab_noncausal", "batched_stab_causal"])
def test_batched_sampled(env, name):
    _sampled(env, name, 256)


def test_long_context_sampled(env):
    _sampled(env, "long_causal", 256)


def test_no_keys(env):
    torch, ex, _, dev = env
    q, _, _ = synth.prefill_inputs_shape(3, 1, 2, 2, 130, 1, 64)
    k = np.zeros((1, 2, 0, 64), np.uint16)
    out, lse = ex.attn_fwd(to_dev(q, dev), to_dev(k, dev), to_dev(k, dev), causal=False)
    torch.cuda.synchronize()
    assert torch.all(out == 0).item()
    assert torch.all(torch.isneginf(lse)).item()


def test_empty_is_noop(env):
    torch, ex, _, dev = env
    q = torch.zeros((1, 2, 0, 128), device=dev, dtype=torch.bfloat16)
    out, lse = ex.attn_fwd(q, q, q)
    assert out.shape == q.shape and lse.shape == (1, 2, 0)


def test_deterministic_and_guard_bands(env):
    """Two runs are bitwise equal, and nothing is written outside out/lse."""
    torch, ex, _, dev = env
    B, Hq, Hkv, N, d = 1, 8, 2, 1000, 128
    q, k, v = synth.prefill_inputs_shape(31, B, Hq, Hkv, N, N, d)
    tq, tk, tv = to_dev(q, dev), to_dev(k, dev), to_dev(v, dev)
    n_out = B * Hq * N * d
    pad = 4096  # elements of NaN guard on both sides (8 KB, keeps 16-byte alignment)
    obuf = torch.full((n_out + 2 * pad,), float("nan"), device=dev, dtype=torch.bfloat16)
    lbuf = torch.full((B * Hq * N + 2 * pad,), float("nan"), device=dev, dtype=torch.float32)
    out = obuf[pad:pad + n_out].view(B, Hq, N, d)
    lse = lbuf[pad:pad + B * Hq * N].view(B, Hq, N)
    ex.attn_fwd(tq, tk, tv, causal=True, out=out, lse=lse)
    first = out.clone(), lse.clone()
    ex.attn_fwd(tq, tk, tv, causal=True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(first[0].view(torch.int16), out.view(torch.int16))
    assert torch.equal(first[1], lse)
    assert torch.all(torch.isnan(obuf[:pad])).item() and torch.all(torch.isnan(obuf[-pad:])).item()
    assert torch.all(torch.isnan(lbuf[:pad])).item() and torch.all(torch.isnan(lbuf[-pad:])).item()


def test_side_stream_and_no_lse(env):
    torch, ex, orc, dev = env
    q, k, v = synth.prefill_inputs_shape(41, 2, 4, 4, 256, 256, 128)
    s = torch.cuda.Stream()
    tq, tk, tv = to_dev(q, dev), to_dev(k, dev), to_dev(v, dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out, lse = ex.attn_fwd(tq, tk, tv, causal=True, return_lse=False)
    s.synchronize()
    assert lse is None
    ref_o, ref_l = orc.attn(q, k, v, 1.0 / math.sqrt(128), True)
    m = metrics(out.float().cpu().numpy(), None, ref_o, ref_l)
    assert_parity(m, "side stream")


def test_explicit_scale(env):
    q, k, v = synth.prefill_inputs_shape(51, 1, 2, 2, 190, 190, 64)
    got_o, got_l = run(env, q, k, v, True, scale=0.37)
    ref_o, ref_l = env[2].attn(q, k, v, 0.37, True)
    assert_parity(metrics(got_o, got_l, ref_o, ref_l), "scale 0.37")
