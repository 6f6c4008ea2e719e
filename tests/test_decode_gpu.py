"""Paged-decode parity: split-KV kernel + LSE merge (through the C ABI)
against the fp64 oracle, which walks the block table token by token."""
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
    return torch, exattn, oracle_mod, torch.device("cuda:0")


def run(env, inp, scale, expect_status=0, **kw):
    torch, ex, _, dev = env
    out, lse = ex.attn_decode_paged(to_dev(inp["q"], dev), to_dev(inp["k_cache"], dev),
                                    to_dev(inp["v_cache"], dev), to_dev(inp["block_table"], dev),
                                    to_dev(inp["ctx_lens"], dev), scale=scale, **kw)
    torch.cuda.synchronize()
    assert ex.attn_get_device_status() == expect_status
    return out.float().cpu().numpy(), (lse.cpu().numpy() if lse is not None else None)


def oracle(env, inp, scale):
    return env[2].decode_paged(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                               inp["ctx_lens"], scale)


def test_decode_config_full(env):
    cfg = synth.DECODE["decode_paged"]
    inp = synth.decode_inputs(cfg)
    got_o, got_l = run(env, inp, cfg.scale)
    ref_o, ref_l = oracle(env, inp, cfg.scale)
    assert_parity(metrics(got_o, got_l, ref_o, ref_l), "decode_paged")


EDGE_LENS = [1, 15, 16, 17, 511, 512, 513, 1024, 1500, 8192]


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 8, 128), (8, 8, 128), (8, 4, 64), (16, 2, 128),
                                      (4, 1, 64),
                                      # groups of 16, 24 and 32 query heads: one, one and a half
                                      # and two 16-row chunks per KV head
                                      (16, 1, 128), (24, 1, 64), (32, 1, 128)])
def test_edge_lengths(env, Hq, Hkv, d):
    inp = synth.decode_inputs_lens(61, np.array(EDGE_LENS, np.int32), Hq, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    got_o, got_l = run(env, inp, scale)
    ref_o, ref_l = oracle(env, inp, scale)
    assert_parity(metrics(got_o, got_l, ref_o, ref_l), "edge %d/%d/%d" % (Hq, Hkv, d))


def test_empty_context_rows(env):
    inp = synth.decode_inputs_lens(62, np.array([0, 33, 0, 700], np.int32), 8, 2, 128)
    got_o, got_l = run(env, inp, 0.1)
    ref_o, ref_l = oracle(env, inp, 0.1)
    assert np.all(got_o[0] == 0) and np.all(got_o[2] == 0)
    assert np.all(got_l[0] == -np.inf) and np.all(got_l[2] == -np.inf)
    assert_parity(metrics(got_o, got_l, ref_o, ref_l), "empty rows")


def test_spare_table_columns_unused(env):
    """Table entries past a sequence's last block are never read."""
    inp = synth.decode_inputs_lens(63, np.array([40, 300], np.int32), 8, 2, 128)
    bt = np.concatenate([inp["block_table"], np.full((2, 5), 123456, np.int32)], axis=1)
    inp2 = dict(inp, block_table=np.where(bt < 0, 987654, bt).astype(np.int32))
    got_o, got_l = run(env, inp2, 0.1)
    ref_o, ref_l = oracle(env, inp, 0.1)
    assert_parity(metrics(got_o, got_l, ref_o, ref_l), "spare columns")


def test_bad_table_entry_is_flagged_not_faulted(env):
    torch, ex, _, _ = env
    inp = synth.decode_inputs_lens(64, np.array([64, 64], np.int32), 4, 1, 128)
    bt = inp["block_table"].copy()
    bt[1, 2] = inp["k_cache"].shape[0] + 7  # out of range: must be skipped and reported
    run(env, dict(inp, block_table=bt), 0.1, expect_status=2)
    # the context is still healthy afterwards
    got_o, got_l = run(env, inp, 0.1)
    ref_o, ref_l = oracle(env, inp, 0.1)
    assert_parity(metrics(got_o, got_l, ref_o, ref_l), "after bad entry")


def test_ctx_len_beyond_table_is_clamped_and_flagged(env):
    inp = synth.decode_inputs_lens(65, np.array([32, 48], np.int32), 4, 1, 128, nan_tail=False)
    lens = inp["ctx_lens"].copy()
    lens[0] = 10 ** 6
    run(env, dict(inp, ctx_lens=lens), 0.1, expect_status=2)


def test_deterministic(env):
    inp = synth.decode_inputs_lens(66, np.array([3000, 17, 900], np.int32), 32, 8, 128)
    a = run(env, inp, 0.1)
    b = run(env, inp, 0.1)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_no_lse_and_workspace_reuse(env):
    torch, ex, _, dev = env
    inp = synth.decode_inputs_lens(67, np.array([100, 1100], np.int32), 8, 2, 128)
    ws = torch.full((ex.attn_decode_workspace_bytes(2, 8, 128, inp["block_table"].shape[1]),),
                    255, device=dev, dtype=torch.uint8)  # garbage contents are fine
    got_o, got_l = run(env, inp, 0.1, workspace=ws, return_lse=False)
    assert got_l is None
    ref_o, ref_l = oracle(env, inp, 0.1)
    assert_parity(metrics(got_o, None, ref_o, ref_l), "no lse")


def test_single_split_tables_write_directly(env):
    """Block tables that cannot reach a second 512-token split: the split
    kernel writes the result itself (no merge launch).  Same bits as the
    merged path, which a wider table (spare columns) forces."""
    inp = synth.decode_inputs_lens(68, np.array([0, 200, 512, 1, 77], np.int32), 8, 2, 128)
    assert inp["block_table"].shape[1] * 16 <= 512
    got_o, got_l = run(env, inp, 0.1)
    ref_o, ref_l = oracle(env, inp, 0.1)
    assert np.all(got_o[0] == 0) and np.all(got_l[0] == -np.inf)
    assert_parity(metrics(got_o, got_l, ref_o, ref_l), "single split")
    wide = np.concatenate([inp["block_table"], np.full((5, 8), -1, np.int32)], axis=1)
    w_o, w_l = run(env, dict(inp, block_table=wide), 0.1)
    assert np.array_equal(got_o, w_o) and np.array_equal(got_l, w_l)
