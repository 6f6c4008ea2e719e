"""CUDA-graph capture of the decode step ("Optimizing LLM Inference ..."
page, section Compilation and CUDA Graphs).  A replay runs exactly the
kernels attn_decode_paged launches, so it must reproduce a direct call bit
for bit, and every replay must match the fp64 oracle at the decode bar, at
capture and after the inputs it was captured with change in place."""
import math

import numpy as np
import pytest

from exact_attention_40_gb300 import synth
from helpers import assert_parity, metrics, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_40_gb300 import build
    build.build()
    from exact_attention_40_gb300 import exattn
    return torch, exattn, torch.device("cuda:0")


def direct(ex, torch, q, kc, vc, bt, cl):
    out, lse = ex.attn_decode_paged(q, kc, vc, bt, cl)
    torch.cuda.synchronize()
    return out.clone(), lse.clone()


def oracle_check(orc, out, lse, q, kc, vc, table, lens, label):
    ref_o, ref_l = orc.decode_paged(q, kc, vc, table, lens, 1.0 / math.sqrt(q.shape[-1]))
    assert_parity(metrics(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l), label)


def test_replay_matches_direct_call_and_oracle(env, oracle_mod):
    torch, ex, dev = env
    lens = np.array([1, 100, 700, 1600, 33], np.int32)
    inp = synth.decode_inputs_lens(60, lens, 32, 8, 128, nan_tail=False)
    q, kc, vc = to_dev(inp["q"], dev), to_dev(inp["k_cache"], dev), to_dev(inp["v_cache"], dev)
    bt, cl = to_dev(inp["block_table"], dev), to_dev(inp["ctx_lens"], dev)
    ref_o, ref_l = direct(ex, torch, q, kc, vc, bt, cl)
    graph, out, lse = ex.attn_decode_graph_capture(q, kc, vc, bt, cl)
    with graph:
        torch.cuda.synchronize()
        for i in range(3):
            out.zero_()
            lse.zero_()
            graph.launch()
            torch.cuda.synchronize()
            assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
            oracle_check(oracle_mod, out, lse, inp["q"], inp["k_cache"], inp["v_cache"],
                         inp["block_table"], inp["ctx_lens"], "replay %d" % i)

        # new contents in the captured buffers: another query, shorter
        # contexts, table entries remapped onto other blocks
        q2 = synth.normal_bf16(61, 0, tuple(q.shape))
        lens2 = np.array([1, 50, 512, 1599, 17], np.int32)
        table = inp["block_table"].copy()
        table[2, :4] = table[3, :4]
        q.copy_(to_dev(q2, dev))
        cl.copy_(to_dev(lens2, dev))
        bt.copy_(to_dev(table, dev))
        graph.launch()
        torch.cuda.synchronize()
        got_o, got_l = out.clone(), lse.clone()
    oracle_check(oracle_mod, got_o, got_l, q2, inp["k_cache"], inp["v_cache"], table, lens2,
                 "replay after in-place change")
    ref_o, ref_l = direct(ex, torch, q, kc, vc, bt, cl)
    assert torch.equal(got_o, ref_o) and torch.equal(got_l, ref_l)
    assert ex.attn_get_device_status() == 0
    with pytest.raises(ValueError):
        graph.launch()


def test_capture_rejects_bad_arguments(env):
    torch, ex, dev = env
    inp = synth.decode_inputs_lens(62, np.array([20, 40], np.int32), 8, 2, 64, nan_tail=False)
    q, kc, vc = to_dev(inp["q"], dev), to_dev(inp["k_cache"], dev), to_dev(inp["v_cache"], dev)
    bt, cl = to_dev(inp["block_table"], dev), to_dev(inp["ctx_lens"], dev)
    small = torch.empty(16, device=dev, dtype=torch.uint8)
    with pytest.raises(ex.ExattnError):
        ex.attn_decode_graph_capture(q, kc, vc, bt, cl, workspace=small)
    graph, out, _ = ex.attn_decode_graph_capture(q, kc, vc, bt, cl)
    graph.launch()
    torch.cuda.synchronize()
    graph.close()
    ref_o, _ = direct(ex, torch, q, kc, vc, bt, cl)
    assert torch.equal(out, ref_o)
