"""CUDA-graph capture of the decode step: a replay runs exactly the kernels
attn_decode_paged launches, so it must reproduce a direct call bit for bit,
also after the inputs it was captured with change in place."""
import numpy as np
import pytest

from exact_attention_40_gb300 import synth
from helpers import to_dev

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


def test_replay_matches_direct_call(env):
    torch, ex, dev = env
    inp = synth.decode_inputs_lens(60, np.array([1, 100, 700, 1600, 33], np.int32), 32, 8, 128,
                                   nan_tail=False)
    q, kc, vc = to_dev(inp["q"], dev), to_dev(inp["k_cache"], dev), to_dev(inp["v_cache"], dev)
    bt, cl = to_dev(inp["block_table"], dev), to_dev(inp["ctx_lens"], dev)
    ref_o, ref_l = direct(ex, torch, q, kc, vc, bt, cl)
    graph, out, lse = ex.attn_decode_graph_capture(q, kc, vc, bt, cl)
    with graph:
        torch.cuda.synchronize()
        for _ in range(3):
            out.zero_()
            lse.zero_()
            graph.launch()
            torch.cuda.synchronize()
            assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)

        # new contents in the captured buffers: another query, shorter
        # contexts, table entries remapped onto other blocks
        q.copy_(to_dev(synth.normal_bf16(61, 0, tuple(q.shape)), dev))
        cl.copy_(torch.tensor([1, 50, 512, 1599, 17], dtype=torch.int32, device=dev))
        table = inp["block_table"].copy()
        table[2, :4] = table[3, :4]
        bt.copy_(to_dev(table, dev))
        graph.launch()
        torch.cuda.synchronize()
        got_o, got_l = out.clone(), lse.clone()
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
