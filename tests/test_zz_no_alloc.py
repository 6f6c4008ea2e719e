"""attn_decode_paged_static: the decode entry point for callers that cannot
allocate device memory (for instance a plugin inside a server whose own
pool owns all device memory, or a decode loop that may not pay cudaMalloc's
implicit synchronisation).  Its split-KV scratch is a static device array
inside the library instead of a caller workspace.

Called through the C ABI with raw pointers, its output must match the
workspace entry point's on two calls in a row (different inputs, so stale
scratch from the first call cannot leak into the second), and a request
beyond the static array's size must be rejected without a launch.  This
file is collected last so that a failure here stops a run only after every
other test has run.
"""
import ctypes
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
    torch.cuda.set_device(0)
    return torch, exattn, torch.device("cuda:0")


def _dev_inputs(torch, inp, dev):
    return {k: to_dev(v, dev) for k, v in inp.items()}


def _call_static(ex, t, out, lse, Hq, Hkv, d, stream):
    nb, _, bs, _ = t["k_cache"].shape
    S, mb = t["block_table"].shape
    return ex.lib.attn_decode_paged_static(
        t["q"].data_ptr(), t["k_cache"].data_ptr(), t["v_cache"].data_ptr(),
        t["block_table"].data_ptr(), t["ctx_lens"].data_ptr(), out.data_ptr(), lse.data_ptr(),
        S, Hq, Hkv, d, bs, nb, mb, ctypes.c_float(1.0 / math.sqrt(d)), stream)


def _call_workspace(ex, torch, t, out, lse, Hq, Hkv, d, dev, stream):
    nb, _, bs, _ = t["k_cache"].shape
    S, mb = t["block_table"].shape
    need = ex.attn_decode_workspace_bytes(S, Hq, d, mb, bs)
    ws = torch.empty(need, device=dev, dtype=torch.uint8)
    rc = ex.lib.attn_decode_paged(
        t["q"].data_ptr(), t["k_cache"].data_ptr(), t["v_cache"].data_ptr(),
        t["block_table"].data_ptr(), t["ctx_lens"].data_ptr(), out.data_ptr(), lse.data_ptr(),
        S, Hq, Hkv, d, bs, nb, mb, ctypes.c_float(1.0 / math.sqrt(d)), ws.data_ptr(), need, stream)
    return rc, ws


def test_static_scratch_matches_workspace_entry_point(env):
    torch, ex, dev = env
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [
        # the full paged-decode workload, then a different mix of lengths
        (synth.decode_inputs(synth.DECODE["decode_paged"]), 32, 8, 128),
        (synth.decode_inputs_lens(81, np.array([1, 600, 17, 5000, 0, 2048], np.int32), 16, 4, 128),
         16, 4, 128),
    ]
    for i, (inp, Hq, Hkv, d) in enumerate(cases):
        t = _dev_inputs(torch, inp, dev)
        S = inp["q"].shape[0]
        out_s = torch.empty((S, Hq, d), device=dev, dtype=torch.bfloat16)
        lse_s = torch.empty((S, Hq), device=dev, dtype=torch.float32)
        out_w, lse_w = torch.empty_like(out_s), torch.empty_like(lse_s)
        assert _call_static(ex, t, out_s, lse_s, Hq, Hkv, d, stream) == 0
        rc, ws = _call_workspace(ex, torch, t, out_w, lse_w, Hq, Hkv, d, dev, stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert ex.attn_get_device_status() == 0
        # the same kernels on the same inputs: bit for bit, so no stale
        # scratch of the previous call can hide under a tolerance
        assert torch.equal(out_s.view(torch.int16), out_w.view(torch.int16)), "static call %d" % (i + 1)
        assert torch.equal(lse_s, lse_w), "static call %d" % (i + 1)
        ref_o = out_w.double().cpu().numpy()
        ref_l = lse_w.double().cpu().numpy()
        m = metrics(out_s.float().cpu().numpy(), lse_s.cpu().numpy(), ref_o, ref_l)
        assert_parity(m, "static call %d" % (i + 1))


def test_static_scratch_rejects_oversize_request(env):
    torch, ex, dev = env
    # 4096 sequences x 64 heads x 8192-token tables need far more than the
    # static array holds: rejected before anything is launched.
    need = ex.attn_decode_workspace_bytes(4096, 64, 128, 512)
    assert need > 32 * 2 ** 20
    rc = ex.lib.attn_decode_paged_static(16, 16, 16, 16, 16, 16, None, 4096, 64, 8, 128, 16, 1,
                                         512, ctypes.c_float(0.1), None)
    assert rc == 4  # EXATTN_ERR_WORKSPACE
