"""Failure path on the GPU without a fault: a bounded wait that runs out
reports a status bit and returns, and the context stays usable."""
import math
import time

import pytest

from exact_attention_40_gb300 import synth
from helpers import assert_parity, metrics, to_dev

pytestmark = pytest.mark.gpu


def test_expired_wait_sets_status_and_context_survives(oracle_mod):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_40_gb300 import build
    build.build()
    from exact_attention_40_gb300 import exattn as ex

    assert ex.attn_get_device_status() == 0
    t0 = time.time()
    ex.attn_debug_expire_wait(50_000_000)  # 50 ms budget on a barrier nothing completes
    status = ex.attn_get_device_status()
    dt = time.time() - t0
    assert status & ex.DEVICE_TIMEOUT_BIT
    assert 0.04 < dt < 5.0
    assert ex.attn_get_device_status() == 0  # reading clears it

    dev = torch.device("cuda:0")
    q, k, v = synth.prefill_inputs_shape(71, 1, 2, 2, 256, 256, 128)
    out, lse = ex.attn_fwd(to_dev(q, dev), to_dev(k, dev), to_dev(v, dev), causal=True)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_mod.attn(q, k, v, 1.0 / math.sqrt(128), True)
    assert_parity(metrics(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l), "after")
    assert ex.attn_get_device_status() == 0
