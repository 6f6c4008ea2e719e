"""Calls from several host threads at once, each on its own CUDA stream.

The library keeps one host-side cache of tensor descriptors and the
per-device status word behind a mutex; the calls themselves are
asynchronous on the caller's stream.  Four threads run the forward and the
decode repeatedly on inputs of their own (different shapes, so their
descriptors differ) while the others do the same; every result must equal,
bit for bit, the one a single thread computes for the same inputs, and the
device status word must stay clear."""
import threading

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


# (B, Hq, Hkv, N, d, causal) of each thread's prefill, and its decode lengths
CASES = [
    ((1, 8, 2, 384, 128, True), [17, 600, 1500]),
    ((2, 4, 4, 200, 64, False), [1, 512, 513]),
    ((1, 16, 2, 640, 128, True), [2048, 33]),
    ((3, 2, 1, 129, 64, True), [4096, 700, 90, 16]),
]


def make_inputs(torch, dev, i, case):
    (B, Hq, Hkv, N, d, causal), lens = case
    q, k, v = synth.prefill_inputs_shape(100 + i, B, Hq, Hkv, N, N, d)
    dinp = synth.decode_inputs_lens(200 + i, np.array(lens, np.int32), Hq, Hkv, d)
    dec = {key: to_dev(val, dev) for key, val in dinp.items()
           if key in ("q", "k_cache", "v_cache", "block_table", "ctx_lens")}
    return (to_dev(q, dev), to_dev(k, dev), to_dev(v, dev), causal), dec


def compute(ex, stream, fwd, dec):
    q, k, v, causal = fwd
    out, lse = ex.attn_fwd(q, k, v, causal=causal, stream=stream)
    dout, dlse = ex.attn_decode_paged(dec["q"], dec["k_cache"], dec["v_cache"], dec["block_table"],
                                      dec["ctx_lens"], stream=stream)
    return out, lse, dout, dlse


def test_threads_on_their_own_streams(env):
    torch, ex, dev = env
    inputs = [make_inputs(torch, dev, i, c) for i, c in enumerate(CASES)]
    # single-threaded results on the default stream
    ref = []
    for fwd, dec in inputs:
        ref.append([t.clone() for t in compute(ex, None, fwd, dec)])
    torch.cuda.synchronize()
    assert ex.attn_get_device_status() == 0

    errors = []
    results = [None] * len(CASES)
    start = threading.Barrier(len(CASES))

    def worker(i):
        try:
            torch.cuda.set_device(dev)
            s = torch.cuda.Stream()
            fwd, dec = inputs[i]
            start.wait()
            got = []
            with torch.cuda.stream(s):
                for _ in range(25):
                    got.append(compute(ex, s, fwd, dec))
            s.synchronize()
            results[i] = got
        except Exception as e:  # reported below, in the main thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(CASES))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert ex.attn_get_device_status() == 0
    for i, got in enumerate(results):
        for rep, outs in enumerate(got):
            for name, a, b in zip(("out", "lse", "decode out", "decode lse"), outs, ref[i]):
                assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                                   b.view(torch.int16) if b.dtype == torch.bfloat16 else b), (i, rep, name)
