"""add_rms_norm parity: the CUDA kernel (through the C ABI) against the fp64
oracle on the same seeded inputs.

Bar, derived from the arithmetic: the kernel adds in fp32 (exact for two
bf16 values within 16 binades of each other), accumulates the mean of
squares in fp32 and rounds each output once to bf16, so
  * residual_out is x + residual rounded to bf16: it must equal the oracle's
    exact sum rounded to bf16 (nearest even), allowing one bf16 step where
    the fp32 sum itself was rounded;
  * out is within half a bf16 step (2^-8 relative) of the fp64 value plus
    fp32 reduction error: |out - ref| <= 4e-3 |ref| + 1e-5 per element; the
    relative RMS over the tensor has the same bound (rounding errors of a
    few elements need not average out)."""
import numpy as np
import pytest

from exact_attention_40_gb300 import synth
from helpers import to_dev

pytestmark = pytest.mark.gpu

REL_ELEM = 4e-3
ABS_ELEM = 1e-5
REL_RMS = 4e-3


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
    return t.contiguous().cpu().view(__import__("torch").int16).numpy().view(np.uint16)


def check(got_out, got_h, ref_out, ref_h, label):
    o = synth.bf16_bits_to_f32(got_out).astype(np.float64)
    assert np.all(np.isfinite(o)), label
    err = np.abs(o - ref_out)
    bad = err > REL_ELEM * np.abs(ref_out) + ABS_ELEM
    assert not bad.any(), "%s: %d elements off, worst %.3e at ref %.3e" % (
        label, int(bad.sum()), float(err.max()), float(ref_out.flat[int(err.argmax())]))
    den = float((ref_out ** 2).sum())
    if den > 0:
        rel = float(np.sqrt((err ** 2).sum() / den))
        assert rel <= REL_RMS, "%s: rel_rms %.3e" % (label, rel)
    want_h = synth.f32_to_bf16_bits(ref_h.astype(np.float32))
    steps = np.abs(got_h.astype(np.int32) - want_h.astype(np.int32))
    assert steps.max(initial=0) <= 1, "%s: residual off by %d bf16 steps" % (label, int(steps.max()))


def run(env, x, r, w, eps, **kw):
    torch, ex, _, dev = env
    out, h = ex.attn_add_rms_norm(to_dev(x, dev), to_dev(r, dev), to_dev(w, dev), eps, **kw)
    torch.cuda.synchronize()
    assert ex.attn_get_device_status() == 0
    return bits(out), bits(h)


def test_page_shape_64x8192(env):
    cfg = synth.NORM["rmsnorm_64x8192"]
    x, r, w = synth.norm_inputs(cfg)
    got_o, got_h = run(env, x, r, w, cfg.eps)
    ref_o, ref_h = env[2].add_rms_norm(x, r, w, cfg.eps)
    check(got_o, got_h, ref_o, ref_h, cfg.name)
    # in practice the residual is bit-exact
    assert np.array_equal(got_h, synth.f32_to_bf16_bits(ref_h.astype(np.float32)))


@pytest.mark.parametrize("rows,hidden", [(1, 8), (3, 24), (7, 2048), (5, 2056), (257, 4096),
                                         (2, 16384), (3, 12296), (1500, 1024)])
def test_shapes(env, rows, hidden):
    # 8 and 24: a single partial warp; 2056 and 12296: vectors past a
    # multiple of the CTA (ragged tail); 16384: the largest row; 1500 rows:
    # more rows than resident CTAs (grid-stride loop)
    x, r, w = synth.norm_inputs_shape(20 + rows % 7, rows, hidden)
    got_o, got_h = run(env, x, r, w, 1e-6)
    ref_o, ref_h = env[2].add_rms_norm(x, r, w, 1e-6)
    check(got_o, got_h, ref_o, ref_h, "%dx%d" % (rows, hidden))


def test_large_batch_sampled_rows(env):
    # the 16384 x 8192 batch the bench streams: every row is independent, so
    # the oracle checks a seeded sample of rows
    cfg = synth.NORM["rmsnorm_16384x8192"]
    x, r, w = synth.norm_inputs(cfg)
    got_o, got_h = run(env, x, r, w, cfg.eps)
    rows = np.sort(synth.permutation(cfg.seed, cfg.rows)[:96])
    ref_o, ref_h = env[2].add_rms_norm(x[rows], r[rows], w, cfg.eps)
    check(got_o[rows], got_h[rows], ref_o, ref_h, "sampled rows")


def test_in_place(env):
    torch, ex, oracle, dev = env
    x, r, w = synth.norm_inputs_shape(31, 33, 4096)
    xd, rd, wd = to_dev(x, dev), to_dev(r, dev), to_dev(w, dev)
    out, h = ex.attn_add_rms_norm(xd, rd, wd, 1e-5, out=xd, residual_out=rd)
    torch.cuda.synchronize()
    assert out.data_ptr() == xd.data_ptr() and h.data_ptr() == rd.data_ptr()
    ref_o, ref_h = oracle.add_rms_norm(x, r, w, 1e-5)
    check(bits(xd), bits(rd), ref_o, ref_h, "in place")


def test_special_rows(env):
    # a zero row, a constant row, a row with one large value, large eps
    D = 256
    x = np.zeros((4, D), np.uint16)
    r = np.zeros((4, D), np.uint16)
    x[1, :] = synth.f32_to_bf16_bits(np.full(D, 3.0, np.float32))
    x[2, 17] = synth.f32_to_bf16_bits(np.array([1000.0], np.float32))[0]
    x[3], r[3] = synth.normal_bf16(40, 0, (D,)), synth.normal_bf16(40, 1, (D,))
    w = synth.norm_inputs_shape(41, 1, D)[2]
    for eps in (1e-6, 1.0):
        got_o, got_h = run(env, x, r, w, eps)
        ref_o, ref_h = env[2].add_rms_norm(x, r, w, eps)
        check(got_o, got_h, ref_o, ref_h, "special rows eps=%g" % eps)
        assert not got_o[0].any()


def test_empty_and_rejected(env):
    torch, ex, _, dev = env
    x = torch.zeros((0, 64), device=dev, dtype=torch.bfloat16)
    w = torch.ones(64, device=dev, dtype=torch.bfloat16)
    out, h = ex.attn_add_rms_norm(x, x.clone(), w)
    assert out.shape == (0, 64) and h.shape == (0, 64)
    y = torch.zeros((2, 12), device=dev, dtype=torch.bfloat16)
    with pytest.raises(ex.ExattnError):
        ex.attn_add_rms_norm(y, y.clone(), torch.ones(12, device=dev, dtype=torch.bfloat16))
    z = torch.zeros((2, 64), device=dev, dtype=torch.bfloat16)
    o = torch.empty_like(z)
    with pytest.raises(ex.ExattnError):
        ex.attn_add_rms_norm(z, z.clone(), w, out=o, residual_out=o)
    torch.cuda.synchronize()
    assert ex.attn_get_device_status() == 0
