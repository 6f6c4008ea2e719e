"""Attention backward parity: dQ, dK, dV from the CUDA kernels (through the
C ABI, fed with the CUDA forward's O and LSE as a training step would be)
against the fp64 oracle, which computes them from Q, K, V and dO alone.

Bar, derived from the arithmetic: the products run on bf16 operands with
fp32 accumulation; P and dS are rounded to bf16 (relative 2^-9) before the
dV, dK and dQ products, D comes from the bf16 forward output, and each
result is rounded to bf16 once.  Each rounding contributes about 2^-9
(2e-3) relative, independently per term, so the sums' relative RMS error
stays near 2^-9 and the forward's bar applies: each gradient must satisfy
rel-RMS = ||g - ref|| / ||ref|| <= 5e-3 and max |g - ref| <= 2e-2 max |ref|
+ 1e-4 (about ten rounding units at the largest entry).  The absolute 1e-4 covers entries whose exact value is 0 while the
kernel's is not: with D taken from the bf16 O, dP - D keeps a residue of
about 2^-9 |dO| |v| where it is exactly zero (a row with one visible key)."""
import numpy as np
import pytest

from exact_attention_40_gb300 import synth
from helpers import to_dev

pytestmark = pytest.mark.gpu

REL_RMS = 5e-3
MAX_REL = 2e-2
MAX_ABS = 1e-4


@pytest.fixture(scope="module")
def env(oracle_mod):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_40_gb300 import build
    build.build()
    from exact_attention_40_gb300 import exattn
    return torch, exattn, oracle_mod, torch.device("cuda:0")


def check(got, ref, label):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), label
    err = np.abs(g - ref)
    den = float(np.sqrt((ref ** 2).sum()))
    rel = float(np.sqrt((err ** 2).sum())) / den if den > 0 else float(err.max())
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    assert rel <= REL_RMS, "%s: rel_rms %.3e" % (label, rel)
    assert float(err.max(initial=0.0)) <= MAX_REL * scale + MAX_ABS, "%s: max err %.3e of %.3e" % (
        label, float(err.max()), scale)
    print("%s: rel_rms %.2e, max err %.2e of %.2e" % (label, rel, float(err.max(initial=0.0)), scale))
    return rel


def run(env, seed, B, Hq, Hkv, Nq, Nk, d, causal):
    torch, ex, oracle, dev = env
    q = synth.normal_bf16(seed, 0, (B, Hq, Nq, d))
    k = synth.normal_bf16(seed, 1, (B, Hkv, Nk, d))
    v = synth.normal_bf16(seed, 2, (B, Hkv, Nk, d))
    do = synth.normal_bf16(seed, 3, (B, Hq, Nq, d))
    qd, kd, vd, dod = to_dev(q, dev), to_dev(k, dev), to_dev(v, dev), to_dev(do, dev)
    scale = d ** -0.5
    out, lse = ex.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = ex.attn_bwd(qd, kd, vd, out, dod, lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ex.attn_get_device_status() == 0
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, scale, causal)
    label = "B%d Hq%d Hkv%d Nq%d Nk%d d%d %s" % (B, Hq, Hkv, Nq, Nk, d, "causal" if causal else "full")
    return [check(dq, rq, label + " dq"), check(dk, rk, label + " dk"), check(dv, rv, label + " dv")]


def test_tiny(env):
    run(env, 80, 1, 2, 2, 128, 128, 64, False)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_gqa_ragged(env, d, causal):
    # 200 rows: three full 64-row tiles and a tail of 8
    run(env, 81, 1, 4, 2, 200, 200, d, causal)


@pytest.mark.parametrize("Nq,Nk", [(96, 160), (160, 96), (1, 130), (130, 1)])
def test_unequal_lengths(env, Nq, Nk):
    # bottom-right causal mask; Nq > Nk leaves the first rows without keys
    run(env, 82, 2, 2, 1, Nq, Nk, 128, True)


@pytest.mark.parametrize("causal", [False, True])
def test_odd_lengths(env, causal):
    # odd Nq: the per-row (lse, D) pairs of each head sit in rows padded to an even count
    run(env, 84, 2, 4, 2, 77, 93, 64, causal)


def test_llama_heads_causal(env):
    # a quarter of the Llama-3-8B heads (8 query, 2 key/value) at 2048 tokens
    run(env, 83, 1, 8, 2, 2048, 2048, 128, True)


def test_rejects(env):
    torch, ex, _, dev = env
    x = torch.zeros((1, 2, 8, 96), device=dev, dtype=torch.bfloat16)
    lse = torch.zeros((1, 2, 8), device=dev, dtype=torch.float32)
    with pytest.raises(ex.ExattnError):
        ex.attn_bwd(x, x, x, x, x, lse)


@pytest.mark.parametrize("Nq,Nk", [(96, 160), (200, 130)])
def test_unequal_lengths_full(env, Nq, Nk):
    run(env, 84, 1, 4, 4, Nq, Nk, 64, False)


def test_empty_sides(env):
    """No keys: dQ = 0 (and nothing to write for dK, dV); no queries: dK = dV = 0."""
    torch, ex, _, dev = env
    q = to_dev(synth.normal_bf16(85, 0, (1, 2, 70, 128)), dev)
    k0 = torch.zeros((1, 2, 0, 128), device=dev, dtype=torch.bfloat16)
    out, lse = ex.attn_fwd(q, k0, k0)
    dq, dk, dv = ex.attn_bwd(q, k0, k0, out, q, lse)
    torch.cuda.synchronize()
    assert torch.all(dq == 0).item() and dk.numel() == 0 and dv.numel() == 0
    kv = to_dev(synth.normal_bf16(85, 1, (1, 2, 90, 128)), dev)
    q0 = torch.zeros((1, 2, 0, 128), device=dev, dtype=torch.bfloat16)
    lse0 = torch.zeros((1, 2, 0), device=dev, dtype=torch.float32)
    dq, dk, dv = ex.attn_bwd(q0, kv, kv, q0, q0, lse0)
    torch.cuda.synchronize()
    assert torch.all(dk == 0).item() and torch.all(dv == 0).item() and dq.numel() == 0
    assert ex.attn_get_device_status() == 0


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (6, 2), (2, 2), (32, 2)])
def test_group_sizes(env, Hq, Hkv):
    # groups of 8, 3 and 16 (fp32 partials and their sum in head order) and
    # 1 (dK, dV written directly)
    run(env, 86, 1, Hq, Hkv, 200, 200, 64, True)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,N", [(128, 256), (64, 192)])
def test_many_small_units(env, d, N, causal):
    # 256 (batch, head) planes of N rows: 512 units of one to four tiles in
    # each pass, so every CTA runs three or four unit changes (stationary
    # copies, D shares, dQ staging, accumulator hand-off) back to back; at
    # d = 64 with N = 192 each plane also ends in a half-filled 128-row tile
    run(env, 87, 8, 32, 8, N, N, d, causal)


def test_empty_units_between_others(env):
    # Nq - Nk = 256 under the bottom-right causal mask: the first two 128-row
    # query tiles of every plane see no key, so two thirds of the dQ pass's
    # 768 units are empty and sit between non-empty ones on the same CTA
    # (their copies, zero dQ and release run in the same protocol)
    run(env, 88, 8, 32, 8, 384, 128, 128, True)


@pytest.mark.parametrize("causal", [False, True])
def test_one_key_many_queries(env, causal):
    # 880 queries against one key: dQ units of one tile (or, causal, none
    # but the last row's), dK/dV units with seven (or one) query tiles
    run(env, 89, 4, 32, 8, 880, 1, 64, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_one_query_many_keys(env, causal):
    # one query against 4000 keys: 8192 dK/dV units of one query tile each,
    # about 54 a CTA, back to back
    run(env, 90, 8, 32, 8, 1, 4000, 128, causal)
