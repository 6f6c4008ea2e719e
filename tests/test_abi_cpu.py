"""The C-ABI library on a host without a GPU: it builds, loads, exports every
function include/exattn.h declares, and rejects bad arguments on the host
before any CUDA call (so none of these calls touches a device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "exattn.h")


@pytest.fixture(scope="module")
def lib():
    from exact_attention_40_gb300 import build
    build.build()
    from exact_attention_40_gb300 import exattn
    return exattn


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("attn_fwd", "attn_decode_paged", "attn_decode_workspace_bytes",
                     "attn_get_device_status", "attn_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(so, name), name


def test_status_strings(lib):
    for code, name in enumerate(["EXATTN_OK", "EXATTN_ERR_INVALID_ARG", "EXATTN_ERR_UNSUPPORTED",
                                 "EXATTN_ERR_ALIGNMENT", "EXATTN_ERR_WORKSPACE", "EXATTN_ERR_CUDA",
                                 "EXATTN_ERR_TIMEOUT", "EXATTN_ERR_DEVICE_BOUNDS"]):
        assert lib.attn_status_string(code) == name
    assert lib.attn_status_string(99) == "EXATTN_UNKNOWN_STATUS"


def test_workspace_arithmetic(lib):
    split = lib.attn_decode_split_tokens()
    assert split == 512 and split % 16 == 0
    # 64 seqs, 32 heads, d=128, up to 512 blocks (8192 tokens) -> 16 splits
    n = lib.attn_decode_workspace_bytes(64, 32, 128, 512, 16)
    rows = 64 * 32 * 16
    assert n == rows * 128 * 4 + ((rows * 4 + 15) // 16) * 16
    assert lib.attn_decode_workspace_bytes(1, 1, 64, 1, 16) == 64 * 4 + 16
    assert lib.attn_decode_workspace_bytes(1, 1, 96, 1, 16) == 0  # unsupported d
    assert lib.attn_decode_workspace_bytes(1, 1, 128, 1, 32) == 0  # unsupported block size


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def fwd(lib, q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=None, B=1, Hq=2, Hkv=1, Nq=8, Nk=8, d=128,
        scale=0.1, causal=0):
    return lib.lib.attn_fwd(q, k, v, out, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, None)


def test_fwd_rejections(lib):
    assert fwd(lib, d=96) == 2
    assert fwd(lib, Hq=3, Hkv=2) == 1
    assert fwd(lib, Hkv=0) == 1
    assert fwd(lib, Nq=-1) == 1
    assert fwd(lib, scale=0.0) == 1
    assert fwd(lib, scale=float("nan")) == 1
    assert fwd(lib, q=None) == 1
    assert fwd(lib, out=FAKE + 8) == 3
    assert fwd(lib, k=FAKE + 2) == 3
    assert fwd(lib, lse=FAKE + 2) == 3
    assert fwd(lib, Nq=(1 << 30) + 1) == 2
    assert fwd(lib, B=70000) == 2
    # empty problems are successful no-ops, even with null pointers
    assert fwd(lib, B=0, q=None, out=None) == 0
    assert fwd(lib, Nq=0, q=None, out=None) == 0


def dec(lib, ws_bytes=None, **kw):
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, cl=FAKE, out=FAKE, lse=None, S=2, Hq=8, Hkv=2,
             d=128, bs=16, nb=10, mb=4, scale=0.1, ws=FAKE)
    a.update(kw)
    if ws_bytes is None:
        ws_bytes = lib.attn_decode_workspace_bytes(a["S"], a["Hq"], a["d"], a["mb"], 16)
    return lib.lib.attn_decode_paged(a["q"], a["kc"], a["vc"], a["bt"], a["cl"], a["out"], a["lse"],
                                     a["S"], a["Hq"], a["Hkv"], a["d"], a["bs"], a["nb"], a["mb"],
                                     a["scale"], a["ws"], ws_bytes, None)


def test_decode_rejections(lib):
    assert dec(lib, bs=32) == 2
    assert dec(lib, d=80) == 2
    assert dec(lib, Hq=6, Hkv=4) == 1
    assert dec(lib, mb=0) == 1
    assert dec(lib, nb=0) == 1
    assert dec(lib, kc=None) == 1
    assert dec(lib, bt=FAKE + 2) == 3
    assert dec(lib, q=FAKE + 4) == 3
    assert dec(lib, ws=None) == 4
    assert dec(lib, ws_bytes=16) == 4
    assert dec(lib, ws=FAKE + 4) == 3
    assert dec(lib, S=0, q=None) == 0
    assert dec(lib, S=70000) == 2


def dec_static(lib, **kw):
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, cl=FAKE, out=FAKE, lse=None, S=2, Hq=8, Hkv=2,
             d=128, bs=16, nb=10, mb=4, scale=0.1)
    a.update(kw)
    return lib.lib.attn_decode_paged_static(a["q"], a["kc"], a["vc"], a["bt"], a["cl"], a["out"],
                                            a["lse"], a["S"], a["Hq"], a["Hkv"], a["d"], a["bs"],
                                            a["nb"], a["mb"], a["scale"], None)


def test_decode_static_rejections_before_any_cuda_call(lib):
    # the same host checks as attn_decode_paged, run before the scratch
    # array's address is looked up (no GPU here: a CUDA call would fail with
    # EXATTN_ERR_CUDA instead)
    assert dec_static(lib, bs=32) == 2
    assert dec_static(lib, d=80) == 2
    assert dec_static(lib, Hq=6, Hkv=4) == 1
    assert dec_static(lib, mb=0) == 1
    assert dec_static(lib, nb=0) == 1
    assert dec_static(lib, scale=0.0) == 1
    assert dec_static(lib, kc=None) == 1
    assert dec_static(lib, bt=FAKE + 2) == 3
    assert dec_static(lib, q=FAKE + 4) == 3
    assert dec_static(lib, S=70000) == 2
    assert dec_static(lib, S=0, q=None) == 0
    # more scratch than the static array holds
    assert lib.attn_decode_workspace_bytes(4096, 64, 128, 512) > 32 * 2 ** 20
    assert dec_static(lib, S=4096, Hq=64, Hkv=8, mb=512) == 4


def test_device_status_needs_an_output(lib):
    assert lib.lib.attn_get_device_status(None, None) == 1


def test_debug_wait_budget_validated(lib):
    assert lib.lib.attn_debug_expire_wait(0, None) == 1
    assert lib.lib.attn_debug_expire_wait(10 ** 11, None) == 1


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """The binding has no fallback: without libexattn.so, importing it raises."""
    import importlib.util
    src = os.path.join(ROOT, "exact_attention_40_gb300", "exattn.py")
    dst = tmp_path / "exattn.py"
    dst.write_text(open(src).read())
    spec = importlib.util.spec_from_file_location("exattn_copy", str(dst))
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


def norm(lib, x=FAKE, r=FAKE + 16, w=FAKE + 32, out=FAKE + 48, h=FAKE + 64, rows=4, hidden=64,
         eps=1e-6):
    return lib.lib.attn_add_rms_norm(x, r, w, out, h, rows, hidden, eps, None)


def test_add_rms_norm_rejections(lib):
    assert norm(lib, hidden=12) == 2
    assert norm(lib, hidden=16392) == 2
    assert norm(lib, hidden=0) == 1
    assert norm(lib, rows=-1) == 1
    assert norm(lib, eps=-1.0) == 1
    assert norm(lib, eps=float("nan")) == 1
    assert norm(lib, eps=float("inf")) == 1
    assert norm(lib, x=None) == 1
    assert norm(lib, h=None) == 1
    assert norm(lib, out=FAKE + 48, h=FAKE + 48) == 1   # both outputs in one buffer
    assert norm(lib, out=FAKE + 32) == 1                # output over the weight
    assert norm(lib, r=FAKE + 8) == 3
    assert norm(lib, out=FAKE + 50) == 3
    # nothing to do: success without touching the (null) pointers
    assert norm(lib, rows=0, x=None, r=None, w=None, out=None, h=None) == 0


def rope(lib, q=FAKE, k=FAKE + 16, v=FAKE + 32, sid=FAKE + 48, pos=FAKE + 64, bt=FAKE + 80,
         kc=FAKE + 96, vc=FAKE + 112, T=4, Hq=8, Hkv=2, d=128, S=2, nb=10, mb=4, base=500000.0):
    return lib.lib.attn_rope_cache_write(q, k, v, sid, pos, bt, kc, vc, T, Hq, Hkv, d, S, nb, mb,
                                         base, None)


def test_rope_cache_write_rejections(lib):
    assert rope(lib, d=24) == 2
    assert rope(lib, d=272) == 2
    assert rope(lib, d=8) == 2
    assert rope(lib, T=-1) == 1
    assert rope(lib, Hkv=0) == 1
    assert rope(lib, S=0) == 1
    assert rope(lib, nb=0) == 1
    assert rope(lib, mb=0) == 1
    assert rope(lib, base=1.0) == 1
    assert rope(lib, base=float("nan")) == 1
    assert rope(lib, q=None) == 1
    assert rope(lib, bt=None) == 1
    assert rope(lib, kc=FAKE + 96, vc=FAKE + 96) == 1
    assert rope(lib, k=FAKE + 8) == 3
    assert rope(lib, pos=FAKE + 2) == 3
    assert rope(lib, T=0, q=None, k=None, v=None, sid=None, pos=None, bt=None, kc=None, vc=None) == 0


def test_rope_cache_write_head_limit(lib):
    # (Hq + 3 Hkv) * d / 16 <= 2048 work items per token
    assert rope(lib, Hq=1024, Hkv=8, d=128) == 2
    assert rope(lib, Hq=8, Hkv=1024, d=16) == 2


def test_graph_calls_validate_on_the_host(lib):
    h = ctypes.c_void_p()
    so = lib.lib
    # bad arguments are rejected before any capture starts
    assert so.attn_decode_graph_capture(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 2, 128, 32, 10,
                                        4, 0.1, FAKE, 1 << 20, ctypes.byref(h)) in (1, 2)
    assert so.attn_decode_graph_capture(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, 8, 2, 128, 16, 10,
                                        4, 0.1, FAKE, 1 << 20, ctypes.byref(h)) == 1
    assert so.attn_decode_graph_capture(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 2, 128, 16, 10,
                                        4, 0.1, FAKE, 1 << 20, None) == 1
    assert not h.value
    assert so.attn_graph_launch(None, None) == 1
    assert so.attn_graph_destroy(None) == 0


def bwd(lib, q=FAKE, k=FAKE, v=FAKE, out=FAKE, do=FAKE, lse=FAKE, dq=FAKE + 16, dk=FAKE + 32,
        dv=FAKE + 48, B=1, Hq=2, Hkv=1, Nq=8, Nk=8, d=128, scale=0.1, causal=1, ws=FAKE + 64,
        ws_bytes=1 << 20):
    return lib.lib.attn_bwd(q, k, v, out, do, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, scale, causal, ws,
                            ws_bytes, None)


def test_bwd_rejections_and_workspace(lib):
    # fp32 (lse * log2 e, D) pairs per query row, rows padded to an even count
    assert lib.lib.attn_bwd_workspace_bytes(2, 4, 4, 10, 7, 64) == 2 * 4 * 10 * 8
    assert lib.lib.attn_bwd_workspace_bytes(1, 1, 1, 3, 5, 128) == 4 * 8
    # query heads sharing a KV head: fp32 dK, dV partials per query head, from a
    # 32-byte boundary of a 16-byte aligned workspace (16 bytes of slack)
    assert lib.lib.attn_bwd_workspace_bytes(1, 4, 2, 8, 6, 64) == 4 * 8 * 8 + 4 * 6 * 64 * 4 * 2 + 16
    assert lib.lib.attn_bwd_workspace_bytes(1, 4, 3, 8, 6, 64) == 0
    assert bwd(lib, d=96) == 2
    assert bwd(lib, Hq=3, Hkv=2) == 1
    assert bwd(lib, scale=-1.0) == 1
    assert bwd(lib, lse=None) == 1
    assert bwd(lib, dk=None) == 1
    assert bwd(lib, dq=FAKE + 8) == 3
    assert bwd(lib, lse=FAKE + 2) == 3
    assert bwd(lib, ws=None) == 4
    assert bwd(lib, ws_bytes=8) == 4
    assert bwd(lib, B=70000) == 2
    # 64-row blocks of a length index the second grid dimension
    assert bwd(lib, Nk=65535 * 64 + 1) == 2
    assert bwd(lib, Nq=65535 * 64 + 1) == 2
    # one-dimensional grids of 2^31 blocks or more
    assert bwd(lib, B=1, Hq=65535, Hkv=65535, Nq=65535 * 64, Nk=8) == 2
    assert bwd(lib, B=1, Hq=65535, Hkv=65535, Nq=8, Nk=65535 * 64) == 2
    assert bwd(lib, B=0, q=None) == 0
