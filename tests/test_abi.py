"""The C ABI on the host (CPU only, no GPU needed).

Loads libcarat.so, checks that it exports every function include/carat.h
declares, and exercises the host-side argument checks: every call here fails
validation, which happens before any CUDA call, so nothing touches a device.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "carat.h")


@pytest.fixture(scope="module")
def lib():
    from sliding_window_gqa_ring_gb300 import build, carat
    if not os.path.exists(carat.LIBRARY):
        build.build()
    return carat.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(carat_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_entry_points():
    names = declared_functions()
    for n in ("carat_ring_append", "carat_swa_attention", "carat_global_verify_attention"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from sliding_window_gqa_ring_gb300 import carat
    names = declared_functions()
    assert set(carat.EXPORTED) <= set(names) | {"carat_abi_version"}
    for n in names:
        assert hasattr(lib, n), f"{n} declared in carat.h but not exported"


def test_abi_version(lib):
    assert lib.carat_abi_version() == 1


def test_status_strings(lib):
    for code in range(5):
        assert lib.carat_status_string(code)
    assert lib.carat_status_string(99) == b"unknown status"


def test_workspace_queries(lib):
    # Tensor-core path: two partial slots (rows per tile x head_dim floats, and
    # a (max, sum) pair per row) for each CTA of the persistent grid -- two
    # CTAs per SM for 16-row tiles at head_dim 256, 152 SMs when no GPU is
    # present -- plus one 16-byte merge entry per (request, KV head, row group)
    # and 256 bytes for unit mode's work counter.
    def a256(x):
        return (x + 255) // 256 * 256

    import torch
    sms = (torch.cuda.get_device_properties(0).multi_processor_count
           if torch.cuda.is_available() else 152)

    def expected(batch, rows_per_tile, head_dim, ctas_per_sm, units_per_request):
        slots = ctas_per_sm * sms * 2 * rows_per_tile
        return (a256(slots * 8) + a256(slots * head_dim * 4)
                + a256(batch * units_per_request * 16) + 256)

    assert lib.carat_swa_workspace_bytes(56, 1, 16, 8, 256, 1024) == expected(56, 16, 256, 2, 8)
    assert lib.carat_swa_workspace_bytes(1, 1, 16, 8, 256, 1024) == expected(1, 16, 256, 2, 8)
    # 8 query heads per KV head x 15 proposals: 64-row tiles, two row groups
    assert (lib.carat_global_workspace_bytes(8, 15, 16, 2, 512, 32768)
            == expected(8, 64, 512, 1, 2 * 2))
    assert lib.carat_swa_workspace_bytes(0, 1, 16, 8, 256, 1024) == 0
    assert lib.carat_swa_workspace_bytes(1, 1, 16, 8, 128, 1024) == 0       # unsupported D
    assert lib.carat_global_workspace_bytes(1, 17, 16, 2, 512, 1024) == 0   # too many proposals
    assert lib.carat_global_workspace_bytes(1, 16, 16, 1, 512, 1024) == 0   # 256 rows > 128
    assert lib.carat_swa_workspace_bytes(1, 1, 128, 1, 256, 1024) == 0      # 128 heads per KV head
    # monotone in batch
    a = lib.carat_global_workspace_bytes(4, 4, 16, 2, 512, 8192)
    b = lib.carat_global_workspace_bytes(8, 4, 16, 2, 512, 8192)
    assert b >= a


FAKE = 0x10000          # aligned, never dereferenced: every call below fails validation
MISALIGNED = 0x10008


def _swa(lib, **kw):
    a = dict(out=FAKE, q=FAKE, kr=FAKE, vr=FAKE, nr=4, ids=None, disp=FAKE, ctx=FAKE, k=1, B=4,
             hq=16, hkv=8, d=256, w=1024, scale=0.0625, ws=FAKE, wsb=0, stream=None)
    a.update(kw)
    return lib.carat_swa_attention(a["out"], a["q"], a["kr"], a["vr"], a["nr"], a["ids"],
                                   a["disp"], a["ctx"], a["k"], a["B"], a["hq"], a["hkv"], a["d"],
                                   a["w"], a["scale"], a["ws"], a["wsb"], a["stream"])


def _glob(lib, **kw):
    a = dict(out=FAKE, q=FAKE, kc=FAKE, vc=FAKE, nc=4, ids=None, ctx=FAKE, k=4, B=4, hq=16, hkv=2,
             d=512, cap=8192, scale=0.04, ws=FAKE, wsb=0, stream=None)
    a.update(kw)
    return lib.carat_global_verify_attention(a["out"], a["q"], a["kc"], a["vc"], a["nc"], a["ids"],
                                             a["ctx"], a["k"], a["B"], a["hq"], a["hkv"], a["d"],
                                             a["cap"], a["scale"], a["ws"], a["wsb"], a["stream"])


def _app(lib, **kw):
    a = dict(kr=FAKE, vr=FAKE, nr=4, ids=None, kn=FAKE, vn=FAKE, ctx=FAKE, k=1, disp=None, B=4,
             hkv=8, d=256, w=1024, stream=None)
    a.update(kw)
    return lib.carat_ring_append(a["kr"], a["vr"], a["nr"], a["ids"], a["kn"], a["vn"], a["ctx"],
                                 a["k"], a["disp"], a["B"], a["hkv"], a["d"], a["w"], a["stream"])


def test_swa_argument_checks(lib):
    from sliding_window_gqa_ring_gb300 import carat as c
    assert _swa(lib, B=-1) == c.CARAT_ERR_INVALID_ARG
    assert _swa(lib, out=None) == c.CARAT_ERR_INVALID_ARG
    assert _swa(lib, q=MISALIGNED) == c.CARAT_ERR_INVALID_ARG
    assert _swa(lib, hq=12, hkv=8) == c.CARAT_ERR_INVALID_ARG        # not a multiple
    assert _swa(lib, d=128) == c.CARAT_ERR_UNSUPPORTED
    assert _swa(lib, k=17) == c.CARAT_ERR_INVALID_ARG
    assert _swa(lib, k=4, disp=None) == c.CARAT_ERR_INVALID_ARG       # k > 1 needs displaced
    assert _swa(lib, k=5, w=4) == c.CARAT_ERR_INVALID_ARG             # k > window
    assert _swa(lib, nr=2) == c.CARAT_ERR_INVALID_ARG                 # fewer rings than requests
    assert _swa(lib, scale=float("nan")) == c.CARAT_ERR_INVALID_ARG
    assert _swa(lib, hq=64, hkv=1, k=4) == c.CARAT_ERR_UNSUPPORTED    # 256 rows per tile
    assert _swa(lib, hq=128, hkv=1, k=1) == c.CARAT_ERR_UNSUPPORTED   # > 64 heads per KV head
    assert _swa(lib, wsb=16) == c.CARAT_ERR_WORKSPACE
    assert _swa(lib, ws=None, wsb=1 << 30) == c.CARAT_ERR_WORKSPACE
    assert _swa(lib, B=0) == c.CARAT_OK                               # empty batch: no launch


def test_global_argument_checks(lib):
    from sliding_window_gqa_ring_gb300 import carat as c
    assert _glob(lib, cap=3) == c.CARAT_ERR_INVALID_ARG               # capacity < proposals
    assert _glob(lib, kc=None) == c.CARAT_ERR_INVALID_ARG
    assert _glob(lib, vc=MISALIGNED) == c.CARAT_ERR_INVALID_ARG
    assert _glob(lib, d=64) == c.CARAT_ERR_UNSUPPORTED
    assert _glob(lib, k=15, hq=32, hkv=2) == c.CARAT_ERR_UNSUPPORTED  # 240 rows
    assert _glob(lib, k=1, hq=128, hkv=1) == c.CARAT_ERR_UNSUPPORTED  # > 64 heads per KV head
    assert _glob(lib, wsb=1024) == c.CARAT_ERR_WORKSPACE
    assert _glob(lib, B=0) == c.CARAT_OK


def test_append_argument_checks(lib):
    from sliding_window_gqa_ring_gb300 import carat as c
    assert _app(lib, k=0) == c.CARAT_ERR_INVALID_ARG
    assert _app(lib, k=1025) == c.CARAT_ERR_INVALID_ARG               # more rows than slots
    assert _app(lib, k=17, disp=FAKE) == c.CARAT_ERR_INVALID_ARG
    assert _app(lib, kn=MISALIGNED) == c.CARAT_ERR_INVALID_ARG
    assert _app(lib, hkv=1, d=4) == c.CARAT_ERR_INVALID_ARG           # 8-byte rows
    assert _app(lib, nr=0) == c.CARAT_ERR_INVALID_ARG
    assert _app(lib, ctx=None) == c.CARAT_ERR_INVALID_ARG
    assert _app(lib, B=0) == c.CARAT_OK


def test_rollback_argument_checks(lib):
    from sliding_window_gqa_ring_gb300 import carat as c

    def rb(**kw):
        a = dict(kr=FAKE, vr=FAKE, nr=4, ids=None, disp=FAKE, ctx=FAKE, acc=FAKE, k=4, B=4,
                 hkv=8, d=256, w=1024)
        a.update(kw)
        return lib.carat_ring_rollback(a["kr"], a["vr"], a["nr"], a["ids"], a["disp"], a["ctx"],
                                       a["acc"], a["k"], a["B"], a["hkv"], a["d"], a["w"], None)
    assert rb(k=1) == c.CARAT_ERR_INVALID_ARG          # nothing can be rejected
    assert rb(k=17) == c.CARAT_ERR_INVALID_ARG
    assert rb(disp=None) == c.CARAT_ERR_INVALID_ARG
    assert rb(acc=None) == c.CARAT_ERR_INVALID_ARG
    assert rb(kr=MISALIGNED) == c.CARAT_ERR_INVALID_ARG
    assert rb(B=0) == c.CARAT_OK


def test_device_status_needs_output_pointer(lib):
    from sliding_window_gqa_ring_gb300 import carat as c
    assert lib.carat_get_device_status(None, 0, None) == c.CARAT_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from sliding_window_gqa_ring_gb300 import carat
    monkeypatch.setattr(carat, "LIBRARY", str(tmp_path / "missing.so"))
    monkeypatch.setattr(carat, "_lib", None)
    with pytest.raises(carat.CaratError):
        carat.library()


def test_python_status_text_matches_library(lib):
    from sliding_window_gqa_ring_gb300 import carat
    for code in range(6):
        assert carat.status_string(code) == lib.carat_status_string(code).decode()


def test_binding_checks_caches_against_queries(lib):
    """The binding rejects caches whose element type, shape or head_dim does
    not match the queries before calling the library (the C ABI sees only
    pointers and sizes, so a kernel would read past such a buffer)."""
    import torch

    from sliding_window_gqa_ring_gb300 import carat
    q = torch.zeros((2, 1, 16, 256), dtype=torch.bfloat16)
    out = torch.zeros((2, 1, 16, 256), dtype=torch.float32)
    ctx = torch.zeros((2,), dtype=torch.int32)
    ring = torch.zeros((2, 1024, 8, 256), dtype=torch.bfloat16)
    ring8 = torch.zeros((2, 1024, 8, 256), dtype=torch.uint8)
    ring_d = torch.zeros((2, 1024, 8, 128), dtype=torch.bfloat16)
    ws = torch.zeros(256, dtype=torch.uint8)
    before = lib.carat_kernel_launches()
    for fn, kw in ((carat.carat_swa_attention, {"workspace": ws}),
                   (carat.carat_swa_attention_noalloc, {})):
        with pytest.raises(TypeError):
            fn(out, q, ring8, ring8, ctx, scale=0.0625, **kw)        # FP8 ring, bf16 kernel
        with pytest.raises(TypeError):
            fn(out, q, ring, ring8, ctx, scale=0.0625, **kw)         # K and V types differ
        with pytest.raises(ValueError):
            fn(out, q, ring_d, ring_d, ctx, scale=0.0625, **kw)      # head_dim 128 vs 256
        with pytest.raises(ValueError):
            fn(out[:1], q, ring, ring, ctx, scale=0.0625, **kw)      # out shape
        with pytest.raises(ValueError):
            fn(out, q, ring, ring, ctx[:1], scale=0.0625, **kw)      # context_lengths shape
    with pytest.raises(TypeError):
        carat.carat_swa_attention_fp8(out, q, ring, ring, ctx, scale=0.0625, k_scale=1.0,
                                      v_scale=1.0, workspace=ws)     # bf16 ring, FP8 kernel
    with pytest.raises(ValueError):
        carat.carat_global_verify_attention(out, q, ring_d, ring_d, ctx, scale=0.0625,
                                            workspace=ws)
    assert lib.carat_kernel_launches() == before
