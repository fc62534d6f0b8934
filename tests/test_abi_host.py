"""The C ABI without a GPU: the library loads, exports every entry point that
include/swa.h declares, and rejects bad arguments on the host before any CUDA
call (so these run on a machine with no GPU)."""

import ctypes
import os
import re

import pytest

from tests._lib import ROOT, ensure_built

HEADER = os.path.join(ROOT, "include", "swa.h")


@pytest.fixture(scope="module")
def swa():
    ensure_built()
    from sliding_window_gqa_swa_gb300 import swa as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^SWA_API\s+[\w\s\*]+?\b(swa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("swa_cache_alloc", "swa_prefill", "swa_compact", "swa_decode", "swa_roll", "swa_build_mask"):
        assert want in names


def test_every_declared_symbol_is_exported(swa):
    lib = ctypes.CDLL(swa.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) == set(swa.EXPORTED)


def test_version_and_status_strings(swa):
    assert swa.lib().swa_version() == 100
    assert swa.lib().swa_status_string(swa.ESTATE).decode() == "SWA_ESTATE"


def _desc(swa, **kw):
    d = dict(kind=swa.CACHE_COMPACT, layers=2, batch=3, kv_heads=2, head_dim=256, window=1024,
             prompt_len=8192, rows=0)
    d.update(kw)
    return swa.CacheDesc(*[d[k] for k in ("kind", "layers", "batch", "kv_heads", "head_dim", "window",
                                          "prompt_len", "rows")])


def test_cache_bytes(swa):
    d = _desc(swa)
    n = swa.lib().swa_cache_bytes(ctypes.byref(d))
    kv = 2 * 3 * 2 * 1088 * 256 * 2
    assert n >= 2 * kv and n - 2 * kv < 4096
    # a short prompt's prefill cache still gets W + 64 rows
    short = _desc(swa, kind=swa.CACHE_PREFILL, prompt_len=100)
    assert swa.lib().swa_cache_bytes(ctypes.byref(short)) == n
    for bad in (_desc(swa, head_dim=96), _desc(swa, window=32), _desc(swa, rows=1000), _desc(swa, layers=0),
                _desc(swa, kind=7), _desc(swa, kind=swa.CACHE_PREFILL, rows=10)):
        assert swa.lib().swa_cache_bytes(ctypes.byref(bad)) == 0
        assert swa.last_error()


def test_alloc_rejects_before_touching_the_device(swa):
    lib = swa.lib()
    out = ctypes.c_void_p()
    d = _desc(swa)
    assert lib.swa_cache_alloc(ctypes.byref(d), None, 1 << 30, None, None, ctypes.byref(out)) == swa.EINVAL
    assert "dev_mem" in swa.last_error()
    assert lib.swa_cache_alloc(ctypes.byref(d), ctypes.c_void_p(0x1000 + 16), 1 << 30, None, None,
                               ctypes.byref(out)) == swa.EINVAL
    assert "aligned" in swa.last_error()
    assert lib.swa_cache_alloc(ctypes.byref(d), ctypes.c_void_p(0x100000), 16, None, None,
                               ctypes.byref(out)) == swa.EINVAL
    assert "bytes" in swa.last_error()
    assert out.value is None


def test_calls_on_null_handles(swa):
    lib = swa.lib()
    assert lib.swa_roll(None, None) == swa.EINVAL
    assert lib.swa_compact(None, None, None) == swa.EINVAL
    assert lib.swa_cache_advance(None, 1) == swa.EINVAL
    assert lib.swa_build_mask(None, swa.MASK_DECODE, None, ctypes.c_void_p(0x1000), None) == swa.EINVAL
    assert lib.swa_build_mask(None, 9, None, ctypes.c_void_p(0x1000), None) == swa.EINVAL
    assert lib.swa_decode_workspace_bytes(None, 4) == 0
    lib.swa_cache_free(None)


def test_prefill_meta_validation(swa):
    lib = swa.lib()
    m = swa.PrefillMeta(2, 100, 90, 20, 16, 0, None, None, None, None)  # chunk past the end
    assert lib.swa_prefill_plan_bytes(ctypes.byref(m)) == 0
    m = swa.PrefillMeta(2, 100, 0, 100, 16, 0, None, None, None, None)
    assert lib.swa_prefill_plan_bytes(ctypes.byref(m)) > 0
    fake = ctypes.c_void_p(0x10000)
    # unsupported head size, bad mode, generic without plan, bad head ratio: rejected on the host
    assert lib.swa_prefill(None, 0, swa.MODE_CAUSAL, 4, 2, 128, ctypes.byref(m), fake, fake, fake, 1.0, fake,
                           None, None) == swa.EUNSUPPORTED
    assert lib.swa_prefill(None, 0, 5, 4, 2, 256, ctypes.byref(m), fake, fake, fake, 1.0, fake, None,
                           None) == swa.EINVAL
    assert lib.swa_prefill(None, 0, swa.MODE_GENERIC, 4, 2, 256, ctypes.byref(m), fake, fake, fake, 1.0, fake,
                           None, None) == swa.EINVAL
    assert "plan" in swa.last_error()
    assert lib.swa_prefill(None, 0, swa.MODE_CAUSAL, 3, 2, 256, ctypes.byref(m), fake, fake, fake, 1.0, fake,
                           None, None) == swa.EINVAL
    # packed documents with padding are unsupported
    m2 = swa.PrefillMeta(1, 100, 0, 100, 16, 2, fake, None, ctypes.c_void_p(0x20000), None)
    assert lib.swa_prefill_plan_bytes(ctypes.byref(m2)) == 0


def test_backward_workspace_and_validation(swa):
    lib = swa.lib()
    fake = ctypes.c_void_p(0x10000)
    plan = ctypes.c_void_p(0x40000)
    # packed documents 4 x 4096, W = 4096: 128 query tiles, a band of 1 + 32 key tiles
    cu = ctypes.c_void_p(0x20000)
    m = swa.PrefillMeta(1, 16384, 0, 16384, 4096, 4, None, None, cu, plan)
    n = lib.swa_prefill_backward_workspace_bytes(16, ctypes.byref(m))
    tiles = 16 * 128 * 33
    assert n == 16384 * 16 * 4 + 3 * tiles * 32768
    # a window of 1 key: one key tile per query tile; images: every key tile (the
    # delta array, 2 x 300 x 4 fp32, is rounded up to 256 bytes: 9728)
    m1 = swa.PrefillMeta(2, 300, 0, 300, 1, 0, None, None, None, plan)
    assert lib.swa_prefill_backward_workspace_bytes(4, ctypes.byref(m1)) == 9728 + 3 * 2 * 4 * 3 * 32768
    mi = swa.PrefillMeta(2, 300, 0, 300, 1, 0, None, ctypes.c_void_p(0x30000), None, plan)
    assert lib.swa_prefill_backward_workspace_bytes(4, ctypes.byref(mi)) == 9728 + 3 * 2 * 4 * 9 * 32768
    # chunks and a missing plan are rejected
    mc = swa.PrefillMeta(1, 300, 0, 200, 64, 0, None, None, None, plan)
    assert lib.swa_prefill_backward_workspace_bytes(4, ctypes.byref(mc)) == 0
    mp = swa.PrefillMeta(1, 300, 0, 300, 64, 0, None, None, None, None)
    assert lib.swa_prefill_backward_workspace_bytes(4, ctypes.byref(mp)) == 0
    assert "plan" in swa.last_error()

    def call(meta, hq=4, hkv=2, d=256, ws=fake, ws_bytes=1 << 40, lse=fake):
        return lib.swa_prefill_backward(hq, hkv, d, ctypes.byref(meta), fake, fake, fake, fake, fake, lse, 0.1,
                                        fake, fake, fake, ws, ws_bytes, None)

    m2 = swa.PrefillMeta(1, 300, 0, 300, 64, 0, None, None, None, plan)
    assert call(mc) == swa.EUNSUPPORTED
    assert call(mp) == swa.EINVAL
    assert call(m2, d=128) == swa.EUNSUPPORTED
    assert call(m2, hq=3) == swa.EINVAL
    assert call(m2, lse=None) == swa.EINVAL
    assert call(m2, ws=ctypes.c_void_p(0x10000 + 16)) == swa.EINVAL
    assert "256-byte" in swa.last_error()
    assert call(m2, ws_bytes=1000) == swa.EINVAL
    assert "workspace too small" in swa.last_error()


def test_degenerate_sizes_are_rejected_on_the_host(swa):
    lib = swa.lib()
    fake = ctypes.c_void_p(0x10000)
    plan = ctypes.c_void_p(0x40000)
    for b, s, c0, cl, w in [(1, 0, 0, 0, 16), (1, 100, 0, 0, 16), (0, 100, 0, 100, 16), (1, 100, 0, 100, 0),
                            (1, 100, 100, 1, 16), (1, 100, -1, 10, 16)]:
        m = swa.PrefillMeta(b, s, c0, cl, w, 0, None, None, None, plan)
        assert lib.swa_prefill_plan_bytes(ctypes.byref(m)) == 0
        assert lib.swa_prefill_backward_workspace_bytes(4, ctypes.byref(m)) == 0
        assert lib.swa_prefill(None, 0, swa.MODE_GENERIC, 4, 2, 256, ctypes.byref(m), fake, fake, fake, 1.0, fake,
                               None, None) == swa.EINVAL
        assert lib.swa_prefill_backward(4, 2, 256, ctypes.byref(m), fake, fake, fake, fake, fake, fake, 1.0, fake,
                                        fake, fake, fake, 1 << 40, None) == swa.EINVAL
    # a non-finite scale
    m = swa.PrefillMeta(1, 100, 0, 100, 16, 0, None, None, None, plan)
    assert lib.swa_prefill_backward(4, 2, 256, ctypes.byref(m), fake, fake, fake, fake, fake, fake, float("nan"),
                                    fake, fake, fake, fake, 1 << 40, None) == swa.EINVAL
    assert "scale" in swa.last_error()


def test_every_declaration_cites_its_source():
    """Each entry point's comment names the page passage that defines it, or
    says that it is library plumbing with no counterpart in the pages."""
    text = open(HEADER).read()
    blocks = re.findall(r"(/\*(?:[^*]|\*(?!/))*\*/)\s*\n(SWA_API[^;]*;)", text)
    names = set()
    for comment, decl in blocks:
        name = re.search(r"\b(swa_\w+)\s*\(", decl).group(1)
        names.add(name)
        assert re.search(r"\[SPYRE\]|\[FASTLLM\]|\[BONSAI\]|Add SDPA attention|no counterpart|Library plumbing",
                         comment), name
    assert names == set(declared_functions())
