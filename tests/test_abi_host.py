"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every function that
include/ffd.h declares, and rejects bad arguments on the host before it enqueues any work.

Every call below fails validation, so no fake pointer ever reaches a kernel.
"""
import ctypes
import math
import os
import re

import pytest

import sparse_quantized_attention_gb300 as ffd
from sparse_quantized_attention_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ffd.h")
FAKE = 0x10000  # 256-byte aligned, never dereferenced: every call here fails validation first


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ffd.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ffd_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("ffd_quantize_keys", "ffd_append_kv", "ffd_decode_attention", "ffd_dense_decode",
                 "ffd_decode_workspace_size", "ffd_dense_workspace_size", "ffd_get_error",
                 "ffd_status_string", "ffd_version"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(_build.LIB)
    for name in declared_functions():
        assert hasattr(raw, name), f"libffd.so does not export {name}"


def test_status_strings(lib):
    for code, name in ffd.ffd.STATUS_NAMES.items():
        assert ffd.ffd_status_string(code) == name
    assert ffd.ffd_version() >= 200


def _params(**kw):
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, num_pages=10, max_blocks_per_seq=5,
                sink=64, local=128, delta=5.0, num_splits=2)
    base.update(kw)
    return ffd.make_params(base.pop("batch"), base.pop("num_q_heads"), base.pop("num_kv_heads"),
                           base.pop("num_pages"), base.pop("max_blocks_per_seq"), **base)


def _decode(lib, p, ws_bytes=1 << 30, **ptrs):
    args = dict(q=FAKE, thumb=FAKE, resid=FAKE, v=FAKE, sl=FAKE, bt=FAKE, out=FAKE, mask=None,
                mt=None, ws=FAKE)
    args.update(ptrs)
    return lib.ffd_decode_attention(ctypes.byref(p), *[args[k] for k in (
        "q", "thumb", "resid", "v", "sl", "bt", "out", "mask", "mt", "ws")], ws_bytes, None)


def test_workspace_sizes(lib):
    p = _params()
    n = ffd.ffd_decode_workspace_size(p)
    assert n > 0 and n % 256 == 0
    assert ffd.ffd_dense_workspace_size(p) > 0
    assert ffd.ffd_decode_workspace_size(_params(num_q_heads=7, num_kv_heads=2)) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(num_q_heads=7, num_kv_heads=2), 1),       # Hq not a multiple of Hkv
    (dict(num_q_heads=18, num_kv_heads=2), 2),      # G = 9 unsupported
    (dict(batch=0), 1),
    (dict(delta=math.nan), 1),
    (dict(delta=-math.inf), 1),
    (dict(sink=-1), 1),
    (dict(num_splits=-2), 1),
    (dict(sm_scale=math.inf), 1),
    (dict(sm_scale=0.0), 1),
    (dict(sm_scale=-0.088), 1),
    (dict(wait_limit_us=-1), 1),                    # a negative wait bound
])
def test_decode_rejects_bad_params(lib, kw, status):
    assert _decode(lib, _params(**kw)) == status


def test_decode_rejects_unsupported_shapes(lib):
    p = _params()
    p.head_dim = 64
    assert _decode(lib, p) == 2
    p = _params()
    p.page_size = 16
    assert _decode(lib, p) == 2


def test_decode_rejects_null_and_misaligned_pointers(lib):
    p = _params()
    for key in ("q", "thumb", "resid", "v", "sl", "bt", "out", "ws"):
        assert _decode(lib, p, **{key: None}) == 1, key
    assert _decode(lib, p, thumb=FAKE + 4) == 1
    assert _decode(lib, p, resid=FAKE + 8) == 1
    assert _decode(lib, p, ws=FAKE + 16) == 1


def test_decode_rejects_small_workspace(lib):
    p = _params()
    need = ffd.ffd_decode_workspace_size(p)
    assert _decode(lib, p, ws_bytes=need - 1) == 3


def test_dense_rejects_bad_arguments(lib):
    p = _params()
    need = ffd.ffd_dense_workspace_size(p)
    call = lambda **kw: lib.ffd_dense_decode(  # noqa: E731
        ctypes.byref(kw.get("p", p)), kw.get("q", FAKE), kw.get("k", FAKE), FAKE, FAKE, FAKE,
        FAKE, FAKE, kw.get("ws_bytes", need), None)
    assert call(q=None) == 1
    assert call(k=FAKE + 2) == 1
    assert call(ws_bytes=need - 256) == 3
    assert call(p=_params(num_q_heads=18, num_kv_heads=2)) == 2


def test_quantize_rejects_bad_arguments(lib):
    good = ffd.CacheDesc(4, 2, 128, 64)
    call = lambda d, k=FAKE, ids=None, nids=0: lib.ffd_quantize_keys(  # noqa: E731
        ctypes.byref(d), k, FAKE, FAKE, ids, nids, None, None)
    assert call(good, k=None) == 1
    assert call(ffd.CacheDesc(0, 2, 128, 64)) == 1
    assert call(ffd.CacheDesc(4, 2, 96, 64)) == 2
    assert call(ffd.CacheDesc(4, 2, 128, 32)) == 2
    assert call(good, ids=FAKE, nids=-1) == 1
    assert call(good, k=FAKE + 8) == 1


def test_append_rejects_bad_arguments(lib):
    good = ffd.CacheDesc(4, 2, 128, 64)

    def call(d=good, batch=2, mb=3, **kw):
        a = dict(kn=FAKE, vn=FAKE, pos=FAKE, bt=FAKE, th=FAKE, rs=FAKE, v=FAKE, k=None)
        a.update(kw)
        return lib.ffd_append_kv(ctypes.byref(d), batch, mb, *[a[x] for x in (
            "kn", "vn", "pos", "bt", "th", "rs", "v", "k")], None, None)

    for key in ("kn", "vn", "pos", "bt", "th", "rs", "v"):
        assert call(**{key: None}) == 1, key
    assert call(batch=0) == 1
    assert call(mb=0) == 1
    assert call(d=ffd.CacheDesc(0, 2, 128, 64)) == 1
    assert call(d=ffd.CacheDesc(4, 2, 64, 64)) == 2
    assert call(d=ffd.CacheDesc(4, 2, 128, 16)) == 2
    assert call(kn=FAKE + 2) == 1
    assert call(k=FAKE + 4) == 1


def test_select_and_masked_reject_bad_arguments(lib):
    p = _params()
    need = ffd.ffd_select_workspace_size(p)
    assert need > 0 and need % 256 == 0
    assert ffd.ffd_select_workspace_size(_params(max_blocks_per_seq=20000)) == 0

    def sel(selector=1, budget=3.0, ws_bytes=need, **kw):
        a = dict(q=FAKE, th=FAKE, sl=FAKE, bt=FAKE, km=FAKE, ws=FAKE)
        a.update(kw)
        return lib.ffd_select_blocks(ctypes.byref(kw.pop("p", p)), selector, budget,
                                     *[a[x] for x in ("q", "th", "sl", "bt", "km", "ws")],
                                     ws_bytes, None)

    for key in ("q", "th", "sl", "bt", "km", "ws"):
        assert sel(**{key: None}) == 1, key
    assert sel(selector=0) == 1 and sel(selector=3) == 1
    assert sel(budget=-1.0) == 1 and sel(budget=2.5) == 1
    assert sel(selector=2, budget=0.0) == 1 and sel(selector=2, budget=1.5) == 1
    assert sel(selector=2, budget=math.nan) == 1
    assert sel(ws_bytes=need - 1) == 3
    assert sel(ws=FAKE + 16) == 1

    dneed = ffd.ffd_decode_workspace_size(p)

    def masked(**kw):
        a = dict(q=FAKE, th=FAKE, rs=FAKE, v=FAKE, sl=FAKE, bt=FAKE, ki=FAKE, out=FAKE, km=None,
                 mt=None, ws=FAKE)
        a.update(kw)
        return lib.ffd_decode_attention_masked(ctypes.byref(p), *[a[x] for x in (
            "q", "th", "rs", "v", "sl", "bt", "ki", "out", "km", "mt", "ws")], dneed, None)

    for key in ("q", "th", "rs", "v", "sl", "bt", "ki", "out", "ws"):
        assert masked(**{key: None}) == 1, key
    assert masked(v=FAKE + 2) == 1


def test_art_rejects_bad_arguments(lib):
    p = _params()
    need = ffd.ffd_art_workspace_size(p)
    # the error word, then one traversal list per (sequence, KV head) unit
    units = p.batch * p.num_kv_heads
    assert need == 256 + (units * p.max_blocks_per_seq * 4 + 255) // 256 * 256

    def art(tau=0.01, phi=0.001, patience=2, ws_bytes=need, **kw):
        a = dict(q=FAKE, th=FAKE, rs=FAKE, v=FAKE, sl=FAKE, bt=FAKE, ki=None, out=FAKE, bu=None,
                 ws=FAKE)
        a.update(kw)
        return lib.ffd_art_attention(
            ctypes.byref(kw.pop("p", p)), tau, phi, patience,
            *[a[x] for x in ("q", "th", "rs", "v", "sl", "bt", "ki", "out", "bu", "ws")],
            ws_bytes, None)

    for key in ("q", "th", "rs", "v", "sl", "bt", "out", "ws"):
        assert art(**{key: None}) == 1, key
    assert art(tau=-1e-3) == 1 and art(phi=-1.0) == 1
    assert art(tau=math.nan) == 1 and art(phi=math.nan) == 1
    assert art(patience=0) == 1 and art(patience=-3) == 1
    assert art(th=FAKE + 4) == 1 and art(v=FAKE + 2) == 1 and art(ws=FAKE + 16) == 1
    assert art(ws_bytes=need - 1) == 3
    bad = _params()
    bad.head_dim = 64
    assert art(p=bad) == 2 and ffd.ffd_art_workspace_size(bad) == 0


def test_suggest_schedule_rejects_bad_counts(lib):
    import sparse_quantized_attention_gb300 as ffd
    for total, kept in ((0, 0), (-5, 1), (100, -1), (100, 101)):
        assert ffd.ffd_suggest_schedule(total, kept) == ffd.SCHEDULE_FUSED
