"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every entry point of include/qsa.h, and rejects bad arguments on the host
before touching any device."""
import ctypes
import os
import re

import pytest

from block_sparse_attention_select_gb300 import build as qbuild
from block_sparse_attention_select_gb300 import qsa

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "qsa.h")


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qsa.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"qsa_index_score", "qsa_topk_exact", "qsa_select_paged_tokens",
            "qsa_workspace_bytes", "qsa_get_device_status", "qsa_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_status_strings(lib):
    for s in range(0, 9):
        assert qsa.status_string(s)
    assert qsa.status_string(0) == "ok"


def test_workspace_size_grows_with_shape(lib):
    a = qsa.workspace_bytes(1616, 46080, 2048)
    b = qsa.workspace_bytes(3232, 46080, 2048)
    assert a > 1616 * 46080 * 4 and b > a
    assert qsa.workspace_bytes(0, 0, 0) > 0


def _call_select(lib, **over):
    keys = qsa.PagedKeysC(16, 4, 16, 128, 16, 1, 4)
    args = dict(q=16, w=16, rows=8, H=4, keys=ctypes.byref(keys), row_req=16, row_visible=16,
                k=8, out_idx=16, out_val=None, ws=256, ws_bytes=1 << 40, stream=None)
    args.update(over)
    vp = ctypes.c_void_p
    return lib.qsa_select_paged_tokens(vp(args["q"]), vp(args["w"]), args["rows"], args["H"],
                                       args["keys"], vp(args["row_req"]), vp(args["row_visible"]),
                                       args["k"], vp(args["out_idx"]), vp(args["out_val"]),
                                       vp(args["ws"]), args["ws_bytes"], vp(args["stream"]))


def test_host_side_argument_checks(lib):
    assert _call_select(lib, rows=0) == qsa.QSA_OK              # nothing to do
    assert _call_select(lib, k=0) == qsa.QSA_OK
    assert _call_select(lib, rows=-1) == qsa.QSA_ERR_INVALID_ARG
    assert _call_select(lib, q=None) == qsa.QSA_ERR_INVALID_ARG
    assert _call_select(lib, q=18) == qsa.QSA_ERR_INVALID_ARG   # not 16-byte aligned
    assert _call_select(lib, H=3) == qsa.QSA_ERR_UNSUPPORTED
    assert _call_select(lib, k=qsa.QSA_MAX_K + 1) == qsa.QSA_ERR_UNSUPPORTED
    assert _call_select(lib, k=-2) == qsa.QSA_ERR_INVALID_ARG
    bad_dim = qsa.PagedKeysC(16, 4, 16, 64, 16, 1, 4)
    assert _call_select(lib, keys=ctypes.byref(bad_dim)) == qsa.QSA_ERR_UNSUPPORTED
    bad_page = qsa.PagedKeysC(16, 4, 12, 128, 16, 1, 4)
    assert _call_select(lib, keys=ctypes.byref(bad_page)) == qsa.QSA_ERR_UNSUPPORTED
    no_table = qsa.PagedKeysC(16, 4, 16, 128, 0, 1, 4)
    assert _call_select(lib, keys=ctypes.byref(no_table)) == qsa.QSA_ERR_INVALID_ARG
    # with every host check passed and no GPU here, the call reports no device
    assert _call_select(lib) in (qsa.QSA_ERR_NO_DEVICE, qsa.QSA_ERR_WORKSPACE)


def test_config_switches(lib):
    assert lib.qsa_set_config(qsa.QSA_CFG_PATH, 1) == qsa.QSA_OK
    assert lib.qsa_set_config(qsa.QSA_CFG_PATH, 0) == qsa.QSA_OK
    assert lib.qsa_set_config(qsa.QSA_CFG_PATH, 5) == qsa.QSA_ERR_INVALID_ARG
    assert lib.qsa_set_config(99, 1) == qsa.QSA_ERR_INVALID_ARG
    assert lib.qsa_set_config(qsa.QSA_CFG_WAIT_LIMIT_NS, 0) == qsa.QSA_ERR_INVALID_ARG
    assert lib.qsa_set_config(qsa.QSA_CFG_WAIT_LIMIT_NS, 2_000_000_000) == qsa.QSA_OK
    assert lib.qsa_set_config(qsa.QSA_CFG_OVERLAP, 0) == qsa.QSA_OK
    assert lib.qsa_set_config(qsa.QSA_CFG_OVERLAP, 2) == qsa.QSA_ERR_INVALID_ARG
    assert lib.qsa_set_config(qsa.QSA_CFG_OVERLAP, 1) == qsa.QSA_OK


def test_topk_host_checks(lib):
    f = lib.qsa_topk_exact
    vp = ctypes.c_void_p
    assert f(vp(16), 10, 0, vp(16), 4, vp(16), None, None, 0, None) == qsa.QSA_OK
    assert f(vp(16), 10, 4, vp(16), -1, vp(16), None, None, 0, None) == qsa.QSA_ERR_INVALID_ARG
    assert f(vp(16), 0, 4, vp(16), 4, vp(16), None, None, 0, None) == qsa.QSA_ERR_INVALID_ARG
    assert f(None, 10, 4, vp(16), 4, vp(16), None, None, 0, None) == qsa.QSA_ERR_INVALID_ARG
    assert f(vp(16), 10, 4, vp(16), qsa.QSA_MAX_K + 1, vp(16), None, None, 0,
             None) == qsa.QSA_ERR_UNSUPPORTED


def test_producer_host_checks(lib):
    vp = ctypes.c_void_p
    keys = qsa.PagedKeysC(16, 4, 16, 128, 16, 1, 4)
    f = lib.qsa_index_key_produce

    def call(**kw):
        a = dict(x=vp(16), pl=None, n=1, ss=vp(16), ps=vp(16), mt=8, g=vp(16), eps=1e-6, rt=vp(16),
                 rb=4, rd=64, win=4, keys=ctypes.byref(keys))
        a.update(kw)
        return f(a["x"], a["pl"], a["n"], a["ss"], a["ps"], a["mt"], a["g"], a["eps"], a["rt"], a["rb"],
                 a["rd"], a["win"], a["keys"], None)

    assert call(win=6) == qsa.QSA_ERR_UNSUPPORTED
    assert call(rd=60) == qsa.QSA_ERR_INVALID_ARG           # not a multiple of 8
    assert call(rd=136) == qsa.QSA_ERR_INVALID_ARG
    assert call(eps=-1.0) == qsa.QSA_ERR_INVALID_ARG
    assert call(eps=float("nan")) == qsa.QSA_ERR_INVALID_ARG
    assert call(n=-1) == qsa.QSA_ERR_INVALID_ARG
    assert call(n=0) == qsa.QSA_OK                           # nothing to do
    assert call(mt=0) == qsa.QSA_OK
    assert call(n=2) == qsa.QSA_ERR_UNSUPPORTED             # more requests than the block table has
    assert call(x=None) == qsa.QSA_ERR_INVALID_ARG
    assert call(x=vp(12)) == qsa.QSA_ERR_INVALID_ARG        # 8-byte alignment
    assert call(g=vp(24)) == qsa.QSA_ERR_INVALID_ARG        # 16-byte alignment
    assert call(rt=None) == qsa.QSA_ERR_INVALID_ARG
    assert call(keys=None) == qsa.QSA_ERR_INVALID_ARG
    assert call() in (qsa.QSA_ERR_NO_DEVICE,)               # every host check passed, no GPU here
    assert call(rd=0, rt=None) in (qsa.QSA_ERR_NO_DEVICE,)  # no table needed without rotation
    r = lib.qsa_rope_table
    assert r(vp(16), 4, 60, 10000.0, None) == qsa.QSA_ERR_INVALID_ARG
    assert r(vp(16), 4, 64, 0.0, None) == qsa.QSA_ERR_INVALID_ARG
    assert r(vp(16), -1, 64, 10000.0, None) == qsa.QSA_ERR_INVALID_ARG
    assert r(None, 0, 64, 10000.0, None) == qsa.QSA_OK
    assert r(vp(20), 4, 64, 10000.0, None) == qsa.QSA_ERR_INVALID_ARG
    assert r(vp(16), 4, 64, 10000.0, None) == qsa.QSA_ERR_NO_DEVICE


def test_consumer_host_checks(lib):
    vp = ctypes.c_void_p
    f = lib.qsa_sparse_attention

    def call(**kw):
        a = dict(q=vp(16), rows=2, hq=24, kc=vp(16), vc=vp(16), npg=4, pt=64, hkv=2, d=256, bt=vp(16), nr=1,
                 mp=4, rr=vp(16), rt=vp(16), sel=vp(16), k=16, scale=0.0625, out=vp(16))
        a.update(kw)
        return f(a["q"], a["rows"], a["hq"], a["kc"], a["vc"], a["npg"], a["pt"], a["hkv"], a["d"], a["bt"],
                 a["nr"], a["mp"], a["rr"], a["rt"], a["sel"], a["k"], a["scale"], a["out"], None)

    assert call(d=128) == qsa.QSA_ERR_UNSUPPORTED
    assert call(hq=25) == qsa.QSA_ERR_UNSUPPORTED          # not a multiple of hkv
    assert call(hq=34) == qsa.QSA_ERR_UNSUPPORTED          # 17 query heads per KV head
    assert call(pt=48) == qsa.QSA_ERR_UNSUPPORTED
    assert call(scale=0.0) == qsa.QSA_ERR_INVALID_ARG
    assert call(rows=-1) == qsa.QSA_ERR_INVALID_ARG
    assert call(rows=0) == qsa.QSA_OK
    assert call(q=None) == qsa.QSA_ERR_INVALID_ARG
    assert call(sel=None) == qsa.QSA_ERR_INVALID_ARG
    assert call(sel=None, k=0) == qsa.QSA_ERR_NO_DEVICE    # k = 0: only the unfinished block
    assert call(out=vp(24)) == qsa.QSA_ERR_INVALID_ARG      # 16-byte alignment
    assert call() == qsa.QSA_ERR_NO_DEVICE


def test_misaligned_arrays_are_rejected_on_the_host(lib):
    """Every int32 / float array is read element by element on the device; a
    pointer that is not 4-byte aligned is refused before any launch."""
    for name in ("w", "row_req", "row_visible", "out_idx"):
        assert _call_select(lib, **{name: 18}) == qsa.QSA_ERR_INVALID_ARG, name
    assert _call_select(lib, out_val=18) == qsa.QSA_ERR_INVALID_ARG
    bad_table = qsa.PagedKeysC(16, 4, 16, 128, 18, 1, 4)
    assert _call_select(lib, keys=ctypes.byref(bad_table)) == qsa.QSA_ERR_INVALID_ARG
    vp = ctypes.c_void_p
    f = lib.qsa_topk_exact
    assert f(vp(18), 10, 4, vp(16), 4, vp(16), None, None, 0, None) == qsa.QSA_ERR_INVALID_ARG
    assert f(vp(16), 10, 4, vp(16), 4, vp(18), None, None, 0, None) == qsa.QSA_ERR_INVALID_ARG
    keys = qsa.PagedKeysC(16, 4, 16, 128, 16, 1, 4)
    p = lib.qsa_index_key_produce
    for pl, ss, ps in ((vp(18), vp(16), vp(16)), (None, vp(18), vp(16)), (None, vp(16), vp(18))):
        assert p(vp(16), pl, 1, ss, ps, 8, vp(16), 1e-6, vp(16), 4, 64, 4, ctypes.byref(keys), None) \
            == qsa.QSA_ERR_INVALID_ARG
    a = lib.qsa_sparse_attention
    for bt, rr, rt, sel in ((18, 16, 16, 16), (16, 18, 16, 16), (16, 16, 18, 16), (16, 16, 16, 18)):
        assert a(vp(16), 2, 24, vp(16), vp(16), 4, 64, 2, 256, vp(bt), 1, 4, vp(rr), vp(rt), vp(sel), 16,
                 0.0625, vp(16), None) == qsa.QSA_ERR_INVALID_ARG


def test_block_select_host_checks(lib):
    vp = ctypes.c_void_p
    f = lib.qsa_block_select                                          # prototypes set by the binding
    assert lib.qsa_block_select_workspace_bytes(1616, 2, 1440, 16) > 1616 * 2 * 1440 * 4   # the score matrix

    def call(**kw):
        a = dict(q=vp(16), rows=4, H=2, kc=vp(16), npg=8, bt=vp(16), nr=1, mb=8, rr=vp(16), rt=vp(16), k=4,
                 oi=vp(16), ov=vp(16), ws=vp(256), wsb=1 << 30)
        a.update(kw)
        return f(a["q"], a["rows"], a["H"], a["kc"], a["npg"], a["bt"], a["nr"], a["mb"], a["rr"], a["rt"], a["k"],
                 a["oi"], a["ov"], a["ws"], a["wsb"], None)

    assert call(rows=-1) == qsa.QSA_ERR_INVALID_ARG
    assert call(k=-1) == qsa.QSA_ERR_INVALID_ARG
    assert call(H=0) == qsa.QSA_ERR_INVALID_ARG
    assert call(npg=0) == qsa.QSA_ERR_INVALID_ARG
    assert call(mb=0) == qsa.QSA_ERR_INVALID_ARG
    assert call(H=17) == qsa.QSA_ERR_UNSUPPORTED
    assert call(k=qsa.QSA_MAX_K + 1) == qsa.QSA_ERR_UNSUPPORTED
    assert call(rows=0) == qsa.QSA_OK                                 # nothing to do
    assert call(k=0) == qsa.QSA_OK
    assert call(q=None) == qsa.QSA_ERR_INVALID_ARG
    assert call(oi=None) == qsa.QSA_ERR_INVALID_ARG
    assert call(q=vp(24)) == qsa.QSA_ERR_INVALID_ARG                  # 16-byte alignment
    assert call(kc=vp(24)) == qsa.QSA_ERR_INVALID_ARG
    assert call(rr=vp(18)) == qsa.QSA_ERR_INVALID_ARG                 # 4-byte alignment
    assert call(ov=vp(18)) == qsa.QSA_ERR_INVALID_ARG
    assert call() == qsa.QSA_ERR_NO_DEVICE
