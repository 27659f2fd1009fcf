"""The C ABI on a machine without a GPU: the library loads, exports every
entry point include/smla.h declares, and rejects bad arguments on the host
with the documented status before touching the device."""
import ctypes
import os
import re

import pytest

from serving_fp8_indexer_gb300 import _lib
from serving_fp8_indexer_gb300 import build as smla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INVALID, UNSUPPORTED = 1, 2


@pytest.fixture(scope="module")
def lib():
    smla_build.build()
    return _lib.load()


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "smla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(smla_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_entry_points()
    assert set(_lib.EXPORTED) <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert lib.smla_version().decode().count(".") == 2


def _seqs(T=4, B=1, page_size=64, max_pages=1, null=False):
    p = None if null else 0x1000
    return _lib.SeqsT(p, p, p, B, max_pages, page_size, T)


def _msg(lib):
    return _lib.last_error(lib)


def test_indexer_validation(lib):
    P = 0x10000  # aligned fake device pointers: validation runs before any launch
    f = lib.smla_indexer_scores
    assert f(P, P, P, P, 64, _seqs(), 5, P, 64, None) == UNSUPPORTED and "H_idx" in _msg(lib)
    assert f(P, P, P, P, 64, _seqs(page_size=48), 64, P, 64, None) == UNSUPPORTED and "page_size" in _msg(lib)
    assert f(P, P, P, P, 64, _seqs(), 64, P, 66, None) == INVALID and "score_stride" in _msg(lib)
    assert f(None, P, P, P, 64, _seqs(), 64, P, 64, None) == INVALID and "null" in _msg(lib)
    assert f(P + 8, P, P, P, 64, _seqs(), 64, P, 64, None) == INVALID and "aligned" in _msg(lib)
    assert f(P, P, P, P, 64, _seqs(null=True), 64, P, 64, None) == INVALID
    bad = _lib.SeqsT(P + 2, P, P, 1, 1, 64, 4)   # seqs pointers need 4-byte alignment
    assert f(P, P, P, P, 64, bad, 64, P, 64, None) == INVALID and "aligned" in _msg(lib)
    assert f(P, P, P, P, 0, _seqs(), 64, P, 64, None) == INVALID and "phys_rows" in _msg(lib)
    assert f(None, None, None, None, 0, _seqs(T=0), 64, None, 64, None) == 0   # empty batch: no-op


def test_topk_validation(lib):
    P = 0x10000
    f = lib.smla_topk
    assert f(P, 64, _seqs(), 0, P, P, None, 0, None) == UNSUPPORTED and "k=" in _msg(lib)
    assert f(P, 64, _seqs(), 70000, P, P, None, 0, None) == UNSUPPORTED
    assert f(P, 62, _seqs(), 8, P, P, None, 0, None) == INVALID
    assert f(P, 64, _seqs(), 8, None, P, None, 0, None) == INVALID
    assert f(P + 4, 64, _seqs(), 8, P, P, None, 0, None) == INVALID and "aligned" in _msg(lib)
    assert f(None, 64, _seqs(T=0), 8, None, None, None, 0, None) == 0
    # workspace: the size query, and a misaligned workspace is refused
    need = lib.smla_topk_workspace_size(16384, 8192, 2048)
    assert need == 0
    assert f(P, 64, _seqs(), 8, P, P, P + 8, 64, None) == INVALID and "workspace" in _msg(lib)


def test_selftest_validation(lib):
    assert lib.smla_selftest_wait_timeout(0, None) == INVALID and "limit_us" in _msg(lib)
    assert lib.smla_selftest_wait_timeout(2000000, None) == INVALID


def test_prefill_validation(lib):
    P = 0x10000
    f = lib.smla_sparse_prefill
    ok = dict(q=P, qd=0, lat=P, rows=64, sc=None, sbs=0, idx=P, st=8, ln=P, T=4, H=64, vd=512, ss=0.04, sink=None,
              out=P)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["qd"], a["lat"], a["rows"], a["sc"], a["sbs"], a["idx"], a["st"], a["ln"], a["T"], a["H"],
                 a["vd"], a["ss"], a["sink"], a["out"], None)

    assert call(qd=7) == INVALID
    assert call(H=24) == UNSUPPORTED and "H=" in _msg(lib)
    assert call(vd=256) == UNSUPPORTED and "v_depth" in _msg(lib)
    assert call(sbs=64) == UNSUPPORTED and "scale_block_size" in _msg(lib)
    assert call(sbs=32, qd=1) == INVALID and "scales" in _msg(lib)
    assert call(sbs=32, sc=P) == UNSUPPORTED and "e4m3 q" in _msg(lib)   # block scales need e4m3 q
    assert call(sink=P + 2) == INVALID and "attn_sink" in _msg(lib)   # the sink is f32 [H], 4-byte aligned
    assert call(ss=float("nan")) == INVALID
    assert call(st=0) == INVALID
    assert call(out=None) == INVALID
    assert call(lat=P + 8) == INVALID
    assert call(idx=P + 2) == INVALID and "aligned" in _msg(lib)
    assert call(sc=P + 2, sbs=576) == INVALID and "aligned" in _msg(lib)
    assert call(T=0, q=None, lat=None, idx=None, ln=None, out=None) == 0
    assert call(T=-1) == INVALID


def test_last_error_truncates(lib):
    lib.smla_topk(None, 64, _seqs(), 0, None, None, None, 0, None)
    full = lib.smla_last_error(None, 0)
    buf = ctypes.create_string_buffer(8)
    assert lib.smla_last_error(buf, 8) == full and len(buf.value) == 7


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(OSError):
        _lib.load(str(tmp_path / "missing.so"))
