"""Host-side checks of the C ABI that need no GPU: the library builds and loads,
exports every entry point include/kpool.h declares, sizes workspaces, and rejects
bad arguments before touching the device."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from sparse_attention_kpool_gb300 import build as kbuild
from sparse_attention_kpool_gb300 import kpool as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kpool.h")

# Fake, 256-byte aligned, never dereferenced addresses: every call below fails
# validation before any pointer is used.
FAKE = 0x7F0000000000


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return K.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kpool_[a-z_]+)\s*\(", text)))


def test_options_struct_layout_matches_header():
    assert ctypes.sizeof(K.kpool_options) == 32


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(K.EXPORTED)


def test_library_exports_every_declared_function(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", K.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared_functions():
        assert name in exported, f"{name} declared in kpool.h but not exported"
        assert hasattr(lib, name)


def test_status_strings(lib):
    for st in range(7):
        assert K.kpool_status_string(st) != "unknown status"
    assert K.kpool_status_string(99) == "unknown status"


def test_workspace_bytes(lib):
    a = K.kpool_workspace_bytes(8192, 2, 32, 128, K.KPOOL_BF16, 4, 2048)
    b = K.kpool_workspace_bytes(16384, 2, 32, 128, K.KPOOL_BF16, 4, 2048)
    assert a > 0 and b > a and a % 256 == 0
    # the pooled keys dominate: P * d * 2 bytes
    assert a >= 2048 * 128 * 2
    assert K.kpool_workspace_bytes(8192, 2, 32, 128, K.KPOOL_BF16, 3, 2048) == 0   # index_topk % kpool
    assert K.kpool_workspace_bytes(8192, 2, 32, 128, K.KPOOL_BF16, 0, 2048) == 0   # kpool < 1
    assert K.kpool_workspace_bytes(8192, 0, 32, 128, K.KPOOL_BF16, 4, 2048) == 0   # no sequences
    assert K.kpool_workspace_bytes(8192, 1, 32, 100, K.KPOOL_BF16, 4, 2048) == 0   # rows not 16-byte multiples
    assert K.kpool_workspace_bytes(-1, 1, 32, 128, K.KPOOL_BF16, 4, 2048) == 0
    assert K.kpool_workspace_bytes(0, 0, 32, 128, K.KPOOL_BF16, 4, 2048) > 0      # empty batch is valid


def _select(lib, T=64, S=1, H=4, d=32, dtype=K.KPOOL_F32, kpool=4, topk=16, scale=0.5, q=FAKE, k=FAKE, w=FAKE,
            cu=FAKE, ids=FAKE, toks=FAKE, scores=None, ws=FAKE, ws_bytes=1 << 30, opts=None):
    P = ctypes.c_void_p
    return lib.kpool_select_ex(P(q), P(k), P(w), P(cu), S, T, H, d, dtype, kpool, topk, scale, P(ids), P(toks),
                               P(scores) if scores else None, P(ws), ws_bytes, None,
                               ctypes.byref(opts) if opts else None)


def test_select_rejects_bad_arguments(lib):
    assert _select(lib, kpool=0) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, kpool=3, topk=16) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, topk=-4) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, H=0) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, d=30) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, dtype=7) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, S=0) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, T=-5) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, scale=float("nan")) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, scale=float("inf")) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, q=0) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, toks=0) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, ids=0) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, q=FAKE + 8) == K.KPOOL_ERR_INVALID_ARG      # q must be 16-byte aligned
    assert _select(lib, k=FAKE + 4) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, ws=0) == K.KPOOL_ERR_WORKSPACE
    assert _select(lib, ws=FAKE + 64) == K.KPOOL_ERR_WORKSPACE     # 256-byte alignment
    assert _select(lib, ws_bytes=1024) == K.KPOOL_ERR_WORKSPACE
    bad = K.kpool_options(K.KPOOL_SCORE_AUTO, 0)
    bad.reserved = 1
    assert _select(lib, opts=bad) == K.KPOOL_ERR_INVALID_ARG
    bad = K.kpool_options(K.KPOOL_SCORE_AUTO, 0)
    bad.flags = 2  # unknown flag
    assert _select(lib, opts=bad) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, opts=K.kpool_options(9, 0)) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, opts=K.kpool_options(0, -1)) == K.KPOOL_ERR_INVALID_ARG


def test_select_rejects_unsupported_kernel_choice(lib):
    # the tensor-core kernel needs bf16, H = 32, d = 128, budget <= 512
    tc = K.kpool_options(K.KPOOL_SCORE_TC, 0)
    assert _select(lib, opts=tc) == K.KPOOL_ERR_UNSUPPORTED                       # fp32, H 4, d 32
    assert _select(lib, H=32, d=128, dtype=K.KPOOL_BF16, topk=4096, opts=tc) == K.KPOOL_ERR_UNSUPPORTED
    assert _select(lib, H=65, d=128, dtype=K.KPOOL_BF16) == K.KPOOL_ERR_UNSUPPORTED
    assert _select(lib, H=4, d=512, dtype=K.KPOOL_BF16) == K.KPOOL_ERR_UNSUPPORTED


def test_empty_batch_is_a_noop(lib):
    assert _select(lib, T=0, S=0, q=0, k=0, w=0, cu=0, ids=0, toks=0, ws=0) == K.KPOOL_OK


def test_pool_keys_and_expand_validation(lib):
    P = ctypes.c_void_p
    assert lib.kpool_pool_keys(P(FAKE), P(FAKE), 1, 64, 32, K.KPOOL_F32, 0, P(FAKE), P(FAKE), 1 << 20,
                               None) == K.KPOOL_ERR_INVALID_ARG
    assert lib.kpool_pool_keys(P(FAKE), P(FAKE), 1, 64, 32, K.KPOOL_F32, 4, P(FAKE), P(FAKE), 16,
                               None) == K.KPOOL_ERR_WORKSPACE
    assert lib.kpool_pool_keys(P(FAKE + 4), P(FAKE), 1, 64, 32, K.KPOOL_F32, 4, P(FAKE), P(FAKE), 1 << 20,
                               None) == K.KPOOL_ERR_INVALID_ARG
    assert lib.kpool_expand(P(FAKE), P(FAKE), 1, 64, 4, 6, P(FAKE), None) == K.KPOOL_ERR_INVALID_ARG
    assert lib.kpool_expand(None, P(FAKE), 1, 64, 4, 16, P(FAKE), None) == K.KPOOL_ERR_INVALID_ARG
    assert lib.kpool_expand(None, None, 0, 0, 4, 16, None, None) == K.KPOOL_OK


def test_selftest_and_error_query_validation(lib):
    P = ctypes.c_void_p
    assert lib.kpool_wait_timeout_selftest(None, 1 << 20, 10, None) == K.KPOOL_ERR_WORKSPACE
    assert lib.kpool_wait_timeout_selftest(P(FAKE), 64, 10, None) == K.KPOOL_ERR_WORKSPACE
    assert lib.kpool_wait_timeout_selftest(P(FAKE), 1 << 20, 0, None) == K.KPOOL_ERR_INVALID_ARG
    assert lib.kpool_last_device_error(None, None) == K.KPOOL_ERR_WORKSPACE
    assert lib.kpool_last_device_error(P(FAKE + 8), None) == K.KPOOL_ERR_WORKSPACE


def _rows(lib, R=4, T=4096, S=1, H=32, d=128, dtype=K.KPOOL_BF16, kpool=4, topk=2048, scale=0.1, q=FAKE, w=FAKE,
          rs=FAKE, rp=FAKE, kp=FAKE, cu=FAKE, ids=FAKE, toks=FAKE, ws=FAKE, ws_bytes=1 << 30):
    P = ctypes.c_void_p
    pp = lambda x: P(x) if x else None  # noqa: E731
    return lib.kpool_select_rows(pp(q), pp(w), pp(rs), pp(rp), R, pp(kp), pp(cu), S, T, H, d, dtype, kpool, topk,
                                 scale, pp(ids), pp(toks), None, pp(ws), ws_bytes, None)


def test_rows_workspace_bytes(lib):
    a = K.kpool_rows_workspace_bytes(16, 262144 * 16, 16, 4, 2048)
    b = K.kpool_rows_workspace_bytes(32, 262144 * 16, 16, 4, 2048)
    assert a > 0 and b > a and a % 256 == 0
    # the score buffer holds T / kpool floats per row
    assert b - a >= 16 * (262144 * 16 // 4) * 4
    assert K.kpool_rows_workspace_bytes(-1, 100, 1, 4, 16) == 0
    assert K.kpool_rows_workspace_bytes(4, 100, 1, 0, 16) == 0
    assert K.kpool_rows_workspace_bytes(4, 100, 1, 3, 16) == 0
    assert K.kpool_rows_workspace_bytes(4, 100, 0, 4, 16) == 0


def test_select_rows_rejects_bad_arguments(lib):
    assert _rows(lib, kpool=0) == K.KPOOL_ERR_INVALID_ARG
    assert _rows(lib, topk=2046) == K.KPOOL_ERR_INVALID_ARG
    assert _rows(lib, R=-1) == K.KPOOL_ERR_INVALID_ARG
    assert _rows(lib, scale=float("nan")) == K.KPOOL_ERR_INVALID_ARG
    assert _rows(lib, T=0, S=0) == K.KPOOL_ERR_INVALID_ARG            # rows need a sequence
    for name in ("q", "w", "rs", "rp", "kp", "cu", "ids", "toks"):
        assert _rows(lib, **{name: 0}) == K.KPOOL_ERR_INVALID_ARG, name
    assert _rows(lib, q=FAKE + 8) == K.KPOOL_ERR_INVALID_ARG           # 16-byte rows for the vector loads
    assert _rows(lib, kp=FAKE + 8) == K.KPOOL_ERR_INVALID_ARG
    assert _rows(lib, rp=FAKE + 2) == K.KPOOL_ERR_INVALID_ARG
    assert _rows(lib, dtype=K.KPOOL_F32, d=128) == K.KPOOL_ERR_UNSUPPORTED
    assert _rows(lib, H=16) == K.KPOOL_ERR_UNSUPPORTED
    assert _rows(lib, topk=4096) == K.KPOOL_ERR_UNSUPPORTED             # budget 1024 > 512
    assert _rows(lib, ws=0) == K.KPOOL_ERR_WORKSPACE
    assert _rows(lib, ws=FAKE + 64) == K.KPOOL_ERR_WORKSPACE
    assert _rows(lib, ws_bytes=4096) == K.KPOOL_ERR_WORKSPACE
    # no rows: nothing to do, nothing checked beyond the shape
    assert _rows(lib, R=0, q=0, w=0, rs=0, rp=0, kp=0, ids=0, toks=0, ws=0) == K.KPOOL_OK


def test_gated_pool_and_pooled_select_validation(lib):
    P = ctypes.c_void_p
    ok = dict(k=P(FAKE), g=P(FAKE), a=P(FAKE), cu=P(FAKE), out=P(FAKE), ws=P(FAKE))

    def gated(**kw):
        v = dict(ok, **kw)
        return lib.kpool_pool_keys_gated(v["k"], v["g"], v["a"], v["cu"], 1, 64, 32, K.KPOOL_F32, 4, v["out"],
                                         v["ws"], 1 << 20, None)
    assert gated(g=None) == K.KPOOL_ERR_INVALID_ARG
    assert gated(a=None) == K.KPOOL_ERR_INVALID_ARG
    assert gated(g=P(FAKE + 2)) == K.KPOOL_ERR_INVALID_ARG
    assert gated(a=P(FAKE + 8)) == K.KPOOL_ERR_INVALID_ARG  # 16-byte vector loads
    assert gated(k=P(FAKE + 4)) == K.KPOOL_ERR_INVALID_ARG
    assert gated(ws=None) == K.KPOOL_ERR_WORKSPACE
    assert lib.kpool_pool_keys_gated(None, None, None, None, 0, 0, 32, K.KPOOL_F32, 4, None, None, 0,
                                     None) == K.KPOOL_OK
    # the pooled select validates like kpool_select_ex, with the pooled keys in k's place
    assert lib.kpool_select_pooled(P(FAKE), None, P(FAKE), P(FAKE), 1, 64, 4, 32, K.KPOOL_F32, 4, 16, 0.5,
                                   P(FAKE), P(FAKE), None, P(FAKE), 1 << 20, None, None) == K.KPOOL_ERR_INVALID_ARG
    assert lib.kpool_select_pooled(P(FAKE), P(FAKE + 8), P(FAKE), P(FAKE), 1, 64, 4, 32, K.KPOOL_F32, 4, 16, 0.5,
                                   P(FAKE), P(FAKE), None, P(FAKE), 1 << 20, None, None) == K.KPOOL_ERR_INVALID_ARG
    assert lib.kpool_select_pooled(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 64, 4, 32, K.KPOOL_F32, 4, 16, 0.5,
                                   P(FAKE), P(FAKE), None, None, 1 << 20, None, None) == K.KPOOL_ERR_WORKSPACE


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(K, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(K, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        K.load()


def _range_opts(b, e, flags=K.KPOOL_OPT_ROW_RANGE):
    o = K.kpool_options(K.KPOOL_SCORE_AUTO, 0)
    o.row_begin, o.row_end, o.flags = b, e, flags
    return o


def test_row_range_validation(lib):
    # bounds: 0 <= row_begin <= row_end <= T
    assert _select(lib, T=64, opts=_range_opts(-1, 10)) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, T=64, opts=_range_opts(10, 9)) == K.KPOOL_ERR_INVALID_ARG
    assert _select(lib, T=64, opts=_range_opts(10, 65)) == K.KPOOL_ERR_INVALID_ARG
    # a range without the flag is a mistake, not a silent whole-batch call
    assert _select(lib, T=64, opts=_range_opts(0, 10, flags=0)) == K.KPOOL_ERR_INVALID_ARG
    # the sharded path returns no index scores (the pages reject that combination)
    assert _select(lib, T=64, scores=FAKE, opts=_range_opts(0, 32)) == K.KPOOL_ERR_INVALID_ARG
    # an empty range is a valid no-op, even with null outputs
    assert _select(lib, T=64, ids=0, toks=0, ws=0, opts=_range_opts(17, 17)) == K.KPOOL_OK
    # a valid range still checks the workspace
    assert _select(lib, T=64, ws=0, opts=_range_opts(0, 32)) == K.KPOOL_ERR_WORKSPACE
    # the decode-rows entry point takes no row range
    P = ctypes.c_void_p
    o = _range_opts(0, 1)
    assert lib.kpool_select_rows_ex(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, P(FAKE), P(FAKE), 1, 64, 32, 128,
                                    K.KPOOL_BF16, 4, 16, 0.5, P(FAKE), P(FAKE), None, P(FAKE), 1 << 30, None,
                                    ctypes.byref(o)) == K.KPOOL_ERR_INVALID_ARG


def _scores(lib, T=64, S=1, H=4, d=32, dtype=K.KPOOL_F32, kpool=4, scale=0.5, q=FAKE, k=FAKE, w=FAKE, cu=FAKE,
            out=FAKE, ld=16, ws=FAKE, ws_bytes=1 << 30, opts=None, pooled=False):
    P = ctypes.c_void_p
    fn = lib.kpool_index_scores_pooled if pooled else lib.kpool_index_scores
    return fn(P(q), P(k), P(w), P(cu), S, T, H, d, dtype, kpool, scale, P(out), ld, P(ws), ws_bytes, None,
              ctypes.byref(opts) if opts else None)


@pytest.mark.parametrize("pooled", [False, True])
def test_index_scores_validation(lib, pooled):
    def sc(**kw):
        return _scores(lib, pooled=pooled, **kw)
    assert sc(kpool=0) == K.KPOOL_ERR_INVALID_ARG
    assert sc(H=0) == K.KPOOL_ERR_INVALID_ARG
    assert sc(d=30) == K.KPOOL_ERR_INVALID_ARG
    assert sc(ld=0) == K.KPOOL_ERR_INVALID_ARG
    assert sc(ld=-3) == K.KPOOL_ERR_INVALID_ARG
    assert sc(ld=1 << 62) == K.KPOOL_ERR_INVALID_ARG             # R * ld elements overflow
    assert sc(scale=float("nan")) == K.KPOOL_ERR_INVALID_ARG
    assert sc(out=0) == K.KPOOL_ERR_INVALID_ARG
    assert sc(out=FAKE + 2) == K.KPOOL_ERR_INVALID_ARG             # fp32 alignment
    assert sc(k=0) == K.KPOOL_ERR_INVALID_ARG
    assert sc(k=FAKE + 8) == K.KPOOL_ERR_INVALID_ARG               # 16-byte rows
    assert sc(ws=0) == K.KPOOL_ERR_WORKSPACE
    assert sc(ws_bytes=1024) == K.KPOOL_ERR_WORKSPACE
    assert sc(T=0, S=0, q=0, k=0, w=0, cu=0, out=0, ws=0) == K.KPOOL_OK
    # row ranges as for kpool_select_ex; an empty one is a no-op
    assert sc(opts=_range_opts(10, 9)) == K.KPOOL_ERR_INVALID_ARG
    assert sc(opts=_range_opts(0, 65)) == K.KPOOL_ERR_INVALID_ARG
    assert sc(opts=_range_opts(0, 10, flags=0)) == K.KPOOL_ERR_INVALID_ARG
    assert sc(out=0, ws=0, opts=_range_opts(9, 9)) == K.KPOOL_OK
    assert sc(ws=0, opts=_range_opts(0, 32)) == K.KPOOL_ERR_WORKSPACE
    # the tensor-core kernel needs bf16, H = 32, d = 128; the SIMT one H <= 64, d <= 256
    assert sc(opts=K.kpool_options(K.KPOOL_SCORE_TC, 0)) == K.KPOOL_ERR_UNSUPPORTED
    assert sc(H=65, d=128, dtype=K.KPOOL_BF16) == K.KPOOL_ERR_UNSUPPORTED
    assert sc(H=32, d=128, dtype=K.KPOOL_BF16, ws=0, opts=K.kpool_options(K.KPOOL_SCORE_TC, 0)) == \
        K.KPOOL_ERR_WORKSPACE
    bad = K.kpool_options(K.KPOOL_SCORE_AUTO, 0)
    bad.reserved = 1
    assert sc(opts=bad) == K.KPOOL_ERR_INVALID_ARG


def test_index_scores_workspace_is_the_selections(lib):
    # the index-score calls take the selection's workspace; index_topk 0 sizes it
    assert K.kpool_workspace_bytes(8192, 2, 32, 128, K.KPOOL_BF16, 4, 0) == \
        K.kpool_workspace_bytes(8192, 2, 32, 128, K.KPOOL_BF16, 4, 2048)


def _pairs_per_row(cu, kpool):
    rows = []
    for b in range(len(cu) - 1):
        rows += [(t + 1) // kpool for t in range(cu[b + 1] - cu[b])]
    return np.array(rows, dtype=np.int64)


@pytest.mark.parametrize("seqlens,kpool,parts,row_weight", [
    ((524288,), 4, 8, 0), ((131072,), 4, 3, 512), ((8192, 16384, 3072, 5120), 4, 8, 0),
    ((5, 0, 130, 1027, 3), 3, 4, 0), ((1, 2, 3), 4, 8, 0), ((100,), 4, 200, 1), ((0, 0), 4, 3, 0)])
def test_balanced_row_split(lib, seqlens, kpool, parts, row_weight):
    cu = np.cumsum([0] + list(seqlens)).astype(np.int32)
    b = K.kpool_balanced_row_split(cu, kpool, parts, row_weight)
    T = int(cu[-1])
    assert len(b) == parts + 1 and b[0] == 0 and b[-1] == T
    assert all(x <= y for x, y in zip(b, b[1:]))
    work = _pairs_per_row(cu, kpool) + row_weight
    prefix = np.concatenate([[0], np.cumsum(work)])
    total = int(prefix[-1])
    for g in range(1, parts):
        # boundary g is the first row whose preceding work reaches g/parts of the total
        target = (total // parts) * g + ((total % parts) * g) // parts
        assert prefix[b[g]] >= target
        assert b[g] == 0 or prefix[b[g] - 1] < target
    # so every range's work is within one row's work of an equal share
    share, row_max = total / parts, int(work.max()) if len(work) else 0
    for g in range(parts):
        assert abs(int(prefix[b[g + 1]] - prefix[b[g]]) - share) <= row_max + 1


def test_balanced_row_split_validation(lib):
    P = ctypes.c_void_p
    cu = np.array([0, 10, 5], dtype=np.int32)
    out = np.zeros(4, dtype=np.int32)
    ptr = lambda a: a.ctypes.data_as(P)  # noqa: E731
    assert lib.kpool_balanced_row_split(ptr(cu), 2, 4, 0, 3, ptr(out)) == K.KPOOL_ERR_INVALID_ARG  # decreasing
    cu = np.array([0, 10], dtype=np.int32)
    assert lib.kpool_balanced_row_split(ptr(cu), 1, 0, 0, 3, ptr(out)) == K.KPOOL_ERR_INVALID_ARG  # kpool
    assert lib.kpool_balanced_row_split(ptr(cu), 1, 4, 0, 0, ptr(out)) == K.KPOOL_ERR_INVALID_ARG  # parts
    assert lib.kpool_balanced_row_split(ptr(cu), 1, 4, -1, 3, ptr(out)) == K.KPOOL_ERR_INVALID_ARG
    assert lib.kpool_balanced_row_split(None, 1, 4, 0, 3, ptr(out)) == K.KPOOL_ERR_INVALID_ARG
