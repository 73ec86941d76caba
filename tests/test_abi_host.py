"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/gqa_attn.h declares, refuses invalid arguments before touching
CUDA, and plans decode splits deterministically."""
import ctypes
import os
import re

import pytest

import gqa_head_gated_gb300 as G
from gqa_head_gated_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
P = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from gqa_head_gated_gb300 import build
        build.build()
    return _lib.load()


def _declared_functions():
    names = set()
    for f in os.listdir(INCLUDE):
        if not f.endswith(".h"):
            continue
        src = open(os.path.join(INCLUDE, f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, re.M):
            names.add(m.group(1))
    return names


def test_exports_every_declared_function(lib):
    names = _declared_functions()
    assert {"gqa_attn_prefill", "gqa_attn_decode", "attn_lse_merge"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), f"libgqa_attn.so does not export {n}"
    assert set(_lib.SIGNATURES) == names


def test_launch_log_without_launches(lib):
    """No kernel has run in this (GPU-less) process: the log is empty, and bad
    arguments are refused with -GQA_ERR_INVALID_ARG."""
    assert G.launch_log() == []
    assert lib.gqa_launch_log(None, 0) == 0
    assert lib.gqa_launch_log(None, 4) == -1
    buf = (_lib.LaunchInfo * 2)()
    assert lib.gqa_launch_log(buf, -1) == -1


def test_status_strings(lib):
    assert lib.gqa_status_string(0) == b"ok"
    assert lib.gqa_status_string(1) == b"invalid argument"
    assert lib.gqa_status_string(99) == b"unknown status"
    assert lib.gqa_version().count(b".") == 2


def _prefill(lib, **kw):
    a = dict(Q=16, K=32, V=48, G=None, out=64, lse=None, B=1, Hq=4, Hkv=2, Lq=8, Lkv=8, off=0)
    a.update(kw)
    return lib.gqa_attn_prefill(P(a["Q"]), P(a["K"]), P(a["V"]), P(a["G"]), P(a["out"]),
                                P(a["lse"]), a["B"], a["Hq"], a["Hkv"], a["Lq"], a["Lkv"],
                                a["off"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(Hq=0), 1), (dict(Hkv=0), 1), (dict(Hq=6, Hkv=4), 1),
    (dict(Lq=-1), 1), (dict(off=-1), 1), (dict(Lq=8, Lkv=7), 1), (dict(off=1, Lq=8, Lkv=8), 1),
    (dict(Q=None), 1), (dict(out=None), 1), (dict(K=None), 1), (dict(Q=8), 1), (dict(out=4), 1),
    (dict(G=2), 1), (dict(lse=2), 1), (dict(Hq=129 * 2, Hkv=2), 2), (dict(Lq=0), 0),
    (dict(Lq=0, Lkv=1, off=1), 0),
])
def test_prefill_rejects_before_launch(lib, kw, code):
    # Pointers are fake (never dereferenced): every case returns before any CUDA call.
    assert _prefill(lib, **kw) == code


def _decode(lib, **kw):
    a = dict(Q=16, K=32, V=48, G=None, kv=80, cu=None, out=64, lse=None, B=2, T=2, Hq=4, Hkv=2,
             Lcap=16, max_rows=1, max_kv=16, ws=96, wsb=1 << 30)
    a.update(kw)
    return lib.gqa_attn_decode(P(a["Q"]), P(a["K"]), P(a["V"]), P(a["G"]), P(a["kv"]),
                               P(a["cu"]), P(a["out"]), P(a["lse"]), a["B"], a["T"], a["Hq"],
                               a["Hkv"], a["Lcap"], a["max_rows"], a["max_kv"], P(a["ws"]),
                               a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(Hq=5), 1), (dict(Hkv=0), 1), (dict(T=3), 1), (dict(max_rows=2), 1),
    (dict(max_kv=17), 1), (dict(max_kv=0), 1), (dict(Lcap=0), 1), (dict(Q=None), 1),
    (dict(kv=None), 1), (dict(out=8), 1), (dict(wsb=10), 5), (dict(ws=None), 5), (dict(ws=8), 1),
    (dict(cu=128, T=5, max_rows=2), 1), (dict(cu=128, T=4, max_rows=3, max_kv=2), 1),
    (dict(T=0, cu=128, max_rows=1), 0),
])
def test_decode_rejects_before_launch(lib, kw, code):
    assert _decode(lib, **kw) == code


def test_merge_rejects_before_launch(lib):
    f = lib.attn_lse_merge
    assert f(P(16), P(32), 0, 4, None, P(64), None, None) == 1
    assert f(P(16), P(32), 2, -1, None, P(64), None, None) == 1
    assert f(P(16), P(32), 2, 0, None, P(64), None, None) == 0
    assert f(None, P(32), 2, 4, None, P(64), None, None) == 1
    assert f(P(8), P(32), 2, 4, None, P(64), None, None) == 1
    assert f(P(16), P(32), 2, 4, P(8), P(64), None, None) == 1


def test_split_rejects_bad_plan(lib):
    f = lib.gqa_attn_decode_split
    args = [P(16), P(32), P(48), P(80), None, P(96), P(112), 2, 2, 4, 2, 1024, 1, 1000]
    assert f(*args, 0, 1024, None) == 1          # no split
    assert f(*args, 2, 100, None) == 1           # not a multiple of 64
    assert f(*args, 2, 448, None) == 1           # 2 * 448 < 1000 keys
    assert f(*args[:-3], 1024, 1, 1025, 2, 576, None) == 1   # max_kv_len > Lcap
    assert f(*args, 2, 0, None) == 1             # balanced shares need >= 3 part slots
    # balanced shares are an mma.sync-path form: 32 rows x GQA 2 = 64 packed rows
    # (more than 16) is not
    assert f(P(16), P(32), P(48), P(80), P(96), P(112), P(128), 2, 64, 4, 2, 1024, 32, 1000,
             16, 0, None) == 2


def plan(lib, *a):
    s, c = ctypes.c_int(), ctypes.c_int()
    code = lib.gqa_attn_decode_plan(*a, ctypes.byref(s), ctypes.byref(c))
    return code, s.value, c.value


def test_decode_plan_rule(lib):
    # Without a GPU the planner assumes GB300's 152 SMs.
    for B, T, Hq, Hkv, R, L in [(16, 16, 24, 4, 1, 32768), (8, 68, 16, 2, 32, 65536),
                                (1, 1, 8, 8, 1, 1), (3, 9, 12, 3, 5, 300), (64, 64, 32, 8, 1, 131072)]:
        code, S, C = plan(lib, B, T, Hq, Hkv, R, L)
        assert code == 0
        assert C % 64 == 0 and C >= 64
        assert S >= 1 and S * C >= L and (S - 1) * C < L        # no empty trailing split
        size = lib.gqa_attn_decode_workspace_size(B, T, Hq, Hkv, R, L)
        # at most 16 packed rows per group and B <= 256: the one-call decode runs
        # balanced shares with 16 part slots per row; otherwise the plan's S
        parts = 16 if R * (Hq // Hkv) <= 16 and B <= 256 else S
        assert size == parts * T * Hq * 257 * 4
    assert plan(lib, 16, 16, 24, 4, 1, 32768)[1:] == (15, 2240)    # 6 x 152 CTAs / 64 units
    # 32 rows x 8 heads per group: tcgen05 path, 3 x 152 CTAs / (8 x 2 x 2 row tiles),
    # whole 128-key tiles
    assert plan(lib, 8, 68, 16, 2, 32, 65536)[1:] == (15, 4480)
    assert plan(lib, 1, 8, 8, 1, 8, 5000)[1:] == (5, 1024)           # at least 1024 keys
    assert plan(lib, 0, 1, 8, 8, 1, 1)[0] == 1
    assert lib.gqa_attn_decode_workspace_size(0, 1, 8, 8, 1, 1) == 0


def test_binding_refuses_cpu_tensors():
    import torch
    import gqa_head_gated_gb300 as G
    q = torch.zeros(1, 2, 4, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        G.prefill(q, q[:, :1], q[:, :1], q)
    with pytest.raises(TypeError):
        G.prefill(q.float(), q, q, q)


def test_verify_tree_rejects_before_launch(lib):
    f = lib.gqa_attn_verify_tree
    base = dict(Q=16, K=32, V=48, G=None, kv=80, cu=96, tm=112, out=128, lse=None, B=2, T=4,
                Hq=4, Hkv=2, Lcap=100, max_rows=2, max_kv=100, ws=144, wsb=1 << 30)
    def call(**kw):
        a = dict(base); a.update(kw)
        return f(P(a["Q"]), P(a["K"]), P(a["V"]), P(a["G"]), P(a["kv"]), P(a["cu"]), P(a["tm"]),
                 P(a["out"]), P(a["lse"]), a["B"], a["T"], a["Hq"], a["Hkv"], a["Lcap"],
                 a["max_rows"], a["max_kv"], P(a["ws"]), a["wsb"], None)
    assert call(max_rows=65, T=4) == 2          # more than 64 new rows: no 64-bit mask
    assert call(tm=None) == 1
    assert call(cu=None) == 1
    assert call(tm=116) == 1                    # mask array not 8-byte aligned
    assert call(wsb=8) == 5
    assert call(T=0) == 0


def test_kv_append_keep_reject_before_launch(lib):
    a = lib.gqa_kv_append
    assert a(P(16), P(32), None, P(48), P(64), P(80), 2, 3, 2, 10, None) == 1   # T != B without cu_rows
    assert a(P(16), P(32), P(96), P(48), P(64), P(80), 0, 3, 2, 10, None) == 1
    assert a(P(8), P(32), P(96), P(48), P(64), P(80), 2, 3, 2, 10, None) == 1    # misaligned
    assert a(P(16), P(32), P(96), P(48), P(64), P(80), 2, 0, 2, 10, None) == 0
    k = lib.gqa_kv_keep
    assert k(P(16), P(32), P(48), P(64), P(80), P(96), P(48), 2, 2, 10, None) == 1  # out aliases in
    assert k(P(16), P(32), P(48), None, P(80), P(96), None, 2, 2, 10, None) == 1
    assert k(P(16), P(32), P(48), P(64), P(80), P(96), None, 0, 2, 10, None) == 1


def _mask_rules():
    path = os.path.join(ROOT, "tests", "golden", "mask_head_rules.txt")
    rows = []
    for line in open(path):
        f = line.split("#")[0].split()
        if f:
            rows.append((int(f[0]), int(f[1]), int(f[2]), int(f[3]), f[4] == "on", f[5]))
    return rows


def test_mask_check_matches_the_head_rule_table(lib):
    """gqa_attn_mask_check (host only) accepts and refuses mask head counts exactly as
    the table derived from the DS4Server README's rule says; batch, row and key
    dimensions must be 1 or the call's size; strides must be >= 0; kinds 0..4."""
    LL4 = ctypes.c_longlong * 4
    for rows, gqa, hkv, hm, chunking, expect in _mask_rules():
        code = lib.gqa_attn_mask_check(1, gqa * hkv, hkv, rows, 2, 1, LL4(1, hm, rows, 2),
                                       LL4(0, rows * 2, 2, 1), int(chunking))
        assert code == (0 if expect == "ok" else 1), (rows, gqa, hkv, hm, chunking)
    chk = lambda shape, strides=(0, 0, 0, 1), kind=1: lib.gqa_attn_mask_check(
        2, 4, 2, 3, 5, kind, LL4(*shape), LL4(*strides), 1)
    assert chk((2, 4, 3, 5)) == 0 and chk((1, 1, 1, 1)) == 0 and chk((1, 1, 3, 1)) == 0
    assert chk((3, 1, 3, 5)) == 1 and chk((1, 1, 2, 5)) == 1 and chk((1, 1, 3, 4)) == 1
    assert chk((1, 2, 3, 5)) == 1 and chk((0, 1, 3, 5)) == 1
    assert chk((1, 1, 3, 5), strides=(0, 0, -5, 1)) == 1
    assert chk((1, 1, 3, 5), kind=5) == 1 and chk((1, 1, 3, 5), kind=-1) == 1
    assert lib.gqa_attn_mask_check(2, 4, 2, 3, 5, 0, None, None, 1) == 0     # no mask
    assert lib.gqa_attn_mask_check(2, 4, 2, 3, 5, 1, None, None, 1) == 1


def test_masked_rejects_before_launch(lib):
    """gqa_attn_masked refuses bad masks, a missing mask pointer, a misaligned
    additive mask and a causal offset past the keys, before any CUDA call."""
    LL4 = ctypes.c_longlong * 4
    f = lib.gqa_attn_masked
    def call(mask=64, kind=1, shape=(1, 1, 3, 5), causal=0, off=0, Lq=3):
        return f(P(16), P(32), P(48), None, P(mask) if mask else None, kind, LL4(*shape),
                 LL4(0, 0, 5, 1), P(80), None, 1, 4, 2, Lq, 5, causal, off, 1, None)
    assert call(shape=(1, 3, 3, 5)) == 1
    assert call(mask=None) == 1
    assert call(mask=66, kind=2) == 1             # fp32 mask not 4-byte aligned
    assert call(causal=1, off=3) == 1             # 3 + 3 rows > 5 keys
    assert call(kind=7) == 1
    assert call(Lq=0, shape=(1, 1, 1, 5)) == 0    # nothing to do
