"""The C ABI library without a GPU: it loads, exports every declared entry
point, plans prefill chunks exactly as the oracle does, and rejects bad
arguments before touching the device."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle
import sparse_attention_indexer_block_gb300 as saib
from sparse_attention_indexer_block_gb300 import binding
from sparse_attention_indexer_block_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return saib.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "indexer.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(indexer_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), f"libsaib.so does not export {n}"
    assert set(names) == set(binding.SIGNATURES), "binding and header disagree"


def _declarations():
    """name -> list of parameter type strings, parsed from the header."""
    text = open(os.path.join(ROOT, "include", "indexer.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(indexer_\w+)\s*\(([^)]*)\)\s*;", text):
        params = [p.strip() for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        out[m.group(1)] = [re.sub(r"\s*\b\w+$", "", p) if not p.endswith("*") else p
                           for p in params]
    return out


def _kind(ctype):
    if ctype in (C.c_void_p, C.c_char_p) or (isinstance(ctype, type) and
                                            issubclass(ctype, C._Pointer)):
        return "ptr"
    return f"int{C.sizeof(ctype) * 8}"


def _header_kind(t):
    if "*" in t:
        return "ptr"
    base = t.replace("const", "").strip()
    return {"int32_t": "int32", "idx_status": "int32", "int64_t": "int64",
            "uint64_t": "int64", "size_t": "int64"}[base]


def test_binding_signatures_match_header_parameters():
    """Every binding signature has the header's parameter count, and each
    parameter the same kind (pointer, 32- or 64-bit integer), so a call cannot
    shift or truncate an argument."""
    decls = _declarations()
    assert set(decls) == set(binding.SIGNATURES)
    for name, params in decls.items():
        _, argtypes = binding.SIGNATURES[name]
        assert len(argtypes) == len(params), f"{name}: {len(argtypes)} vs {len(params)}"
        for i, (t, a) in enumerate(zip(params, argtypes)):
            assert _header_kind(t) == _kind(a), f"{name} parameter {i}: {t} vs {a}"


def test_status_strings(lib):
    assert saib.indexer_status_string(0) == "ok"
    assert saib.indexer_status_string(3) == "workspace too small"


def _golden_plans():
    path = os.path.join(ROOT, "tests", "golden", "prefill_chunk_plans.txt")
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        _, rest = line.split(" ", 1)
        name, sl, ql, ws, budget, _plan = [x.strip() for x in rest.split("|")]
        yield [int(x) for x in sl.split()], [int(x) for x in ql.split()], int(ws), int(budget)


def test_planner_matches_oracle_bit_exact(lib):
    cases = list(_golden_plans())
    rng = np.random.default_rng(8)
    for _ in range(400):
        n = int(rng.integers(0, 14))
        sl = rng.integers(0, 9000, n)
        ql = np.minimum(rng.integers(0, 4000, n), sl)
        cases.append((sl, ql, int(rng.integers(1, 30000)), int(rng.integers(4, 4 * 10 ** 8))))
    for sl, ql, ws, budget in cases:
        got = saib.indexer_plan_prefill_chunks(sl, ql, ws, budget)
        assert got == oracle.plan_prefill_chunks(sl, ql, ws, budget)


def test_planner_capacity_status(lib):
    sl = np.array([1000], np.int32)
    ql = np.array([100], np.int32)
    buf = np.zeros((2, 4), np.int32)
    n = C.c_int32(0)
    st = lib.indexer_plan_prefill_chunks(sl.ctypes.data, ql.ctypes.data, 1, 10 ** 6, 40000,
                                         buf.ctypes.data, 2, C.byref(n))
    assert st == 5 and n.value == 10


FAKE = 1 << 20  # an aligned non-null address; these calls fail before using it


def _decode(lib, **over):
    a = dict(q=FAKE, w=FAKE, cache=FAKE, pages=10, bt=FAKE, bt_stride=4, bt_width=4, lens=FAKE,
             R=2, next_n=1, H=64, D=128, k=2048, out=FAKE, ws=FAKE, ws_bytes=1 << 40, err=None)
    a.update(over)
    return lib.indexer_decode_topk(a["q"], a["w"], a["cache"], a["pages"], a["bt"], a["bt_stride"],
                                   a["bt_width"], a["lens"], a["R"], a["next_n"], a["H"], a["D"],
                                   a["k"], a["out"], a["ws"], a["ws_bytes"], a["err"], None)


def test_decode_argument_validation(lib):
    assert _decode(lib, q=None) == 1
    assert _decode(lib, H=32) == 2
    assert _decode(lib, D=64) == 2
    assert _decode(lib, k=0) == 2
    assert _decode(lib, k=2049) == 2
    assert _decode(lib, next_n=3) == 2
    assert _decode(lib, bt_stride=2) == 1
    assert _decode(lib, pages=0) == 1
    assert _decode(lib, q=FAKE + 8) == 1          # q must be 16-byte aligned
    assert _decode(lib, ws=FAKE + 16) == 1        # workspace must be 256-byte aligned
    assert _decode(lib, ws_bytes=16) == 3         # too small
    assert _decode(lib, R=0) == 0                 # nothing to do


def test_expand_and_quantize_validation(lib):
    f = lib.indexer_expand_decode_rows
    assert f(FAKE, FAKE, 2, 1, None, 0, 0, 2, FAKE, None, 0, 2, None, None) == 1   # bad mode
    assert f(FAKE, FAKE, 2, 2, None, 0, 0, 0, FAKE, None, 0, 3, None, None) == 5   # grid too small
    assert f(None, FAKE, 2, 1, None, 0, 0, 0, FAKE, None, 0, 2, None, None) == 1
    q = lib.indexer_quantize_q
    assert q(FAKE, FAKE, 4, 32, 128, FAKE, FAKE, None) == 2
    assert q(FAKE, FAKE, -1, 64, 128, FAKE, FAKE, None) == 1
    assert q(FAKE, FAKE, 0, 64, 128, FAKE, FAKE, None) == 0


def test_insert_keys_validation(lib):
    f = lib.indexer_insert_keys
    assert f(FAKE, FAKE, 4, 64, FAKE, 8, None, None) == 2      # head_dim must be 128
    assert f(FAKE, FAKE, -1, 128, FAKE, 8, None, None) == 1    # negative count
    assert f(FAKE, FAKE, 4, 128, FAKE, -1, None, None) == 1    # negative page count
    assert f(None, FAKE, 4, 128, FAKE, 8, None, None) == 1     # missing keys
    assert f(FAKE, FAKE, 4, 128, FAKE + 8, 8, None, None) == 1  # cache not 16-byte aligned
    assert f(FAKE, FAKE, 0, 128, FAKE, 8, None, None) == 0     # nothing to do


def test_prefill_validation(lib):
    sl = np.array([10, 5], np.int32)
    ql = np.array([11, 5], np.int32)   # query_len > seq_len is invalid
    out = C.c_size_t(0)
    st = lib.indexer_prefill_workspace_bytes(sl.ctypes.data, ql.ctypes.data, 2, 2048, 1000,
                                             1 << 20, C.byref(out))
    assert st == 1


def _values(lib, **over):
    a = dict(q=FAKE, w=FAKE, cache=FAKE, pages=10, bt=FAKE, bt_stride=4, bt_width=4, lens=FAKE,
             R=2, next_n=1, H=64, D=128, k=2048, ratio=1, rank=0, world=2, inter=64, out=FAKE,
             val=FAKE, ws=FAKE, ws_bytes=16, err=None)
    a.update(over)
    return lib.indexer_decode_topk_values(
        a["q"], a["w"], a["cache"], a["pages"], a["bt"], a["bt_stride"], a["bt_width"], a["lens"],
        a["R"], a["next_n"], a["H"], a["D"], a["k"], a["ratio"], a["rank"], a["world"],
        a["inter"], a["out"], a["val"], a["ws"], a["ws_bytes"], a["err"], None)


def test_key_sharded_argument_validation(lib):
    # the checks come before any device work (ws_bytes = 16 ends a valid call
    # at the workspace check)
    assert _values(lib) == 3
    assert _values(lib, val=None) == 1
    assert _values(lib, world=0) == 1
    assert _values(lib, rank=2) == 1
    assert _values(lib, rank=-1) == 1
    assert _values(lib, inter=0) == 1
    assert _values(lib, ratio=0) == 1
    assert _values(lib, H=32) == 2
    assert _values(lib, R=0) == 0
    f = lib.indexer_index_key_counts
    assert f(FAKE, 4, 1, 0, 0, 1, FAKE, None) == 1      # world < 1
    assert f(FAKE, 4, 1, 2, 2, 1, FAKE, None) == 1      # rank >= world
    assert f(FAKE, 4, 1, 0, 2, 0, FAKE, None) == 1      # interleave < 1
    assert f(FAKE, 4, 0, 0, 2, 1, FAKE, None) == 1      # ratio < 1
    assert f(None, 4, 1, 0, 2, 1, FAKE, None) == 1
    assert f(FAKE, -1, 1, 0, 2, 1, FAKE, None) == 1
    assert f(FAKE, 0, 1, 0, 2, 1, FAKE, None) == 0      # nothing to do
    sl = np.array([10, 5], np.int32)
    ql = np.array([4, 5], np.int32)
    p = lib.indexer_prefill_topk_values
    base = [FAKE, FAKE, FAKE, 10, FAKE, 4, 4, FAKE, FAKE, sl.ctypes.data, ql.ctypes.data, 2, 64,
            128, 2048]
    tail = [1000, 1 << 20, FAKE, FAKE, FAKE, 16, None, None]
    assert p(*base, 1, 0, 2, 64, *tail) == 3             # valid up to the workspace size
    assert p(*base, 0, 0, 2, 64, *tail) == 1             # ratio < 1
    assert p(*base, 1, 2, 2, 64, *tail) == 1             # rank >= world
    assert p(*base, 4, 0, 1, 1, *tail[:3], None, *tail[4:]) == 1   # no out_val
    m = lib.indexer_dcp_merge
    assert m(FAKE, FAKE, 9, 4, 2048, FAKE, None, None) == 2   # 9 * 2048 > 16384 candidates
    assert m(FAKE, FAKE, 2, 4, 0, FAKE, None, None) == 2
    assert m(FAKE, FAKE, 2, 4, 2049, FAKE, None, None) == 2
    assert m(FAKE, FAKE, 0, 4, 64, FAKE, None, None) == 1
    assert m(None, FAKE, 2, 4, 64, FAKE, None, None) == 1
    assert m(FAKE, FAKE, 2, 0, 64, FAKE, None, None) == 0


def test_mxfp4_argument_validation(lib):
    f = lib.indexer_decode_topk_mxfp4
    args = [FAKE, FAKE, FAKE, 10, FAKE, 4, 4, FAKE, 2]
    tail = [64, 128, 2048, FAKE, FAKE, 16, None, None]
    assert f(*args, 2, *tail) == 2                    # next_n must be 1
    assert f(*args, 1, *tail) == 3                    # valid up to the workspace size
    assert f(FAKE, FAKE, FAKE + 8, 10, FAKE, 4, 4, FAKE, 2, 1, *tail) == 1   # cache alignment


def test_block_selection_argument_validation(lib):
    f = lib.indexer_block_topk
    assert f(FAKE, 4096, FAKE, 2, 0, 4, 0, 0, FAKE, 4, None, None) == 1       # block size 0
    assert f(FAKE, 4096, FAKE, 2, 64, -1, 0, 0, FAKE, 4, None, None) == 1     # negative k
    assert f(FAKE, 4096, FAKE, 2, 64, 4, 0, 0, FAKE, 0, None, None) == 1      # no output room
    assert f(FAKE, 1 << 21, FAKE, 2, 64, 4, 0, 0, FAKE, 4, None, None) == 2   # > 16384 blocks
    assert f(None, 4096, FAKE, 2, 64, 4, 0, 0, FAKE, 4, None, None) == 1
    assert f(FAKE, 4096, FAKE, 0, 64, 4, 0, 0, FAKE, 4, None, None) == 0      # nothing to do
    g = lib.indexer_expand_pools
    assert g(FAKE, 4, None, FAKE, 2, 0, FAKE, 16, None, None) == 1            # pool size 0
    assert g(FAKE, 4, None, None, 2, 64, FAKE, 16, None, None) == 1
    assert g(FAKE, 4, None, FAKE, 0, 64, FAKE, 16, None, None) == 0
