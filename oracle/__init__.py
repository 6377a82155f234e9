"""Plain CPU oracle of the sparse-attention indexer (test infrastructure).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``. The product library never imports
it and shares no code with it. The arithmetic lives in ``indexer_oracle.c``
(plain C, fp64 except the fp32 steps that decide the fp8 codes of q); this
module only builds it with gcc, loads it with ctypes and marshals numpy arrays.

Every function states the passage of the pages it restates; see the header of
``indexer_oracle.c`` for the readings taken where the pages are silent.
Parity pins: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle.py`` (library routines, closed forms, worked examples from
the pages, brute force, invariants).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "indexer_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

PAGE_TOKENS = 64
DIM = 128
PAGE_BYTES = PAGE_TOKENS * (DIM + 4)


def build(force: bool = False) -> str:
    """Compile ``indexer_oracle.c`` into ``liboracle.so`` next to it (gcc)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = C.CDLL(_LIB_PATH)
        P = C.c_void_p
        i32, i64, u8 = C.c_int32, C.c_int64, C.c_uint8
        lib.ora_e4m3_decode.restype = C.c_double
        lib.ora_e4m3_decode.argtypes = [u8]
        lib.ora_e4m3_encode.restype = u8
        lib.ora_e4m3_encode.argtypes = [C.c_float]
        lib.ora_quantize_q.restype = None
        lib.ora_quantize_q.argtypes = [P, P, i64, i32, i32, P, P, P]
        lib.ora_insert_keys.restype = None
        lib.ora_insert_keys.argtypes = [P, P, i64, P, i64]
        lib.ora_expand_rows.restype = i64
        lib.ora_expand_rows.argtypes = [P, P, i32, i32, i32, P, i64, i32, P, P, i64, i64]
        lib.ora_row_logits.restype = C.c_int
        lib.ora_row_logits.argtypes = [P, P, i32, i32, P, i64, P, i64, P, P, P]
        lib.ora_topk_row.restype = None
        lib.ora_topk_row.argtypes = [P, i64, i32, P]
        lib.ora_score_select_rows.restype = C.c_int
        lib.ora_score_select_rows.argtypes = [P, P, i32, i32, P, i64, P, i64, P, P, P, i64,
                                              i32, P, P, P, P, P, i32]
        lib.ora_num_threads.restype = C.c_int
        lib.ora_num_threads.argtypes = []
        lib.ora_plan_prefill_chunks.restype = i64
        lib.ora_plan_prefill_chunks.argtypes = [P, P, i32, i64, i64, P, i64]
        lib.ora_prefill_rows.restype = None
        lib.ora_prefill_rows.argtypes = [P, P, i32, P, P]
        lib.ora_e2m1_decode.restype = C.c_double
        lib.ora_e2m1_decode.argtypes = [u8]
        lib.ora_ue8m0_decode.restype = C.c_double
        lib.ora_ue8m0_decode.argtypes = [u8]
        lib.ora_e2m1_encode.restype = u8
        lib.ora_e2m1_encode.argtypes = [C.c_double]
        lib.ora_mxfp4_quantize_token.restype = None
        lib.ora_mxfp4_quantize_token.argtypes = [P, P]
        lib.ora_row_logits_mxfp4.restype = C.c_int
        lib.ora_row_logits_mxfp4.argtypes = [P, P, i32, i32, P, i64, P, i64, P, P, P]
        lib.ora_topk_row_values.restype = None
        lib.ora_topk_row_values.argtypes = [P, i64, i32, P, P]
        lib.ora_dcp_local_len.restype = i64
        lib.ora_dcp_local_len.argtypes = [i64, i32, i32, i32]
        lib.ora_dcp_global_index.restype = i64
        lib.ora_dcp_global_index.argtypes = [i64, i32, i32, i32]
        lib.ora_index_key_count.restype = i64
        lib.ora_index_key_count.argtypes = [i64, i32, i32, i32, i32]
        lib.ora_block_topk.restype = i32
        lib.ora_block_topk.argtypes = [P, i64, i32, i32, i32, i32, P, i32]
        lib.ora_expand_pools.restype = i32
        lib.ora_expand_pools.argtypes = [P, i32, i64, i32, P, i32]
        lib.ora_merge_candidates.restype = None
        lib.ora_merge_candidates.argtypes = [P, P, i64, i32, P, P]
        _lib = lib
        return lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return C.c_void_p(a.ctypes.data)


def num_threads() -> int:
    return int(_load().ora_num_threads())


# --------------------------------------------------------------------------
# fp8 e4m3fn codec (closed-form definition; no infinities, max 448)
# --------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.ora_e4m3_decode(int(x)) for x in c], dtype=np.float64).reshape(
        np.shape(codes))


def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even onto the e4m3fn grid, saturating at +-448."""
    lib = _load()
    v = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.ora_e4m3_encode(float(f)) for f in v], dtype=np.uint8).reshape(
        np.shape(x))


# --------------------------------------------------------------------------
# q quantisation (per token row and head)
# --------------------------------------------------------------------------

def quantize_q(q_bf16_bits: np.ndarray, w: np.ndarray):
    """q_bf16_bits: uint16 [rows, H, D] raw bf16; w: float32 [rows, H].

    Returns (q8 uint8 [rows, H, D], sq float64 [rows, H], wprime float64 [rows, H])
    with amax = max|q|, inv = 448/amax (fp32), q8 = e4m3(q*inv) (fp32 product),
    sq = amax/448, wprime = w*sq.
    """
    q = np.ascontiguousarray(q_bf16_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, H, D = q.shape
    q8 = np.empty((rows, H, D), np.uint8)
    sq = np.empty((rows, H), np.float64)
    wp = np.empty((rows, H), np.float64)
    _load().ora_quantize_q(_p(q), _p(w), rows, H, D, _p(q8), _p(sq), _p(wp))
    return q8, sq, wp


# --------------------------------------------------------------------------
# index-key cache insert
# --------------------------------------------------------------------------

def insert_keys(k_bf16_bits: np.ndarray, slots, cache: np.ndarray) -> np.ndarray:
    """Quantises each token of k (uint16 raw bf16 [n, 128]) with scale =
    amax/448 and codes e4m3(x/scale) (fp32 steps) into a copy of cache (uint8
    [pages, 8448]) at slots (int64 [n]; negative or out-of-range skipped).
    Restates the insert step behind the INDEXER page's slot_mapping."""
    k = np.ascontiguousarray(k_bf16_bits, dtype=np.uint16)
    sl = np.ascontiguousarray(slots, dtype=np.int64)
    out = np.array(cache, dtype=np.uint8, copy=True, order="C")
    _load().ora_insert_keys(_p(k), _p(sl), int(k.shape[0]), _p(out), int(out.shape[0]))
    return out


# --------------------------------------------------------------------------
# decode row expansion
# --------------------------------------------------------------------------

def expand_rows(seq_lens, decode_lens, next_n: int, mode: int = 0, block_table=None,
                num_out_rows: int | None = None):
    """mode 0: padded [R, next_n] grid; mode 1: flatten (sum d_b rows, zero tail).

    Returns (row_lens int32, row_block_table int32 or None, token_rows).
    """
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    dl = np.ascontiguousarray(decode_lens, dtype=np.int32)
    R = sl.shape[0]
    if num_out_rows is None:
        num_out_rows = R * next_n
    row_lens = np.zeros(num_out_rows, np.int32)
    row_bt = None
    W, stride, bt = 0, 0, None
    if block_table is not None:
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        W = bt.shape[1]
        stride = W
        row_bt = np.full((num_out_rows, W), -7, np.int32)
    n = _load().ora_expand_rows(_p(sl), _p(dl), R, next_n, mode, _p(bt), stride, W,
                                _p(row_lens), _p(row_bt), W, num_out_rows)
    if n < 0:
        raise ValueError("token rows do not fit in num_out_rows")
    return row_lens, row_bt, int(n)


# --------------------------------------------------------------------------
# scoring and selection
# --------------------------------------------------------------------------

def row_logits(q8_row, wprime_row, cache, bt_row, length: int):
    """Logits and tolerance magnitudes (A, B) of one token row, fp64."""
    q8_row = np.ascontiguousarray(q8_row, dtype=np.uint8)
    wp = np.ascontiguousarray(wprime_row, dtype=np.float64)
    cache = np.ascontiguousarray(cache, dtype=np.uint8)
    bt_row = np.ascontiguousarray(bt_row, dtype=np.int32)
    H, D = q8_row.shape
    lg = np.empty(max(length, 1), np.float64)
    ta = np.empty_like(lg)
    tb = np.empty_like(lg)
    rc = _load().ora_row_logits(_p(q8_row), _p(wp), H, D, _p(cache), cache.shape[0], _p(bt_row),
                                length, _p(lg), _p(ta), _p(tb))
    if rc != 0:
        raise ValueError(f"oracle: bad page id in block table (rc={rc})")
    return lg[:length], ta[:length], tb[:length]


# --------------------------------------------------------------------------
# MXFP4 index keys (e2m1 values in blocks of 32 sharing a ue8m0 scale)
# --------------------------------------------------------------------------

MX_TOKEN_BYTES = 68    # 64 bytes of packed e2m1 values + 4 ue8m0 block scales
MX_PAGE_BYTES = 64 * MX_TOKEN_BYTES


def e2m1_decode(codes) -> np.ndarray:
    """e2m1 value of each 4-bit code (closed form; no infinities, max 6)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.ora_e2m1_decode(int(x)) for x in c], dtype=np.float64).reshape(
        np.shape(codes))


def ue8m0_decode(codes) -> np.ndarray:
    """2^(E - 127) for each exponent byte (255: NaN)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.ora_ue8m0_decode(int(x)) for x in c], dtype=np.float64).reshape(
        np.shape(codes))


def e2m1_encode(x) -> np.ndarray:
    """Round-to-nearest-even onto the e2m1 grid, saturating at +-6."""
    lib = _load()
    v = np.asarray(x, dtype=np.float64).ravel()
    return np.array([lib.ora_e2m1_encode(float(f)) for f in v], dtype=np.uint8).reshape(
        np.shape(x))


def mxfp4_quantize(keys) -> np.ndarray:
    """MXFP4 entries uint8 [T, 68] of keys float32 [T, 128] (the MX
    shared-exponent rule per block of 32)."""
    k = np.ascontiguousarray(keys, dtype=np.float32)
    out = np.zeros((k.shape[0], MX_TOKEN_BYTES), np.uint8)
    lib = _load()
    for t in range(k.shape[0]):
        lib.ora_mxfp4_quantize_token(_p(k[t]), _p(out[t]))
    return out


def mxfp4_values(entries) -> np.ndarray:
    """float64 [T, 128] key values of MXFP4 entries uint8 [T, 68]."""
    e = np.asarray(entries, dtype=np.uint8)
    codes = np.empty(e.shape[:-1] + (128,), np.uint8)
    codes[..., 0::2] = e[..., :64] & 0xF
    codes[..., 1::2] = e[..., :64] >> 4
    table = e2m1_decode(np.arange(16, dtype=np.uint8))
    scales = ue8m0_decode(e[..., 64:68])
    return table[codes] * np.repeat(scales, 32, axis=-1)


def row_logits_mxfp4(q8_row, wprime_row, cache, bt_row, length: int):
    """Logits and tolerance magnitudes (A, B) of one token row over an MXFP4
    cache uint8 [pages, 4352], fp64."""
    q8_row = np.ascontiguousarray(q8_row, dtype=np.uint8)
    wp = np.ascontiguousarray(wprime_row, dtype=np.float64)
    cache = np.ascontiguousarray(cache, dtype=np.uint8)
    bt_row = np.ascontiguousarray(bt_row, dtype=np.int32)
    H, D = q8_row.shape
    lg = np.empty(max(length, 1), np.float64)
    ta = np.empty_like(lg)
    tb = np.empty_like(lg)
    rc = _load().ora_row_logits_mxfp4(_p(q8_row), _p(wp), H, D, _p(cache), cache.shape[0],
                                      _p(bt_row), length, _p(lg), _p(ta), _p(tb))
    if rc != 0:
        raise ValueError(f"oracle: bad page id in block table (rc={rc})")
    return lg[:length], ta[:length], tb[:length]


def decode_topk_mxfp4(q_bf16_bits, w, cache, block_table, row_lens, next_n: int, k: int):
    """Decode top-k over an MXFP4 cache: row r = b * next_n + j reads
    block-table row b; rows with len <= k give the causal row."""
    q8, _, wp = quantize_q(q_bf16_bits, w)
    rows = np.asarray(row_lens).shape[0]
    out = np.empty((rows, k), np.int32)
    for r in range(rows):
        L = int(row_lens[r])
        lg, _, _ = row_logits_mxfp4(q8[r], wp[r], cache, block_table[r // next_n], L)
        out[r] = topk_row(lg, L, k)
    return out


def topk_row(logits, length: int, k: int) -> np.ndarray:
    lg = np.ascontiguousarray(logits, dtype=np.float64)
    out = np.empty(k, np.int32)
    _load().ora_topk_row(_p(lg), length, k, _p(out))
    return out


def score_select_rows(q8, wprime, cache, block_table, qrows, bt_rows, lens, k: int | None,
                      want_logits: bool = False, threads: int = 0):
    """Scores (and selects top-k of) token rows in parallel.

    q8 [rows, H, D], wprime [rows, H]; qrows[i] picks the q row, bt_rows[i] the
    block-table row and lens[i] the key count of output row i. Returns
    (out_idx [n, k] or None, logits list or None, tol_a list, tol_b list).
    """
    q8 = np.ascontiguousarray(q8, dtype=np.uint8)
    wp = np.ascontiguousarray(wprime, dtype=np.float64)
    cache = np.ascontiguousarray(cache, dtype=np.uint8)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    qrows = np.ascontiguousarray(qrows, dtype=np.int64)
    bt_rows = np.ascontiguousarray(bt_rows, dtype=np.int64)
    lens = np.ascontiguousarray(lens, dtype=np.int64)
    n = lens.shape[0]
    H, D = q8.shape[1], q8.shape[2]
    out = np.empty((n, k), np.int32) if k is not None else None
    off = lg = ta = tb = None
    if want_logits:
        off = np.zeros(n, np.int64)
        if n > 1:
            off[1:] = np.cumsum(lens[:-1])
        total = int(lens.sum())
        lg = np.zeros(max(total, 1), np.float64)
        ta = np.zeros_like(lg)
        tb = np.zeros_like(lg)
    rc = _load().ora_score_select_rows(
        _p(q8), _p(wp), H, D, _p(cache), cache.shape[0], _p(bt), bt.shape[1], _p(qrows),
        _p(bt_rows), _p(lens), n, k if k is not None else 0, _p(out), _p(off), _p(lg), _p(ta),
        _p(tb), threads)
    if rc != 0:
        raise ValueError(f"oracle: bad page id in block table (rc={rc})")
    if not want_logits:
        return out, None, None, None
    split = lambda a: [a[o:o + l] for o, l in zip(off, lens)]
    return out, split(lg), split(ta), split(tb)


def decode_topk(q_bf16_bits, w, cache, block_table, row_lens, next_n: int, k: int,
                rows=None, want_logits: bool = False, threads: int = 0):
    """The decode indexer for token rows laid out as a [R, next_n] grid (row
    b*next_n + j uses block-table row b). ``rows`` restricts the work to a
    sample of token rows. Returns (out_idx [n, k], logits, tol_a, tol_b, rows)."""
    q8, _, wp = quantize_q(q_bf16_bits, w)
    row_lens = np.asarray(row_lens, dtype=np.int64)
    if rows is None:
        rows = np.arange(row_lens.shape[0], dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    out, lg, ta, tb = score_select_rows(q8, wp, cache, block_table, rows, rows // next_n,
                                        row_lens[rows], k, want_logits, threads)
    return out, lg, ta, tb, rows


# --------------------------------------------------------------------------
# key-sharded (decode context parallel) decode
# --------------------------------------------------------------------------

def topk_row_values(logits, length: int, k: int):
    """(indices int32 [k], logits float64 [k]) of a row: all keys when
    length <= k (-1 / -inf past length), else the k best."""
    lg = np.ascontiguousarray(logits, dtype=np.float64)
    out = np.empty(k, np.int32)
    val = np.empty(k, np.float64)
    _load().ora_topk_row_values(_p(lg), length, k, _p(out), _p(val))
    return out, val


def dcp_local_lens(lens, rank: int, world: int, interleave: int) -> np.ndarray:
    """Rank `rank`'s key count of each length (the INDEXER page's DCP rule)."""
    lib = _load()
    a = np.asarray(lens, dtype=np.int64).ravel()
    return np.array([lib.ora_dcp_local_len(int(L), rank, world, interleave) for L in a],
                    dtype=np.int64).reshape(np.shape(lens))


def index_key_counts(lens, ratio: int = 1, rank: int = 0, world: int = 1,
                     interleave: int = 1) -> np.ndarray:
    """Cache entries a row of each length sees: one per `ratio` tokens (a
    compressed cache), then rank `rank`'s local count of them."""
    lib = _load()
    a = np.asarray(lens, dtype=np.int64).ravel()
    return np.array([lib.ora_index_key_count(int(L), ratio, rank, world, interleave) for L in a],
                    dtype=np.int64).reshape(np.shape(lens))


def dcp_global_index(local, rank: int, world: int, interleave: int) -> np.ndarray:
    """Global token of each of rank `rank`'s local keys (negative stays -1)."""
    lib = _load()
    a = np.asarray(local, dtype=np.int64).ravel()
    return np.array([lib.ora_dcp_global_index(int(j), rank, world, interleave) if j >= 0 else -1
                     for j in a], dtype=np.int64).reshape(np.shape(local))


def merge_candidates(vals, idx, k: int):
    """Per row: the k best (logit desc, index asc) of candidates vals / idx
    [..., rows, n] flattened over the leading axes per row (idx < 0 empty)."""
    v = np.asarray(vals, dtype=np.float64)
    x = np.asarray(idx, dtype=np.int32)
    rows = v.shape[-2]
    v = np.ascontiguousarray(np.moveaxis(v, -2, 0).reshape(rows, -1))
    x = np.ascontiguousarray(np.moveaxis(x, -2, 0).reshape(rows, -1))
    out = np.empty((rows, k), np.int32)
    ov = np.empty((rows, k), np.float64)
    lib = _load()
    for r in range(rows):
        lib.ora_merge_candidates(_p(v[r]), _p(x[r]), v.shape[1], k, _p(out[r]), _p(ov[r]))
    return out, ov


def dcp_rank_topk_values(q_bf16_bits, w, cache, block_table, row_lens, next_n: int, k: int,
                         rank: int, world: int, interleave: int, ratio: int = 1,
                         bt_rows=None):
    """One rank's part: for token row r (block-table row r // next_n of the
    rank's local cache, or bt_rows[r]) the top k of its local keys (the
    rank's count of row_lens[r] // ratio entries) with their logits, the
    indices in global entry positions. Returns (idx [rows, k], val [rows, k],
    local lens, logits list, tol_a list, tol_b list) (logits over local keys)."""
    q8, _, wp = quantize_q(q_bf16_bits, w)
    local = index_key_counts(np.asarray(row_lens, dtype=np.int64), ratio, rank, world,
                             interleave)
    rows = local.shape[0]
    if bt_rows is None:
        bt_rows = np.arange(rows) // next_n
    out = np.empty((rows, k), np.int32)
    val = np.empty((rows, k), np.float64)
    lgs, tas, tbs = [], [], []
    for r in range(rows):
        L = int(local[r])
        lg, ta, tb = row_logits(q8[r], wp[r], cache, block_table[bt_rows[r]], L)
        o, v = topk_row_values(lg, L, k)
        out[r] = dcp_global_index(o, rank, world, interleave)
        val[r] = v
        lgs.append(lg)
        tas.append(ta)
        tbs.append(tb)
    return out, val, local, lgs, tas, tbs


def dcp_decode_topk(q_bf16_bits, w, shards, row_lens, next_n: int, k: int, interleave: int,
                    ratio: int = 1, bt_rows=None):
    """Key-sharded decode top-k: shards[r] = (cache, block_table) of rank r
    (its local keys in order); each rank's candidates, then their merge.
    Returns (idx [rows, k] by (logit desc, index asc), val [rows, k])."""
    world = len(shards)
    vals, idxs = [], []
    for rank, (cache, bt) in enumerate(shards):
        o, v, *_ = dcp_rank_topk_values(q_bf16_bits, w, cache, bt, row_lens, next_n, k, rank,
                                        world, interleave, ratio, bt_rows)
        vals.append(v)
        idxs.append(o)
    return merge_candidates(np.stack(vals), np.stack(idxs), k)


def dcp_prefill_topk(q_bf16_bits, w, shards, seq_lens, query_start_loc, k: int,
                     interleave: int, ratio: int = 1):
    """Key-sharded (and compressed) prefill top-k: query i of request r sees
    the rank's local count of (L - Q + 1 + i) // ratio cache entries on each
    rank (INDEXER page, _build_prefill_chunk_metadata_kernel with
    COMPRESS_RATIO and the DCP branch); the ranks' candidates are merged.
    Returns (idx [rows, k] by (logit desc, index asc), val [rows, k])."""
    req, ln = prefill_rows(seq_lens, query_start_loc)
    return dcp_decode_topk(q_bf16_bits, w, shards, ln, 1, k, interleave, ratio, bt_rows=req)


# --------------------------------------------------------------------------
# block / pool selection
# --------------------------------------------------------------------------

def block_topk(logits, length: int, block: int, k: int, n_init: int = 0, n_local: int = 0,
               cap: int | None = None):
    """Selected blocks of one row (ascending, -1 after) and their count: the
    first n_init and last n_local blocks of `block` tokens plus the k best of
    the others by their largest logit."""
    lg = np.ascontiguousarray(logits, dtype=np.float64)
    cap = k + n_init + n_local if cap is None else cap
    out = np.empty(max(cap, 1), np.int32)
    n = _load().ora_block_topk(_p(lg), length, block, k, n_init, n_local, _p(out), cap)
    return out[:cap], int(n)


def expand_pools(pools, length: int, pool: int, cap: int):
    """Tokens of the selected complete pools, then the row's tail after its
    last complete pool (-1 after them), and their count."""
    pl = np.ascontiguousarray(pools, dtype=np.int32)
    out = np.empty(max(cap, 1), np.int32)
    n = _load().ora_expand_pools(_p(pl), pl.shape[0], length, pool, _p(out), cap)
    return out[:cap], int(n)


# --------------------------------------------------------------------------
# prefill
# --------------------------------------------------------------------------

def plan_prefill_chunks(seq_lens, query_lens, workspace_tokens: int, logits_budget_bytes: int):
    """Greedy chunk plan: list of (req_begin, req_end, q_begin, q_end)."""
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    ql = np.ascontiguousarray(query_lens, dtype=np.int32)
    cap = 16
    while True:
        buf = np.zeros((cap, 4), np.int32)
        n = _load().ora_plan_prefill_chunks(_p(sl), _p(ql), sl.shape[0], workspace_tokens,
                                            logits_budget_bytes, _p(buf), cap)
        if n >= 0:
            return [tuple(int(v) for v in buf[i]) for i in range(n)]
        cap *= 4


def prefill_rows(seq_lens, query_start_loc):
    """Per query token: (request id, number of visible keys)."""
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    total = int(qsl[-1])
    req = np.zeros(total, np.int64)
    ln = np.zeros(total, np.int64)
    _load().ora_prefill_rows(_p(sl), _p(qsl), sl.shape[0], _p(req), _p(ln))
    return req, ln


def prefill_topk(q_bf16_bits, w, cache, block_table, seq_lens, query_start_loc, k: int,
                 rows=None, want_logits: bool = False, threads: int = 0):
    """The prefill indexer: query token i of request r sees keys [0, len_i).
    Chunking does not change the result, so the oracle scores rows directly."""
    q8, _, wp = quantize_q(q_bf16_bits, w)
    req, ln = prefill_rows(seq_lens, query_start_loc)
    if rows is None:
        rows = np.arange(ln.shape[0], dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    out, lg, ta, tb = score_select_rows(q8, wp, cache, block_table, rows, req[rows], ln[rows],
                                        k, want_logits, threads)
    return out, lg, ta, tb, rows
