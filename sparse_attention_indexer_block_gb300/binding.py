"""Thin ctypes binding of the indexer's C ABI (``include/indexer.h``).

Argument marshalling only: every function forwards torch tensors' device
pointers, sizes and the current CUDA stream to the function of the same name
in ``libsaib.so`` and raises :class:`IndexerError` on a non-OK status. Torch is
used for device memory (outputs and workspaces the caller did not pass) and
streams. There is no fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsaib.so")

IDX_OK = 0
STATUS_NAMES = {0: "IDX_OK", 1: "IDX_ERR_INVALID_ARG", 2: "IDX_ERR_UNSUPPORTED",
                3: "IDX_ERR_WORKSPACE", 4: "IDX_ERR_CUDA", 5: "IDX_ERR_CAPACITY"}
DEV_BAD_BLOCK, DEV_BAD_LEN, DEV_TIMEOUT, DEV_OVERFLOW = 1, 2, 4, 8
NUM_HEADS, HEAD_DIM, PAGE_TOKENS, PAGE_BYTES, MAX_TOPK = 64, 128, 64, 8448, 2048
DCP_MAX_CANDIDATES = 16384

# exported symbols and their ctypes signatures (kept in step with indexer.h)
_P, _I32, _I64, _SZ = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
SIGNATURES = {
    "indexer_status_string": (C.c_char_p, [C.c_int]),
    "indexer_last_cuda_error": (C.c_char_p, []),
    "indexer_expand_decode_rows": (C.c_int, [_P, _P, _I32, _I32, _P, _I64, _I32, _I32, _P, _P,
                                             _I64, _I64, _P, _P]),
    "indexer_quantize_q": (C.c_int, [_P, _P, _I64, _I32, _I32, _P, _P, _P]),
    "indexer_insert_keys": (C.c_int, [_P, _P, _I64, _I32, _P, _I64, _P, _P]),
    "indexer_decode_workspace_bytes": (C.c_int, [_I32, _I32, _I32, C.POINTER(_SZ)]),
    "indexer_decode_topk": (C.c_int, [_P, _P, _P, _I64, _P, _I64, _I32, _P, _I32, _I32, _I32,
                                      _I32, _I32, _P, _P, _SZ, _P, _P]),
    "indexer_decode_topk_from_lens": (C.c_int, [_P, _P, _P, _I64, _P, _I64, _I32, _P, _P, _I32,
                                                _I32, _I32, _I32, _I32, _P, _P, _SZ, _P, _P]),
    "indexer_decode_logits": (C.c_int, [_P, _P, _P, _I64, _P, _I64, _I32, _P, _I32, _I32, _I32,
                                        _I32, _I32, _P, _I64, _P, _SZ, _P, _P]),
    "indexer_plan_prefill_chunks": (C.c_int, [_P, _P, _I32, _I64, _I64, _P, _I32,
                                              C.POINTER(_I32)]),
    "indexer_prefill_workspace_bytes": (C.c_int, [_P, _P, _I32, _I32, _I64, _I64,
                                                  C.POINTER(_SZ)]),
    "indexer_prefill_topk": (C.c_int, [_P, _P, _P, _I64, _P, _I64, _I32, _P, _P, _P, _P, _I32,
                                       _I32, _I32, _I32, _I64, _I64, _P, _P, _SZ, _P, _P]),
    "indexer_profile_events": (C.c_int, [_P, _P]),
    "indexer_trace_buffer": (C.c_int, [_P, _SZ]),
    "indexer_debug_wait_limit": (C.c_int, [C.c_uint64, _I32]),
    "indexer_debug_divide": (C.c_int, [_P, _P, _I64, _P, _P, _P]),
    "indexer_debug_decode_plan": (C.c_int, [_I32, _I32, _I32, C.POINTER(_I64),
                                            C.POINTER(_I32), C.POINTER(_I32)]),
    "indexer_decode_topk_noalloc": (C.c_int, [_P, _P, _P, _I64, _P, _I64, _I32, _P, _I32, _I32,
                                              _I32, _I32, _I32, _P, _P, _P]),
    "indexer_index_key_counts": (C.c_int, [_P, _I64, _I32, _I32, _I32, _I32, _P, _P]),
    "indexer_decode_topk_values": (C.c_int, [_P, _P, _P, _I64, _P, _I64, _I32, _P, _I32, _I32,
                                             _I32, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P,
                                             _SZ, _P, _P]),
    "indexer_prefill_topk_values": (C.c_int, [_P, _P, _P, _I64, _P, _I64, _I32, _P, _P, _P, _P,
                                              _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                                              _I64, _I64, _P, _P, _P, _SZ, _P, _P]),
    "indexer_dcp_merge": (C.c_int, [_P, _P, _I32, _I64, _I32, _P, _P, _P]),
    "indexer_block_topk": (C.c_int, [_P, _I64, _P, _I64, _I32, _I32, _I32, _I32, _P, _I32, _P,
                                     _P]),
    "indexer_expand_pools": (C.c_int, [_P, _I32, _P, _P, _I64, _I32, _P, _I32, _P, _P]),
    "indexer_decode_topk_mxfp4": (C.c_int, [_P, _P, _P, _I64, _P, _I64, _I32, _P, _I32, _I32,
                                            _I32, _I32, _I32, _P, _P, _SZ, _P, _P]),
    "indexer_decode_logits_mxfp4": (C.c_int, [_P, _P, _P, _I64, _P, _I64, _I32, _P, _I32, _I32,
                                              _I32, _I32, _I32, _P, _I64, _P, _SZ, _P, _P]),
}

_lock = threading.Lock()
_lib = None


class IndexerError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        msg = f"{fn} failed: {STATUS_NAMES.get(status, status)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))
        self.status = status


def load(path: str = LIB_PATH):
    """Loads libsaib.so (build it with ``build.build()`` first)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"indexer CUDA library not built ({path}); run "
                               "sparse_attention_indexer_block_gb300.build.build()")
        lib = C.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return C.c_void_p(t)
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


def _check(name, st):
    if st != IDX_OK:
        detail = load().indexer_last_cuda_error().decode() if st == 4 else ""
        raise IndexerError(name, st, detail)


def _host_i32(t):
    import numpy as np
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().numpy()
    return np.ascontiguousarray(t, dtype=np.int32)


def indexer_status_string(status: int) -> str:
    return load().indexer_status_string(status).decode()


def indexer_expand_decode_rows(seq_lens, decode_lens, next_n: int, mode: int = 0,
                               block_table=None, row_seq_lens=None, row_block_table=None,
                               num_out_rows: int | None = None, want_block_table: bool = False,
                               dev_error=None, stream=None):
    R = int(seq_lens.shape[0])
    if num_out_rows is None:
        num_out_rows = R * next_n
    dev = seq_lens.device
    if row_seq_lens is None:
        row_seq_lens = torch.empty(num_out_rows, dtype=torch.int32, device=dev)
    W, bt_stride, out_stride = 0, 0, 0
    if block_table is not None:
        W = int(block_table.shape[1])
        bt_stride = int(block_table.stride(0))
        if row_block_table is None and want_block_table:
            row_block_table = torch.zeros((num_out_rows, W), dtype=torch.int32, device=dev)
        if row_block_table is not None:
            out_stride = int(row_block_table.stride(0))
    st = load().indexer_expand_decode_rows(
        _ptr(seq_lens), _ptr(decode_lens), R, next_n, _ptr(block_table), bt_stride, W, mode,
        _ptr(row_seq_lens), _ptr(row_block_table), out_stride, num_out_rows, _ptr(dev_error),
        _stream(stream))
    _check("indexer_expand_decode_rows", st)
    return row_seq_lens, row_block_table


def indexer_quantize_q(q, weights, q_fp8=None, weights_scaled=None, stream=None):
    rows = int(q.shape[0])
    if q_fp8 is None:
        q_fp8 = torch.empty((rows, NUM_HEADS, HEAD_DIM), dtype=torch.uint8, device=q.device)
    if weights_scaled is None:
        weights_scaled = torch.empty((rows, NUM_HEADS), dtype=torch.float32, device=q.device)
    st = load().indexer_quantize_q(_ptr(q), _ptr(weights), rows, int(q.shape[1]),
                                   int(q.shape[2]), _ptr(q_fp8), _ptr(weights_scaled),
                                   _stream(stream))
    _check("indexer_quantize_q", st)
    return q_fp8, weights_scaled


def indexer_insert_keys(k, slot_mapping, index_cache, dev_error=None, stream=None):
    """Quantises k (bf16 [T, 128]) per token and writes it into the paged
    index cache (uint8 [pages, 8448]) at slot_mapping (int64 [T]); in place."""
    st = load().indexer_insert_keys(_ptr(k), _ptr(slot_mapping), int(k.shape[0]), int(k.shape[1]),
                                    _ptr(index_cache), int(index_cache.shape[0]),
                                    _ptr(dev_error), _stream(stream))
    _check("indexer_insert_keys", st)
    return index_cache


def indexer_decode_workspace_bytes(num_reqs: int, next_n: int, topk: int) -> int:
    out = C.c_size_t(0)
    _check("indexer_decode_workspace_bytes",
           load().indexer_decode_workspace_bytes(num_reqs, next_n, topk, C.byref(out)))
    return int(out.value)


def decode_workspace(num_reqs: int, next_n: int, topk: int, device="cuda"):
    n = indexer_decode_workspace_bytes(num_reqs, next_n, topk)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def indexer_decode_topk(q, weights, index_cache, block_table, row_seq_lens, next_n: int,
                        topk: int = MAX_TOPK, out_idx=None, workspace=None, dev_error=None,
                        stream=None):
    R = int(block_table.shape[0])
    rows = R * next_n
    if out_idx is None:
        out_idx = torch.empty((rows, topk), dtype=torch.int32, device=q.device)
    if workspace is None:
        workspace = decode_workspace(R, next_n, topk, q.device)
    st = load().indexer_decode_topk(
        _ptr(q), _ptr(weights), _ptr(index_cache), int(index_cache.shape[0]), _ptr(block_table),
        int(block_table.stride(0)), int(block_table.shape[1]), _ptr(row_seq_lens), R, next_n,
        int(q.shape[1]), int(q.shape[2]), topk, _ptr(out_idx), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _ptr(dev_error), _stream(stream))
    _check("indexer_decode_topk", st)
    return out_idx


def indexer_decode_topk_from_lens(q, weights, index_cache, block_table, seq_lens, decode_lens,
                                  next_n: int, topk: int = MAX_TOPK, out_idx=None,
                                  workspace=None, dev_error=None, stream=None):
    """indexer_decode_topk with the row expansion done on the device by the
    launch itself: seq_lens, decode_lens int32 [num_reqs]."""
    R = int(block_table.shape[0])
    rows = R * next_n
    if out_idx is None:
        out_idx = torch.empty((rows, topk), dtype=torch.int32, device=q.device)
    if workspace is None:
        workspace = decode_workspace(R, next_n, topk, q.device)
    st = load().indexer_decode_topk_from_lens(
        _ptr(q), _ptr(weights), _ptr(index_cache), int(index_cache.shape[0]), _ptr(block_table),
        int(block_table.stride(0)), int(block_table.shape[1]), _ptr(seq_lens), _ptr(decode_lens),
        R, next_n, int(q.shape[1]), int(q.shape[2]), topk, _ptr(out_idx), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _ptr(dev_error), _stream(stream))
    _check("indexer_decode_topk_from_lens", st)
    return out_idx


def indexer_index_key_counts(row_seq_lens, compress_ratio: int = 1, dcp_rank: int = 0,
                             dcp_world: int = 1, dcp_interleave: int = 1, key_counts=None,
                             stream=None):
    """Cache entries each row sees on rank dcp_rank of a compressed and / or
    key-sharded cache (int32 tensors)."""
    n = int(row_seq_lens.numel())
    if key_counts is None:
        key_counts = torch.empty_like(row_seq_lens)
    st = load().indexer_index_key_counts(_ptr(row_seq_lens), n, compress_ratio, dcp_rank,
                                         dcp_world, dcp_interleave, _ptr(key_counts),
                                         _stream(stream))
    _check("indexer_index_key_counts", st)
    return key_counts


def indexer_decode_topk_values(q, weights, index_cache, block_table, row_seq_lens, next_n: int,
                               topk: int = MAX_TOPK, compress_ratio: int = 1, dcp_rank: int = 0,
                               dcp_world: int = 1, dcp_interleave: int = 1, out_idx=None,
                               out_val=None, workspace=None, dev_error=None, stream=None):
    """Top-k with the selected logits on one rank of a key-sharded cache
    (the whole cache when dcp_world == 1); indices in global positions.
    Returns (out_idx int32, out_val float32), both [rows, topk]."""
    R = int(block_table.shape[0])
    rows = R * next_n
    if out_idx is None:
        out_idx = torch.empty((rows, topk), dtype=torch.int32, device=q.device)
    if out_val is None:
        out_val = torch.empty((rows, topk), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = decode_workspace(R, next_n, topk, q.device)
    st = load().indexer_decode_topk_values(
        _ptr(q), _ptr(weights), _ptr(index_cache), int(index_cache.shape[0]), _ptr(block_table),
        int(block_table.stride(0)), int(block_table.shape[1]), _ptr(row_seq_lens), R, next_n,
        int(q.shape[1]), int(q.shape[2]), topk, compress_ratio, dcp_rank, dcp_world,
        dcp_interleave, _ptr(out_idx), _ptr(out_val), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _ptr(dev_error), _stream(stream))
    _check("indexer_decode_topk_values", st)
    return out_idx, out_val


def indexer_dcp_merge(cand_val, cand_idx, topk: int = MAX_TOPK, out_idx=None, out_val=None,
                      stream=None):
    """The top k of the ranks' candidates cand_val float32 / cand_idx int32
    [world, rows, topk]. Returns (out_idx, out_val) [rows, topk]."""
    world, rows = int(cand_idx.shape[0]), int(cand_idx.shape[1])
    if out_idx is None:
        out_idx = torch.empty((rows, topk), dtype=torch.int32, device=cand_idx.device)
    st = load().indexer_dcp_merge(_ptr(cand_val), _ptr(cand_idx), world, rows, topk,
                                  _ptr(out_idx), _ptr(out_val), _stream(stream))
    _check("indexer_dcp_merge", st)
    return out_idx, out_val


def indexer_decode_topk_mxfp4(q, weights, index_cache, block_table, row_seq_lens,
                              topk: int = MAX_TOPK, out_idx=None, workspace=None, dev_error=None,
                              stream=None):
    """Decode top-k (next_n = 1) over an MXFP4 cache uint8 [pages, 4352]."""
    R = int(block_table.shape[0])
    if out_idx is None:
        out_idx = torch.empty((R, topk), dtype=torch.int32, device=q.device)
    if workspace is None:
        workspace = decode_workspace(R, 1, topk, q.device)
    st = load().indexer_decode_topk_mxfp4(
        _ptr(q), _ptr(weights), _ptr(index_cache), int(index_cache.shape[0]), _ptr(block_table),
        int(block_table.stride(0)), int(block_table.shape[1]), _ptr(row_seq_lens), R, 1,
        int(q.shape[1]), int(q.shape[2]), topk, _ptr(out_idx), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _ptr(dev_error), _stream(stream))
    _check("indexer_decode_topk_mxfp4", st)
    return out_idx


def indexer_decode_logits_mxfp4(q, weights, index_cache, block_table, row_seq_lens,
                                topk: int = MAX_TOPK, out_logits=None, workspace=None,
                                dev_error=None, stream=None):
    R = int(block_table.shape[0])
    ld = int(block_table.shape[1]) * PAGE_TOKENS
    if out_logits is None:
        out_logits = torch.full((R, ld), float("nan"), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = decode_workspace(R, 1, topk, q.device)
    st = load().indexer_decode_logits_mxfp4(
        _ptr(q), _ptr(weights), _ptr(index_cache), int(index_cache.shape[0]), _ptr(block_table),
        int(block_table.stride(0)), int(block_table.shape[1]), _ptr(row_seq_lens), R, 1,
        int(q.shape[1]), int(q.shape[2]), topk, _ptr(out_logits), ld, _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _ptr(dev_error), _stream(stream))
    _check("indexer_decode_logits_mxfp4", st)
    return out_logits


def indexer_block_topk(logits, row_lens, block_size: int, topk_blocks: int, init_blocks: int = 0,
                       local_blocks: int = 0, out_cap: int | None = None, out=None, cnt=None,
                       stream=None):
    """Selected blocks per row (ascending, -1 after) and their counts."""
    rows = int(logits.shape[0])
    cap = out_cap or (topk_blocks + init_blocks + local_blocks)
    if out is None:
        out = torch.empty((rows, cap), dtype=torch.int32, device=logits.device)
    if cnt is None:
        cnt = torch.empty(rows, dtype=torch.int32, device=logits.device)
    st = load().indexer_block_topk(_ptr(logits), int(logits.stride(0)), _ptr(row_lens), rows,
                                   block_size, topk_blocks, init_blocks, local_blocks, _ptr(out),
                                   cap, _ptr(cnt), _stream(stream))
    _check("indexer_block_topk", st)
    return out, cnt


def indexer_expand_pools(pools, row_lens, pool_size: int, out_cap: int, pool_counts=None,
                         stream=None):
    """Token indices of the listed pools then each row's tail, and counts."""
    rows, pcap = int(pools.shape[0]), int(pools.shape[1])
    out = torch.empty((rows, out_cap), dtype=torch.int32, device=pools.device)
    cnt = torch.empty(rows, dtype=torch.int32, device=pools.device)
    st = load().indexer_expand_pools(_ptr(pools), pcap, _ptr(pool_counts), _ptr(row_lens), rows,
                                     pool_size, _ptr(out), out_cap, _ptr(cnt), _stream(stream))
    _check("indexer_expand_pools", st)
    return out, cnt


def indexer_decode_logits(q, weights, index_cache, block_table, row_seq_lens, next_n: int,
                          topk: int = MAX_TOPK, out_logits=None, workspace=None, dev_error=None,
                          stream=None):
    R = int(block_table.shape[0])
    rows = R * next_n
    ld = int(block_table.shape[1]) * PAGE_TOKENS
    if out_logits is None:
        out_logits = torch.full((rows, ld), float("nan"), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = decode_workspace(R, next_n, topk, q.device)
    st = load().indexer_decode_logits(
        _ptr(q), _ptr(weights), _ptr(index_cache), int(index_cache.shape[0]), _ptr(block_table),
        int(block_table.stride(0)), int(block_table.shape[1]), _ptr(row_seq_lens), R, next_n,
        int(q.shape[1]), int(q.shape[2]), topk, _ptr(out_logits), int(out_logits.stride(0)),
        _ptr(workspace), int(workspace.numel() * workspace.element_size()), _ptr(dev_error),
        _stream(stream))
    _check("indexer_decode_logits", st)
    return out_logits


def indexer_plan_prefill_chunks(seq_lens, query_lens, workspace_tokens: int,
                                logits_budget_bytes: int):
    import numpy as np
    sl, ql = _host_i32(seq_lens), _host_i32(query_lens)
    lib = load()
    cap = 64
    while True:
        buf = np.zeros((cap, 4), np.int32)
        n = C.c_int32(0)
        st = lib.indexer_plan_prefill_chunks(sl.ctypes.data, ql.ctypes.data, sl.shape[0],
                                             workspace_tokens, logits_budget_bytes,
                                             buf.ctypes.data, cap, C.byref(n))
        if st == 5:  # capacity
            cap = int(n.value)
            continue
        _check("indexer_plan_prefill_chunks", st)
        return [tuple(int(v) for v in buf[i]) for i in range(n.value)]


def indexer_prefill_workspace_bytes(seq_lens_host, query_lens_host, topk: int,
                                    workspace_tokens: int, logits_budget_bytes: int) -> int:
    sl, ql = _host_i32(seq_lens_host), _host_i32(query_lens_host)
    out = C.c_size_t(0)
    _check("indexer_prefill_workspace_bytes",
           load().indexer_prefill_workspace_bytes(sl.ctypes.data, ql.ctypes.data, sl.shape[0], topk,
                                                  workspace_tokens, logits_budget_bytes,
                                                  C.byref(out)))
    return int(out.value)


def indexer_prefill_topk(q, weights, index_cache, block_table, seq_lens, query_start_loc,
                         seq_lens_host, query_lens_host, topk: int = MAX_TOPK,
                         workspace_tokens: int = 40 * 8192, logits_budget_bytes: int = 512 << 20,
                         out_idx=None, workspace=None, dev_error=None, stream=None):
    sl, ql = _host_i32(seq_lens_host), _host_i32(query_lens_host)
    total_q = int(q.shape[0])
    if out_idx is None:
        out_idx = torch.empty((total_q, topk), dtype=torch.int32, device=q.device)
    if workspace is None:
        n = indexer_prefill_workspace_bytes(sl, ql, topk, workspace_tokens, logits_budget_bytes)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    st = load().indexer_prefill_topk(
        _ptr(q), _ptr(weights), _ptr(index_cache), int(index_cache.shape[0]), _ptr(block_table),
        int(block_table.stride(0)), int(block_table.shape[1]), _ptr(seq_lens),
        _ptr(query_start_loc), sl.ctypes.data, ql.ctypes.data, sl.shape[0], int(q.shape[1]),
        int(q.shape[2]), topk, workspace_tokens, logits_budget_bytes, _ptr(out_idx),
        _ptr(workspace), int(workspace.numel() * workspace.element_size()), _ptr(dev_error),
        _stream(stream))
    _check("indexer_prefill_topk", st)
    return out_idx


def indexer_prefill_topk_values(q, weights, index_cache, block_table, seq_lens, query_start_loc,
                                seq_lens_host, query_lens_host, topk: int = MAX_TOPK,
                                compress_ratio: int = 1, dcp_rank: int = 0, dcp_world: int = 1,
                                dcp_interleave: int = 1, workspace_tokens: int = 40 * 8192,
                                logits_budget_bytes: int = 512 << 20, out_idx=None, out_val=None,
                                workspace=None, dev_error=None, stream=None):
    """Prefill top-k with the selected logits on one rank of a compressed and
    / or key-sharded cache. Returns (out_idx int32, out_val float32)."""
    sl, ql = _host_i32(seq_lens_host), _host_i32(query_lens_host)
    total_q = int(q.shape[0])
    if out_idx is None:
        out_idx = torch.empty((total_q, topk), dtype=torch.int32, device=q.device)
    if out_val is None:
        out_val = torch.empty((total_q, topk), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = indexer_prefill_workspace_bytes(sl, ql, topk, workspace_tokens, logits_budget_bytes)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    st = load().indexer_prefill_topk_values(
        _ptr(q), _ptr(weights), _ptr(index_cache), int(index_cache.shape[0]), _ptr(block_table),
        int(block_table.stride(0)), int(block_table.shape[1]), _ptr(seq_lens),
        _ptr(query_start_loc), sl.ctypes.data, ql.ctypes.data, sl.shape[0], int(q.shape[1]),
        int(q.shape[2]), topk, compress_ratio, dcp_rank, dcp_world, dcp_interleave,
        workspace_tokens, logits_budget_bytes, _ptr(out_idx), _ptr(out_val), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _ptr(dev_error), _stream(stream))
    _check("indexer_prefill_topk_values", st)
    return out_idx, out_val


def indexer_profile_events(start_event=None, stop_event=None):
    """Records the given torch.cuda.Event pair around every score/select launch
    made from this thread (None, None turns it off)."""
    a = C.c_void_p(start_event.cuda_event) if start_event is not None else None
    b = C.c_void_p(stop_event.cuda_event) if stop_event is not None else None
    _check("indexer_profile_events", load().indexer_profile_events(a, b))


def indexer_trace_buffer(buffer=None):
    """Per-CTA trace stamps of later score/select launches go to ``buffer``
    (a uint64/int64 CUDA tensor of >= 128 * SM-count entries: 64 per tile
    stream, two streams per SM); None turns it off."""
    if buffer is None:
        _check("indexer_trace_buffer", load().indexer_trace_buffer(None, 0))
    else:
        _check("indexer_trace_buffer", load().indexer_trace_buffer(
            _ptr(buffer), int(buffer.numel() * buffer.element_size())))


def indexer_debug_decode_plan(num_reqs: int, next_n: int, topk: int = MAX_TOPK):
    """Where the decode work split lives in a workspace: returns (offsets
    dict of byte offsets, grid, (penalty, divisor))."""
    offs = (_I64 * 4)()
    grid = _I32(0)
    pen = (_I32 * 2)()
    _check("indexer_debug_decode_plan",
           load().indexer_debug_decode_plan(num_reqs, next_n, topk, offs, C.byref(grid), pen))
    names = ("wr_tile_start", "cta_tile", "row_ctas", "cta_row")
    return dict(zip(names, [int(v) for v in offs])), int(grid.value), (int(pen[0]), int(pen[1]))


def indexer_debug_divide(a, b, stream=None):
    """(the insert's quotient, the IEEE quotient) of float32 tensors a / b."""
    q = torch.empty_like(a)
    qi = torch.empty_like(a)
    st = load().indexer_debug_divide(_ptr(a), _ptr(b), int(a.numel()), _ptr(q), _ptr(qi),
                                     _stream(stream))
    _check("indexer_debug_divide", st)
    return q, qi


def indexer_debug_wait_limit(limit_ns: int = 0, stall_split_rows: bool = False):
    """Score/select launches from this thread give up their waits after
    ``limit_ns`` (0 restores the 2 s default); with ``stall_split_rows`` their
    split-row waits wait for a segment that never comes. For failure-detection
    tests."""
    _check("indexer_debug_wait_limit",
           load().indexer_debug_wait_limit(int(limit_ns), 1 if stall_split_rows else 0))


def indexer_decode_topk_noalloc(q, weights, index_cache, block_table, row_seq_lens, next_n: int,
                                topk: int = MAX_TOPK, out_idx=None, dev_error=None, stream=None):
    """indexer_decode_topk on the library's own scratch, for callers that
    cannot allocate a workspace (the output buffer is the caller's)."""
    R = int(block_table.shape[0])
    if out_idx is None:
        out_idx = torch.empty((R * next_n, topk), dtype=torch.int32, device=q.device)
    st = load().indexer_decode_topk_noalloc(
        _ptr(q), _ptr(weights), _ptr(index_cache), int(index_cache.shape[0]), _ptr(block_table),
        int(block_table.stride(0)), int(block_table.shape[1]), _ptr(row_seq_lens), R, next_n,
        int(q.shape[1]), int(q.shape[2]), topk, _ptr(out_idx), _ptr(dev_error), _stream(stream))
    _check("indexer_decode_topk_noalloc", st)
    return out_idx
