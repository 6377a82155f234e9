"""indexer_decode_topk_noalloc: the decode top-k for callers that cannot
allocate device memory where they run it (inside stream capture, in serving
loops that forbid allocator calls, or with memory owned by another allocator).
It runs on the library's own scratch array. Its output must agree with
indexer_decode_topk's within the tolerance the parity tests use, on two calls
in a row (the second runs on whatever the first left in the scratch).
This file is collected last so that a run stopping at the first failure has
already run every other test."""
import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_attention_indexer_block_gb300 as saib
from _util import tolerance

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_attention_indexer_block_gb300 import build as libbuild
    libbuild.build()
    saib.load()
    torch.cuda.set_device(DEV)


def _agree(a, b, logits, tol_a, tol_b, k, length):
    """Two selections of one row agree when they differ only in keys whose
    membership the tolerance band leaves open."""
    if length <= k:
        assert np.array_equal(a, b)
        return
    assert len(np.unique(b)) == k and b.min() >= 0 and b.max() < length
    o = np.asarray(logits)[:length]
    tol = tolerance(tol_a, tol_b)[:length]
    hi, lo = o + tol, o - tol
    must = lo > np.sort(hi)[::-1][k]
    never = hi < np.sort(lo)[::-1][k - 1]
    diff = np.setxor1d(a, b)
    assert not (must[diff].any() or never[diff].any()), "selections differ beyond tolerance"


def test_noalloc_matches_workspace_path_on_two_calls():
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for seq_lens, seed in [([9000, 3000, 2048, 2500, 40000], 81), ([5000, 2049, 700], 82)]:
        d = synth.make_decode_from_lens(seq_lens, [1] * len(seq_lens), 1, seed=seed)
        q, w, cache = d.q.to(DEV), d.w.to(DEV), d.cache.to(DEV)
        bt = d.block_table.to(DEV)
        lens, _ = saib.indexer_expand_decode_rows(d.seq_lens.to(DEV), d.decode_lens.to(DEV), 1,
                                                  dev_error=err)
        ref = saib.indexer_decode_topk(q, w, cache, bt, lens, 1, 2048, dev_error=err)
        first = saib.indexer_decode_topk_noalloc(q, w, cache, bt, lens, 1, 2048, dev_error=err)
        second = saib.indexer_decode_topk_noalloc(q, w, cache, bt, lens, 1, 2048, dev_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        lens_h = lens.cpu().numpy()
        _, lg, ta, tb, rows = oracle.decode_topk(synth.bf16_bits(d.q), d.w.numpy(),
                                                 d.cache.numpy(), d.block_table.numpy(), lens_h,
                                                 1, 2048, want_logits=True)
        r0, r1, r2 = ref.cpu().numpy(), first.cpu().numpy(), second.cpu().numpy()
        for i, r in enumerate(rows):
            _agree(r0[r], r1[r], lg[i], ta[i], tb[i], 2048, int(lens_h[r]))
            _agree(r0[r], r2[r], lg[i], ta[i], tb[i], 2048, int(lens_h[r]))


def test_noalloc_rejects_batches_beyond_its_scratch():
    R = 8192  # the fp8 q images alone (8 KB per token row) fill the 64 MiB scratch
    assert saib.indexer_decode_workspace_bytes(R, 1, 2048) > 64 << 20
    q = torch.zeros((R, 64, 128), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((R, 64), dtype=torch.float32, device=DEV)
    cache = torch.zeros((1, 8448), dtype=torch.uint8, device=DEV)
    bt = torch.zeros((R, 1), dtype=torch.int32, device=DEV)
    lens = torch.zeros(R, dtype=torch.int32, device=DEV)
    with pytest.raises(saib.IndexerError) as e:
        saib.indexer_decode_topk_noalloc(q, w, cache, bt, lens, 1, 2048)
    assert e.value.status == 3
