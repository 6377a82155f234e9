"""Key-sharded (decode context parallel) decode on the GPU vs the CPU oracle.

The rank-local counts are bit-exact; the top-k with values is checked like
the top-k (tolerance band around the k-th value) plus every returned logit
against the oracle's; the merge is exact on distinct values; the whole
sharded path (every rank's call on its own cache, then the merge) is checked
against the unsharded oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_attention_indexer_block_gb300 as saib
from _util import check_logits, check_topk_row

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_attention_indexer_block_gb300 import build as libbuild
    libbuild.build()
    saib.load()
    torch.cuda.set_device(DEV)


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _inputs(seq, dl, next_n, seed):
    d = synth.make_decode_from_lens(np.asarray(seq, np.int32), np.asarray(dl, np.int32), next_n,
                                    seed=seed, device=DEV)
    lens, _, _ = oracle.expand_rows(np.asarray(seq, np.int32), np.asarray(dl, np.int32), next_n)
    return d, lens


def _check_values_rows(idx, val, lens, lg, ta, tb, k):
    """Rows of a values output against the oracle's logits of the same keys
    (lg / ta / tb per row, over the row's keys). Returns the worst open count."""
    worst = 0
    for r in range(idx.shape[0]):
        L = int(lens[r])
        sel, v = idx[r], val[r]
        n = min(L, k)
        valid = sel >= 0
        assert valid.sum() == n, f"row {r}: {valid.sum()} indices for {L} keys"
        assert np.all(np.isneginf(v[~valid])), f"row {r}: empty slots must hold -inf"
        s = sel[valid]
        if L <= k:
            assert np.array_equal(np.sort(s), np.arange(L)), f"row {r}: short row not whole"
        else:
            worst = max(worst, check_topk_row(s, lg[r], ta[r], tb[r], k, L))
        if n:
            check_logits(v[valid], lg[r][s], ta[r][s], tb[r][s])
    return worst


# ---------------------------------------------------------------------------
# local key counts: bit-exact
# ---------------------------------------------------------------------------

def test_index_key_counts_bit_exact():
    rng = np.random.default_rng(40)
    lens = np.concatenate([np.arange(0, 600), rng.integers(0, 1 << 20, 3000)]).astype(np.int32)
    lt = torch.from_numpy(lens).to(DEV)
    for ratio in (1, 4):
        for world, inter in ((1, 1), (2, 1), (2, 64), (3, 5), (4, 64), (8, 1), (8, 256)):
            for rank in range(world):
                got = saib.indexer_index_key_counts(lt, ratio, rank, world, inter)
                torch.cuda.synchronize()
                ref = oracle.index_key_counts(lens, ratio, rank, world, inter)
                assert np.array_equal(got.cpu().numpy(), ref), (ratio, world, inter, rank)


# ---------------------------------------------------------------------------
# top-k with values (one rank, or the whole cache)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", ["mixed", "short_split", "two_token"])
def test_topk_values_whole_cache_matches_oracle(case):
    k = 2048
    if case == "mixed":      # empty, short, k - 1 .. k + 1, long rows split over many CTAs
        seq, dl, nn = [0, 1, 100, 2047, 2048, 2049, 5000, 40000, 300], [1] * 9, 1
    elif case == "short_split":  # few short rows: their tiles spread over many CTAs
        seq, dl, nn = [2000, 1500, 2048, 700, 1, 129], [1] * 6, 1
    else:
        seq, dl, nn = [3000, 20000, 2048, 5, 9000, 64], [2, 1, 2, 2, 1, 2], 2
    d, lens = _inputs(seq, dl, nn, seed=50 + len(case))
    err = _err()
    lens_d = torch.from_numpy(lens).to(DEV)
    idx, val = saib.indexer_decode_topk_values(d.q, d.w, d.cache, d.block_table, lens_d, nn, k,
                                               dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _, lg, ta, tb, _ = oracle.decode_topk(synth.bf16_bits(d.q), d.w.cpu().numpy(),
                                          d.cache.cpu().numpy(), d.block_table.cpu().numpy(),
                                          lens, nn, k, want_logits=True)
    _check_values_rows(idx.cpu().numpy(), val.cpu().numpy(), lens, lg, ta, tb, k)


def test_topk_values_small_k_and_every_row_split():
    # k = 64 over rows of a few hundred keys: rows longer and shorter than k,
    # each spread over several CTAs
    k = 64
    seq = [40, 64, 65, 700, 1000, 3, 256, 129, 0, 5000]
    d, lens = _inputs(seq, [1] * len(seq), 1, seed=61)
    idx, val = saib.indexer_decode_topk_values(d.q, d.w, d.cache, d.block_table,
                                               torch.from_numpy(lens).to(DEV), 1, k)
    torch.cuda.synchronize()
    _, lg, ta, tb, _ = oracle.decode_topk(synth.bf16_bits(d.q), d.w.cpu().numpy(),
                                          d.cache.cpu().numpy(), d.block_table.cpu().numpy(),
                                          lens, 1, k, want_logits=True)
    _check_values_rows(idx.cpu().numpy(), val.cpu().numpy(), lens, lg, ta, tb, k)


def test_topk_values_leave_the_plain_topk_unchanged():
    # the values mode is a separate launch configuration: a plain top-k call
    # right after it still gives the causal rows and the same long-row sets
    k = 2048
    seq = [100, 9000, 2048, 30000]
    d, lens = _inputs(seq, [1] * 4, 1, seed=62)
    lens_d = torch.from_numpy(lens).to(DEV)
    ws = saib.decode_workspace(4, 1, k, DEV)
    iv, _ = saib.indexer_decode_topk_values(d.q, d.w, d.cache, d.block_table, lens_d, 1, k,
                                            workspace=ws)
    it = saib.indexer_decode_topk(d.q, d.w, d.cache, d.block_table, lens_d, 1, k, workspace=ws)
    torch.cuda.synchronize()
    iv, it = iv.cpu().numpy(), it.cpu().numpy()
    assert np.array_equal(it[0], np.concatenate([np.arange(100), -np.ones(1948, np.int32)]))
    assert np.array_equal(it[2], np.arange(2048))
    for r in (1, 3):   # the same scores; only equal logits at the k-th may be swapped
        assert len(set(iv[r]) ^ set(it[r])) <= 4


# ---------------------------------------------------------------------------
# merge
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("world,k", [(2, 2048), (4, 64), (8, 2048), (3, 100)])
def test_dcp_merge_matches_oracle(world, k):
    rng = np.random.default_rng(70 + world)
    rows = 12
    # distinct values on rows 0..7; heavy ties on rows 8..9; rows 10..11 with
    # fewer candidates than k
    vals = rng.permutation(world * rows * k).astype(np.float32).reshape(world, rows, k) - 1000.0
    vals[:, 8:10] = np.round(rng.standard_normal((world, 2, k)), 0)
    idx = rng.permutation(world * rows * k).astype(np.int32).reshape(world, rows, k)
    drop = rng.random((world, rows, k)) < 0.1
    drop[:, 10:12] = rng.random((world, 2, k)) < (1.0 - 0.6 / world)
    idx[drop] = -1
    vals[drop] = -np.inf
    out, ov = saib.indexer_dcp_merge(torch.from_numpy(vals).to(DEV), torch.from_numpy(idx).to(DEV),
                                     k, out_val=torch.empty((rows, k), device=DEV))
    torch.cuda.synchronize()
    out, ov = out.cpu().numpy(), ov.cpu().numpy()
    ref, rv = oracle.merge_candidates(vals, idx, k)
    for r in range(rows):
        valid = out[r] >= 0
        nref = int((ref[r] >= 0).sum())
        assert valid.sum() == nref and np.all(np.isneginf(ov[r][~valid]))
        assert len(np.unique(out[r][valid])) == nref
        # each output value is that candidate's own value
        lookup = dict(zip(idx[:, r].ravel().tolist(), vals[:, r].ravel().tolist()))
        assert all(lookup[i] == v for i, v in zip(out[r][valid], ov[r][valid]))
        # the multiset of values is the oracle's (ties may pick other indices)
        assert np.array_equal(np.sort(ov[r][valid]), np.sort(rv[r][:nref]))
        if r < 8 or r >= 10:
            assert set(out[r][valid]) == set(ref[r][:nref])


# ---------------------------------------------------------------------------
# the sharded decode: every rank, then the merge
# ---------------------------------------------------------------------------

def _sharded(d, lens, nn, k, world, inter):
    shards = synth.shard_decode(d, world, inter, seed=7)
    rows = lens.shape[0]
    lens_d = torch.from_numpy(lens).to(DEV)
    cv = torch.empty((world, rows, k), dtype=torch.float32, device=DEV)
    ci = torch.empty((world, rows, k), dtype=torch.int32, device=DEV)
    err = _err()
    for r, (cache, bt) in enumerate(shards):
        saib.indexer_decode_topk_values(d.q, d.w, cache, bt, lens_d, nn, k, dcp_rank=r,
                                        dcp_world=world, dcp_interleave=inter, out_idx=ci[r],
                                        out_val=cv[r], dev_error=err)
    out, ov = saib.indexer_dcp_merge(cv, ci, k, out_val=torch.empty((rows, k), device=DEV))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return shards, ci.cpu().numpy(), cv.cpu().numpy(), out.cpu().numpy(), ov.cpu().numpy()


@pytest.mark.parametrize("world,inter,nn", [(2, 1, 1), (2, 64, 2), (4, 64, 1), (3, 5, 1)])
def test_dcp_decode_matches_unsharded_oracle(world, inter, nn):
    k = 2048
    rng = np.random.default_rng(80 + world * 10 + inter)
    R = 10
    seq = rng.integers(2, 24000, R).astype(np.int32)
    seq[0], seq[1], seq[2] = 1500, 2 * k + 1, 6000      # rows whose rank counts sit near k
    dl = rng.integers(1, nn + 1, R).astype(np.int32) if nn == 2 else np.ones(R, np.int32)
    d, lens = _inputs(seq, dl, nn, seed=90 + world)
    shards, ci, cv, out, ov = _sharded(d, lens, nn, k, world, inter)
    qb, w = synth.bf16_bits(d.q), d.w.cpu().numpy()
    # every rank's candidates against the oracle's rank step (local logits)
    for r, (cache, bt) in enumerate(shards):
        ref, _, local, lg, ta, tb = oracle.dcp_rank_topk_values(
            qb, w, cache.cpu().numpy(), bt.cpu().numpy(), lens, nn, k, r, world, inter)
        for row in range(lens.shape[0]):
            g2l = {int(g): j for j, g in enumerate(
                oracle.dcp_global_index(np.arange(local[row]), r, world, inter))}
            sel = ci[r, row]
            loc = np.array([g2l[int(g)] if g >= 0 else -1 for g in sel], np.int64)
            _check_values_rows(loc[None], cv[r, row][None], local[row:row + 1],
                               [lg[row]], [ta[row]], [tb[row]], k)
    # the merged rows against the unsharded oracle
    _, lg, ta, tb, _ = oracle.decode_topk(qb, w, d.cache.cpu().numpy(),
                                          d.block_table.cpu().numpy(), lens, nn, k,
                                          want_logits=True)
    worst = _check_values_rows(out, ov, lens, lg, ta, tb, k)
    print(f"world {world} interleave {inter}: max open keys per row {worst}")


def test_dcp_decode_batch_workload_full():
    # the decode-batch workload (32 requests, 2048..32768 keys) over 2 ranks
    # dealt in runs of 64 tokens, every row checked
    k = 2048
    d = synth.make_decode("decode", device=DEV)
    lens = d.seq_lens.cpu().numpy().astype(np.int64)
    _, _, _, out, ov = _sharded(d, lens.astype(np.int32), 1, k, 2, 64)
    _, lg, ta, tb, _ = oracle.decode_topk(synth.bf16_bits(d.q), d.w.cpu().numpy(),
                                          d.cache.cpu().numpy(), d.block_table.cpu().numpy(),
                                          lens, 1, k, want_logits=True)
    worst = _check_values_rows(out, ov, lens, lg, ta, tb, k)
    print(f"decode batch over 2 ranks: max open keys per row {worst}")


# ---------------------------------------------------------------------------
# compressed caches (one entry per compress_ratio tokens), decode and prefill
# ---------------------------------------------------------------------------

def test_compressed_decode_values_matches_oracle():
    # token rows of L tokens see L // 4 entries of a compressed cache
    k, C = 2048, 4
    seq = np.array([9000, 40001, 4, 8195, 30000, 16384], np.int32)
    dl = np.array([2, 1, 2, 2, 1, 2], np.int32)
    rl, _, _ = oracle.expand_rows(seq, dl, 2)
    ent = (seq // C).astype(np.int32)
    d = synth.make_decode_from_lens(ent, dl, 2, seed=71, device=DEV)
    idx, val = saib.indexer_decode_topk_values(d.q, d.w, d.cache, d.block_table,
                                               torch.from_numpy(rl).to(DEV), 2, k,
                                               compress_ratio=C)
    torch.cuda.synchronize()
    n_ent = rl // C
    _, lg, ta, tb, _ = oracle.decode_topk(synth.bf16_bits(d.q), d.w.cpu().numpy(),
                                          d.cache.cpu().numpy(), d.block_table.cpu().numpy(),
                                          n_ent, 2, k, want_logits=True)
    _check_values_rows(idx.cpu().numpy(), val.cpu().numpy(), n_ent, lg, ta, tb, k)


def _prefill_inputs(seq, ql, ratio, seed):
    ent = (np.asarray(seq) // ratio).astype(np.int32)
    cache_src = synth.make_decode_from_lens(ent, np.ones(len(seq), np.int32), 1, seed=seed,
                                            device=DEV)
    pre = synth.make_prefill(seq_lens=seq, query_lens=ql, seed=seed + 1, device=DEV)
    qsl = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    return cache_src, pre, qsl


@pytest.mark.parametrize("world,inter,ratio", [(1, 1, 1), (1, 1, 4), (2, 64, 4), (2, 1, 1)])
def test_prefill_values_sharded_and_compressed_match_oracle(world, inter, ratio):
    k = 2048
    seq = np.array([9000, 3000, 20000], np.int32)
    ql = np.array([300, 3000, 40], np.int32)
    src, pre, qsl = _prefill_inputs(seq, ql, ratio, seed=81 + ratio)
    shards = synth.shard_decode(src, world, inter, seed=8)
    rows = int(qsl[-1])
    cv = torch.empty((world, rows, k), dtype=torch.float32, device=DEV)
    ci = torch.empty((world, rows, k), dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for r, (cache, bt) in enumerate(shards):
        saib.indexer_prefill_topk_values(pre.q, pre.w, cache, bt, pre.seq_lens,
                                         pre.query_start_loc, seq, ql, k, compress_ratio=ratio,
                                         dcp_rank=r, dcp_world=world, dcp_interleave=inter,
                                         out_idx=ci[r], out_val=cv[r], dev_error=err)
    out, ov = saib.indexer_dcp_merge(cv, ci, k, out_val=torch.empty((rows, k), device=DEV))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # the merged rows against the unsharded compressed oracle, on a sample of
    # query rows (every request's first, last and a spread between)
    req, ln = oracle.prefill_rows(seq, qsl)
    n_ent = ln // ratio
    sample = np.unique(np.concatenate([qsl[:-1], qsl[1:] - 1,
                                       np.linspace(0, rows - 1, 60).astype(np.int64)]))
    q8, _, wp = oracle.quantize_q(synth.bf16_bits(pre.q), pre.w.cpu().numpy())
    cache_h, bt_h = src.cache.cpu().numpy(), src.block_table.cpu().numpy()
    out, ov = out.cpu().numpy(), ov.cpu().numpy()
    lg, ta, tb = [], [], []
    for i in sample:
        a, b_, c = oracle.row_logits(q8[i], wp[i], cache_h, bt_h[req[i]], int(n_ent[i]))
        lg.append(a)
        ta.append(b_)
        tb.append(c)
    worst = _check_values_rows(out[sample], ov[sample], n_ent[sample], lg, ta, tb, k)
    print(f"prefill world {world} ratio {ratio}: max open keys per row {worst}")


def test_dcp_long_context_sampled():
    # the long-context workload (1% heavy-tail keys) over 2 ranks dealt in
    # runs of 1 token, as the bench times it; 8 rows against the unsharded
    # oracle
    k = 2048
    d = synth.make_decode("long", device=DEV)
    lens = d.seq_lens.cpu().numpy().astype(np.int32)
    _, _, _, out, ov = _sharded(d, lens, 1, k, 2, 1)
    rows = np.array([0, 21, 42, 63, 64, 85, 106, 127])
    _, lg, ta, tb, _ = oracle.decode_topk(synth.bf16_bits(d.q), d.w.cpu().numpy(),
                                          d.cache.cpu().numpy(), d.block_table.cpu().numpy(),
                                          lens.astype(np.int64), 1, k, rows=rows,
                                          want_logits=True)
    worst = _check_values_rows(out[rows], ov[rows], lens[rows], lg, ta, tb, k)
    print(f"long context over 2 ranks: max open keys per row {worst}")
