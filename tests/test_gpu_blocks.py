"""Block and pool selection on the GPU vs the CPU oracle.

On seeded random logits (distinct values) the selected blocks must equal the
oracle's exactly; with ties, the counts, the forced blocks and the multiset
of selected block scores must; pool expansion is integer work and must match
bit for bit. End to end, blocks chosen from the GPU's own decode logits are
checked against the oracle's logits with the tolerance band.
"""
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


LENS = [0, 1, 63, 64, 65, 1000, 5000, 40000, 131072]


@pytest.mark.parametrize("B,k,ni,nl", [(64, 4, 1, 2), (64, 32, 0, 0), (16, 64, 1, 4),
                                       (64, 2048, 0, 0), (9, 5, 3, 3)])
def test_block_topk_matches_oracle(B, k, ni, nl):
    g = torch.Generator(device=DEV).manual_seed(B * 1000 + k)
    ld = 131072
    lg = torch.randn((len(LENS), ld), generator=g, device=DEV)
    lens = torch.tensor(LENS, dtype=torch.int32, device=DEV)
    cap = k + ni + nl
    out, cnt = saib.indexer_block_topk(lg, lens, B, k, ni, nl)
    torch.cuda.synchronize()
    out, cnt, lg_h = out.cpu().numpy(), cnt.cpu().numpy(), lg.cpu().numpy().astype(np.float64)
    for r, L in enumerate(LENS):
        ref, n = oracle.block_topk(lg_h[r], L, B, k, ni, nl, cap)
        assert cnt[r] == n and np.array_equal(out[r], ref), (r, L)


def test_block_topk_with_ties():
    g = torch.Generator(device=DEV).manual_seed(5)
    ld, B, k, ni, nl = 20000, 64, 16, 1, 2
    lg = torch.round(torch.randn((6, ld), generator=g, device=DEV) * 2) / 2   # few distinct
    lens_h = [20000, 19999, 4096, 640, 65, 2000]
    out, cnt = saib.indexer_block_topk(lg, torch.tensor(lens_h, dtype=torch.int32, device=DEV),
                                       B, k, ni, nl)
    torch.cuda.synchronize()
    out, cnt, lg_h = out.cpu().numpy(), cnt.cpu().numpy(), lg.cpu().numpy().astype(np.float64)
    for r, L in enumerate(lens_h):
        ref, n = oracle.block_topk(lg_h[r], L, B, k, ni, nl)
        got = out[r][:cnt[r]]
        assert cnt[r] == n and np.all(out[r][cnt[r]:] == -1)
        assert np.all(np.diff(got) > 0)                          # ascending, no duplicates
        nb = -(-L // B)
        forced = set(range(min(ni, nb))) | set(range(max(0, nb - nl), nb))
        assert forced <= set(got.tolist())
        score = lambda b: lg_h[r][b * B:min(L, b * B + B)].max()
        assert sorted(score(b) for b in got if b not in forced) == \
            sorted(score(b) for b in ref[:n] if b not in forced)


def test_expand_pools_matches_oracle():
    rng = np.random.default_rng(9)
    rows, pcap, P = 40, 24, 64
    lens = rng.integers(0, 5000, rows).astype(np.int32)
    lens[:3] = [0, 64, 130]
    pools = rng.integers(-2, 90, (rows, pcap)).astype(np.int32)
    counts = rng.integers(0, pcap + 1, rows).astype(np.int32)
    cap = pcap * P + P
    for pc in (None, counts):
        out, cnt = saib.indexer_expand_pools(
            torch.from_numpy(pools).to(DEV), torch.from_numpy(lens).to(DEV), P, cap,
            pool_counts=None if pc is None else torch.from_numpy(pc).to(DEV))
        torch.cuda.synchronize()
        out, cnt = out.cpu().numpy(), cnt.cpu().numpy()
        for r in range(rows):
            n_in = pcap if pc is None else int(pc[r])
            ref, n = oracle.expand_pools(pools[r, :n_in], int(lens[r]), P, cap)
            assert cnt[r] == n and np.array_equal(out[r], ref), r


def test_blocks_from_decode_logits_end_to_end():
    # decode logits (one pass over the keys) then block selection, against
    # the oracle's logits: every block whose largest logit beats the
    # (k+1)-th competitor even at worst is chosen, none that loses to k
    d = synth.make_decode_from_lens([40000, 9000, 2600, 700], [1, 1, 1, 1], 1, seed=33)
    dd = synth.DecodeInputs(q=d.q.to(DEV), w=d.w.to(DEV), cache=d.cache.to(DEV),
                            block_table=d.block_table.to(DEV), seq_lens=d.seq_lens.to(DEV),
                            decode_lens=d.decode_lens.to(DEV), next_n=1, topk=2048)
    B, k, ni, nl = 64, 16, 1, 2
    lg = saib.indexer_decode_logits(dd.q, dd.w, dd.cache, dd.block_table, dd.seq_lens, 1)
    out, cnt = saib.indexer_block_topk(lg, dd.seq_lens, B, k, ni, nl)
    torch.cuda.synchronize()
    out, cnt = out.cpu().numpy(), cnt.cpu().numpy()
    _, olg, ta, tb, _ = oracle.decode_topk(synth.bf16_bits(d.q), d.w.numpy(), d.cache.numpy(),
                                           d.block_table.numpy(), d.seq_lens.numpy(), 1, 2048,
                                           want_logits=True)
    for r, L in enumerate(d.seq_lens.numpy().tolist()):
        nb = -(-L // B)
        forced = set(range(min(ni, nb))) | set(range(max(0, nb - nl), nb))
        got = set(out[r][:cnt[r]].tolist())
        assert cnt[r] == len(forced) + min(k, nb - len(forced)) and forced <= got
        tol = tolerance(ta[r], tb[r])
        hi = np.array([(olg[r][b * B:b * B + B] + tol[b * B:b * B + B]).max() for b in range(nb)])
        lo = np.array([(olg[r][b * B:b * B + B] - tol[b * B:b * B + B]).max() for b in range(nb)])
        rest = [b for b in range(nb) if b not in forced]
        if len(rest) <= k:
            assert set(rest) <= got
            continue
        hs, ls = np.sort(hi[rest])[::-1], np.sort(lo[rest])[::-1]
        for b in rest:
            if lo[b] > hs[k]:
                assert b in got, f"row {r}: block {b} certainly in the top {k} is missing"
            if hi[b] < ls[k - 1]:
                assert b not in got, f"row {r}: block {b} certainly outside was chosen"
