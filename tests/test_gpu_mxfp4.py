"""MXFP4 index keys on the GPU vs the CPU oracle (row_logits_mxfp4, the
block-scaled dot of the e2m1 values and their ue8m0 scales in fp64).

Logits are compared element by element within the tolerance of
tests/_util.py; selected sets with the tolerance band around the k-th value;
rows of <= k keys must be the exact causal row.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_attention_indexer_block_gb300 as saib
from _util import check_logits, check_topk_row, relative_error_where_uncancelled

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_attention_indexer_block_gb300 import build as libbuild
    libbuild.build()
    saib.load()
    torch.cuda.set_device(DEV)


def _inputs(seq, seed, **kw):
    seq = np.asarray(seq, np.int32)
    return synth.make_decode_mxfp4_from_lens(seq, np.ones(len(seq), np.int32), 1, seed=seed,
                                             device=DEV, **kw)


def _oracle(d, lens, rows):
    q8, _, wp = oracle.quantize_q(synth.bf16_bits(d.q), d.w.cpu().numpy())
    cache, bt = d.cache.cpu().numpy(), d.block_table.cpu().numpy()
    return [oracle.row_logits_mxfp4(q8[r], wp[r], cache, bt[r], int(lens[r])) for r in rows]


@pytest.mark.parametrize("exps", [(124, 127), (113, 127)])
def test_mxfp4_logits_match_oracle(exps):
    # (113, 127): blocks up to 14 binades below the key's largest, so the
    # re-encoding also takes its e4m3-subnormal table (still exact there)
    seq = [1, 64, 130, 1000, 2048, 3000, 4096, 9000]
    d = _inputs(seq, 101 + exps[0], scale_exponents=exps)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lens = torch.tensor(seq, dtype=torch.int32, device=DEV)
    lg = saib.indexer_decode_logits_mxfp4(d.q, d.w, d.cache, d.block_table, lens, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    lg = lg.cpu().numpy()
    worst = rel = 0.0
    for r, (o, a, b) in enumerate(_oracle(d, seq, range(len(seq)))):
        worst = max(worst, check_logits(lg[r, :seq[r]], o, a, b))
        rel = max(rel, relative_error_where_uncancelled(lg[r, :seq[r]], o, a)[0])
    print(f"max |gpu - oracle| / (A + 0.01 B): {worst:.3g}; / |logit| where |logit| >= A/2: "
          f"{rel:.3g}")
    assert rel <= 1e-3


def test_mxfp4_topk_matches_oracle():
    # empty, single, k - 1 .. k + 1, and long rows split over many CTAs
    k = 2048
    seq = [0, 1, 2047, 2048, 2049, 5000, 40000, 65536, 300]
    d = _inputs(seq, 111)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = saib.indexer_decode_topk_mxfp4(d.q, d.w, d.cache, d.block_table,
                                         torch.tensor(seq, dtype=torch.int32, device=DEV), k,
                                         dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    out = out.cpu().numpy()
    for r, (o, a, b) in enumerate(_oracle(d, seq, range(len(seq)))):
        check_topk_row(out[r], o, a, b, k, seq[r])


def test_mxfp4_decode_batch_shape_every_row():
    # the decode batch's shape (32 requests, 2048 .. 32768 keys) with MXFP4 keys
    k = 2048
    seq = synth.draw_seq_lens(synth.WORKLOADS["decode"], synth.MASTER_SEED)
    d = _inputs(seq, 121)
    out = saib.indexer_decode_topk_mxfp4(d.q, d.w, d.cache, d.block_table, d.seq_lens, k)
    torch.cuda.synchronize()
    out = out.cpu().numpy()
    worst = 0
    for r, (o, a, b) in enumerate(_oracle(d, seq, range(len(seq)))):
        worst = max(worst, check_topk_row(out[r], o, a, b, k, int(seq[r])))
    print(f"max open keys per row {worst}")
    assert worst <= 4 + (3 * k) // 20


def test_mxfp4_long_context_sampled():
    # the long-context shape the bench times (128 requests x 131072 keys, the
    # launch splitting every row over several CTAs), 8 rows checked
    k = 2048
    seq = synth.draw_seq_lens(synth.WORKLOADS["long"], synth.MASTER_SEED)
    d = _inputs(seq, 131)
    out = saib.indexer_decode_topk_mxfp4(d.q, d.w, d.cache, d.block_table, d.seq_lens, k)
    torch.cuda.synchronize()
    out = out.cpu().numpy()
    rows = [0, 17, 38, 63, 64, 90, 111, 127]
    for r, (o, a, b) in zip(rows, _oracle(d, seq, rows)):
        check_topk_row(out[r], o, a, b, k, int(seq[r]))
