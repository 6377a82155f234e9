"""The synthetic input recipe (CPU only): the five workloads (tiny, decode
batch, MTP, long context, prefill) have the shapes and distributions stated in
synth's docstring, the draws are seeded, and the paged layout is
[64 x 128 fp8][64 x fp32 scale] per page, so parity and benchmark runs measure
the configurations they claim."""
import numpy as np
import torch

import oracle
import synth


def test_workload_table_matches_the_stated_configurations():
    W = synth.WORKLOADS
    assert W["tiny"].seq_lens == (1000, 2048, 3000, 4096) and W["tiny"].next_n == 1
    assert (W["decode"].num_reqs, W["decode"].next_n, W["decode"].seq_range) == \
        (32, 1, (2048, 32768))
    assert (W["mtp"].num_reqs, W["mtp"].next_n, W["mtp"].seq_range,
            W["mtp"].decode_len_choices) == (64, 2, (4096, 65536), (1, 2))
    assert W["long"].seq_lens == (131072,) * 128 and W["long"].heavy_tail_frac == 0.01
    assert W["prefill"].seq_lens == (8192,) * 4 and W["prefill"].query_len == 8192
    assert all(w.topk == 2048 for w in W.values())


def test_seeded_draws_are_in_range_and_reproducible():
    for name in ("decode", "mtp"):
        wl = synth.WORKLOADS[name]
        a = synth.draw_seq_lens(wl, 7)
        assert np.array_equal(a, synth.draw_seq_lens(wl, 7))
        assert a.min() >= wl.seq_range[0] and a.max() <= wl.seq_range[1]
        assert not np.array_equal(a, synth.draw_seq_lens(wl, 8))
    dl = synth.draw_decode_lens(synth.WORKLOADS["mtp"], 7)
    assert set(np.unique(dl)) <= {1, 2} and len(np.unique(dl)) == 2


def test_page_table_is_a_permutation_covering_every_request():
    lens = np.array([1, 64, 65, 1000, 4096], np.int32)
    bt, P, owner, index = synth.page_table(lens, 3)
    need = (lens.astype(np.int64) + 63) // 64
    assert P == need.sum()
    used = np.concatenate([bt[b, :need[b]] for b in range(len(lens))])
    assert np.array_equal(np.sort(used), np.arange(P))  # every page exactly once
    for b in range(len(lens)):
        for j in range(need[b]):
            assert owner[bt[b, j]] == b and index[bt[b, j]] == j


def test_cache_pages_hold_codes_then_per_token_scales():
    """Each token's 128 codes times its fp32 scale reproduce keys whose
    largest magnitude is exactly 448 codes' worth (scale = amax / 448)."""
    d = synth.make_decode_from_lens([130], [1], 1, seed=4)
    cache = d.cache.numpy()
    codes = cache[:, :8192].reshape(-1, 64, 128)
    scales = cache[:, 8192:].copy().view(np.float32).reshape(-1, 64)
    assert cache.shape[1] == 8448 and (scales > 0).all()
    deq = oracle.e4m3_decode(codes)
    assert np.allclose(np.abs(deq).max(axis=-1), 448.0)  # the amax key maps to +-448


def test_heavy_tail_shifts_the_stated_fraction_of_tokens():
    """With the heavy tail on, the keys' mean projection on the request's
    direction grows by about fraction x 4 (the shift) over the same keys
    without it."""
    lens = [20000]
    plain = synth.make_decode_from_lens(lens, [1], 1, seed=9)
    tail = synth.make_decode_from_lens(lens, [1], 1, seed=9, heavy_tail_frac=0.05)

    def mean_projection(d):
        q = d.q.float()[0]
        w = d.w[0]
        u = (w[:, None] * q).sum(0)
        u = u / u.norm()
        cache = d.cache.numpy()
        codes = oracle.e4m3_decode(cache[:, :8192].reshape(-1, 64, 128))
        scales = cache[:, 8192:].copy().view(np.float32).reshape(-1, 64, 1)
        keys = torch.from_numpy((codes * scales).reshape(-1, 128))
        return float((keys.float() @ u).mean())

    gain = mean_projection(tail) - mean_projection(plain)
    assert abs(gain - 0.05 * 4.0) < 0.05


def test_shard_decode_places_each_token_once():
    seq = np.array([130, 5], np.int32)
    inp = synth.make_decode_from_lens(seq, np.ones(2, np.int32), 1, seed=3)
    shards = synth.shard_decode(inp, 2, 64, seed=9)
    c, bt = inp.cache.numpy(), inp.block_table.numpy()
    def entry(cache, btab, b, t):
        pg, sl = btab[b, t // 64], t % 64
        return (bytes(cache[pg, sl * 128:(sl + 1) * 128]),
                bytes(cache[pg, 8192 + 4 * sl:8192 + 4 * sl + 4]))
    for b, L in enumerate(seq):
        for t in range(L):
            r = (t // 64) % 2
            j = (t // 128) * 64 + t % 64
            sc, sbt = shards[r]
            assert entry(c, bt, b, t) == entry(sc.numpy(), sbt.numpy(), b, j)


def test_mxfp4_cache_draws_are_seeded_and_laid_out_as_stated():
    seq = np.array([130, 64, 1], np.int32)
    a = synth.make_decode_mxfp4_from_lens(seq, np.ones(3, np.int32), 1, seed=4)
    b = synth.make_decode_mxfp4_from_lens(seq, np.ones(3, np.int32), 1, seed=4)
    c = synth.make_decode_mxfp4_from_lens(seq, np.ones(3, np.int32), 1, seed=5)
    assert torch.equal(a.cache, b.cache) and torch.equal(a.q, b.q)
    assert not torch.equal(a.cache, c.cache)
    P = a.cache.shape[0]
    assert a.cache.shape == (P, 64 * 68) and P == 3 + 1 + 1      # ceil(L / 64) pages each
    ent = a.cache.numpy().reshape(P, 64, 68)
    scales = ent[..., 64:]
    assert scales.min() >= 124 and scales.max() <= 127             # stated exponent range
    codes = np.concatenate([ent[..., :64] & 15, ent[..., :64] >> 4]).ravel()
    counts = np.bincount(codes, minlength=16)
    assert counts.min() > 0.8 * counts.mean()                      # every e2m1 code drawn
    # a key read through the oracle's MXFP4 decoding is finite and scaled by
    # its blocks' exponents
    vals = oracle.mxfp4_values(ent[0, :2])
    assert np.all(np.isfinite(vals)) and np.abs(vals).max() <= 6 * 2.0 ** 0
