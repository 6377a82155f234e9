"""Pins of the CPU oracle against things other than itself (CPU only).

Each test ties one oracle function to the pages' worked examples, a library
routine, a closed form, brute force or an invariant, chosen so that a dropped
term, a wrong sign or index or a transposed operand fails.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


# --------------------------------------------------------------------------
# e4m3fn codec
# --------------------------------------------------------------------------

def test_e4m3_decode_matches_golden_codes():
    for line in _golden_lines("e4m3_codes.txt"):
        code, val = line.split()
        got = float(oracle.e4m3_decode([int(code, 16)])[0])
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def _torch_e4m3(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def test_e4m3_encode_roundtrip_midpoints_and_neighbours():
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = oracle.e4m3_decode(finite).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), finite)      # round trip, incl. -0
    pos = np.sort(oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)          # exact in fp32
    probes = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                             np.nextafter(mids, np.float32(1000)), -mids])
    assert np.array_equal(oracle.e4m3_encode(probes), _torch_e4m3(probes))
    # ties go to the even code
    enc = oracle.e4m3_encode(mids)
    assert np.all((enc & 1) == 0)


def test_e4m3_encode_random_and_saturation():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-448, 448, 4000),
                        rng.standard_normal(4000) * 1e-2,
                        rng.standard_normal(2000) * 1e-3]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), _torch_e4m3(x))
    sat = oracle.e4m3_encode(np.array([448.0, 464.0, 1e6, np.inf, -np.inf, -500.0], np.float32))
    assert list(sat) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


# --------------------------------------------------------------------------
# q quantisation
# --------------------------------------------------------------------------

def _bf16(vals):
    return torch.tensor(vals, dtype=torch.bfloat16)


def test_quantize_q_hand_example():
    head = [0.0] * 128
    head[0], head[1], head[2] = 2.0, -1.0, 0.5
    q = _bf16([[head, [0.0] * 128]])                              # 1 row, 2 heads
    w = np.array([[0.25, -3.0]], np.float32)
    q8, sq, wp = oracle.quantize_q(synth.bf16_bits(q), w)
    # amax 2 -> inv 224 -> 448, -224, 112 -> codes 0x7E, 0xF6, 0x6E
    assert list(q8[0, 0, :3]) == [0x7E, 0xF6, 0x6E]
    assert np.all(q8[0, 0, 3:] == 0)
    assert sq[0, 0] == 2.0 / 448.0 and wp[0, 0] == 0.25 * 2.0 / 448.0
    # an all-zero head quantises to zero codes and a zero weight
    assert np.all(q8[0, 1] == 0) and sq[0, 1] == 0.0 and wp[0, 1] == 0.0


def test_quantize_q_matches_library_cast_and_bounds():
    g = torch.Generator().manual_seed(3)
    q = torch.randn(5, 64, 128, generator=g).to(torch.bfloat16)
    q[1, 3] = 0.0
    w = (torch.randn(5, 64, generator=g) / 8).numpy()
    q8, sq, wp = oracle.quantize_q(synth.bf16_bits(q), w)
    qf = q.float().numpy()
    amax = np.abs(qf).max(axis=-1, keepdims=True)
    safe = np.where(amax > 0, amax, np.float32(1.0)).astype(np.float32)
    inv = np.float32(448.0) / safe                               # IEEE fp32 division
    x = np.where(amax > 0, qf * inv, 0).astype(np.float32)       # fp32 product
    ref = _torch_e4m3(x)
    ref[1, 3] = 0
    assert np.array_equal(q8, ref)
    # the largest magnitude maps onto +-448 exactly
    mx = np.abs(oracle.e4m3_decode(q8.reshape(-1, 128)[:64])).max(axis=-1)
    assert np.all(mx == 448.0)
    # dequantised q is within half an e4m3 step (relative 2^-4) of q for normal codes
    codes = oracle.e4m3_decode(q8)
    deq = codes * sq[..., None]
    normal = (np.abs(codes) >= 2.0 ** -6) & (qf != 0)
    rel = np.abs(deq - qf)[normal] / np.abs(qf)[normal]
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)
    assert np.allclose(wp, w * sq, rtol=0, atol=0)


# --------------------------------------------------------------------------
# row expansion
# --------------------------------------------------------------------------

def _worked_example():
    d = {}
    for line in _golden_lines("flatten_worked_example.txt"):
        key, *vals = line.split()
        d[key] = [int(v) for v in vals]
    return d


# --------------------------------------------------------------------------
# index-key cache insert
# --------------------------------------------------------------------------

def _bf16_tokens(n, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((n, 128), generator=g) * scale).to(torch.bfloat16)
    return x, x.view(torch.int16).numpy().view(np.uint16)


def test_insert_keys_matches_torch_quantisation():
    """The insert equals torch's per-token quantisation (amax/448 scale,
    x/scale cast by torch's own float8_e4m3fn conversion) slot by slot."""
    n, pages = 300, 6
    x, bits = _bf16_tokens(n, 5, scale=3.0)
    rng = np.random.default_rng(5)
    slots = rng.permutation(pages * 64)[:n].astype(np.int64)
    got = oracle.insert_keys(bits, slots, np.zeros((pages, 8448), np.uint8))
    xf = x.float()
    amax = xf.abs().amax(dim=-1, keepdim=True)
    scale = amax / 448.0
    codes = (xf / scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    sbytes = scale.reshape(-1).numpy().astype(np.float32).view(np.uint8).reshape(n, 4)
    for i, sl in enumerate(slots):
        pg, t = divmod(int(sl), 64)
        assert np.array_equal(got[pg, t * 128:(t + 1) * 128], codes[i])
        assert np.array_equal(got[pg, 8192 + 4 * t:8192 + 4 * t + 4], sbytes[i])


def test_insert_keys_hand_example_zero_token_and_skips():
    """A hand-worked token (amax 448 -> scale 1: codes of 448, 1, -0.5, 0 are
    0x7E, 0x38, 0xB0, 0x00), an all-zero token (zero codes, scale 0), padding
    and out-of-range slots skipped, every other byte untouched."""
    x = torch.zeros((4, 128), dtype=torch.float32)
    x[0, :4] = torch.tensor([448.0, 1.0, -0.5, 0.0])
    x[2, 5] = -2.0
    x[3, 0] = 1.0
    bits = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    base = np.full((2, 8448), 0xA5, np.uint8)
    got = oracle.insert_keys(bits, np.array([70, 3, -1, 128], np.int64), base)
    row = got[1, 6 * 128:7 * 128]
    assert list(row[:4]) == [0x7E, 0x38, 0xB0, 0x00] and not row[4:].any()
    assert np.frombuffer(got[1, 8192 + 24:8192 + 28].tobytes(), np.float32)[0] == 1.0
    assert not got[0, 3 * 128:4 * 128].any()
    assert np.frombuffer(got[0, 8192 + 12:8192 + 16].tobytes(), np.float32)[0] == 0.0
    touched = np.zeros_like(base, bool)
    touched[1, 6 * 128:7 * 128] = touched[1, 8192 + 24:8192 + 28] = True
    touched[0, 3 * 128:4 * 128] = touched[0, 8192 + 12:8192 + 16] = True
    assert (got[~touched] == 0xA5).all()  # slot -1 (token 2) and slot 128 (token 3) skipped


def test_insert_keys_dequantisation_error_bound():
    """code * scale is within e4m3's rounding bound of x: half a step, i.e.
    2^-4 relative for normal codes, 2^-10 * scale below the normal range."""
    x, bits = _bf16_tokens(64, 6, scale=0.01)
    got = oracle.insert_keys(bits, np.arange(64, dtype=np.int64), np.zeros((1, 8448), np.uint8))
    codes = got[0, :8192].reshape(64, 128)
    scale = np.frombuffer(got[0, 8192:].tobytes(), np.float32).astype(np.float64)
    deq = oracle.e4m3_decode(codes) * scale[:, None]
    xf = x.double().numpy()
    bound = np.maximum(np.abs(xf) * 2.0 ** -4, 2.0 ** -10 * scale[:, None]) * (1 + 1e-6)
    assert (np.abs(deq - xf) <= bound).all()
    assert np.allclose(np.abs(xf).max(axis=1), 448.0 * scale, rtol=1e-6)


def test_expand_flatten_matches_pages_worked_example():
    ex = _worked_example()
    bt = np.arange(4 * 3, dtype=np.int32).reshape(4, 3) + 100
    n_out = 10
    lens, rbt, n = oracle.expand_rows(ex["seq_lens"], ex["decode_lens"], 4, mode=1,
                                      block_table=bt, num_out_rows=n_out)
    assert n == len(ex["flat_row_lens"])
    assert list(lens[:n]) == ex["flat_row_lens"]
    assert np.all(lens[n:] == 0)                                  # zero tail
    owners = np.repeat(np.arange(4), ex["decode_lens"])
    assert np.array_equal(rbt[:n], bt[owners])                    # request's row per token
    assert np.all(rbt[n:, 0] == 0)                                # padded rows: column 0 = 0


def test_expand_padded_grid_agrees_with_flatten_and_pads_zero():
    ex = _worked_example()
    lens, _, n = oracle.expand_rows(ex["seq_lens"], ex["decode_lens"], 4, mode=0)
    grid = lens.reshape(4, 4)
    dl = np.array(ex["decode_lens"])
    for b in range(4):
        assert np.all(grid[b, dl[b]:] == 0)                       # padded rows have seq_len 0
    real = [int(grid[b, j]) for b in range(4) for j in range(dl[b])]
    assert real == ex["flat_row_lens"]


def test_expand_uniform_matches_token_rows_docstring():
    # token j of a request with q query tokens sees seq_len - (q - 1 - j) keys
    # ("vllm.models.minimax_m3.amd.mono.runner", token_rows).
    seq = np.array([100, 50, 3000, 7], np.int32)
    q = 3
    lens, _, _ = oracle.expand_rows(seq, np.full(4, q, np.int32), q, mode=0)
    for b in range(4):
        for j in range(q):
            assert lens[b * q + j] == seq[b] - (q - 1 - j)


# --------------------------------------------------------------------------
# scoring
# --------------------------------------------------------------------------

def _one_page_cache(k_codes, scales):
    page = np.zeros((1, oracle.PAGE_BYTES), np.uint8)
    for t, codes in enumerate(k_codes):
        page[0, t * 128:t * 128 + 128] = codes
    page[0, 8192:8192 + 4 * len(scales)] = np.asarray(scales, np.float32).view(np.uint8)
    return page


def test_logits_hand_computed_single_key():
    k = np.zeros(128, np.uint8)
    k[0] = 0x38                                                    # key = e_0, value 1.0
    cache = _one_page_cache([k, k], [0.5, 0.0])
    q = np.zeros((1, 2, 128), np.float32)
    q[0, 0, 0] = 1.0                                               # head 0 aligned
    q[0, 1, 0] = -1.0                                              # head 1 anti-aligned
    w = np.array([[0.25, 7.0]], np.float32)
    q8, _, wp = oracle.quantize_q(synth.bf16_bits(torch.from_numpy(q).to(torch.bfloat16)), w)
    lg, ta, tb = oracle.row_logits(q8[0], wp[0], cache, np.array([0], np.int32), 2)
    # head 0: ReLU(0.5 * 1 * 1) * 0.25; head 1: ReLU(-0.5) = 0; key 1 has scale 0
    assert lg[0] == 0.125 and lg[1] == 0.0
    assert ta[0] == 0.125 and tb[0] == pytest.approx(0.5 * (0.25 + 7.0))


def _dense_reference(q8, wp, cache, bt_row, length):
    """Independent numpy restatement used only to pin the C loops."""
    s = np.arange(length)
    pages = bt_row[s // 64]
    slots = s % 64
    vals = cache[pages[:, None], slots[:, None] * 128 + np.arange(128)[None, :]]
    kd = oracle.e4m3_decode(vals)                                  # [len, 128]
    scale = cache[pages[:, None], 8192 + 4 * slots[:, None] + np.arange(4)[None, :]]
    scale = scale.copy().view(np.float32)[:, 0].astype(np.float64)
    qd = oracle.e4m3_decode(q8)                                    # [H, 128]
    dots = kd @ qd.T                                               # [len, H]
    return scale * (np.maximum(dots, 0) @ wp), dots


def test_logits_match_dense_numpy_and_are_exact_dots():
    d = synth.make_decode_from_lens([300, 130], [1, 1], 1, seed=11, bt_min_width=8)
    q8, _, wp = oracle.quantize_q(synth.bf16_bits(d.q), d.w.numpy())
    cache = d.cache.numpy()
    bt = d.block_table.numpy()
    for r, L in enumerate([300, 130]):
        lg, _, _ = oracle.row_logits(q8[r], wp[r], cache, bt[r], L)
        ref, dots = _dense_reference(q8[r], wp[r], cache, bt[r], L)
        assert np.allclose(lg, ref, rtol=1e-12, atol=1e-12)
        # the fp64 dot of e4m3 values is exact: every product is a multiple of 2^-18
        qi = (oracle.e4m3_decode(q8[r]) * 2 ** 9).astype(np.int64)
        s = np.arange(L)
        vals = cache[bt[r][s // 64][:, None], (s % 64)[:, None] * 128 + np.arange(128)]
        ki = (oracle.e4m3_decode(vals) * 2 ** 9).astype(np.int64)
        assert np.array_equal((ki @ qi.T).astype(np.float64) / 2 ** 18, dots)


def test_logits_invariant_under_page_permutation_and_linear_in_w():
    d = synth.make_decode_from_lens([700], [1], 1, seed=5)
    q8, _, wp = oracle.quantize_q(synth.bf16_bits(d.q), d.w.numpy())
    cache = d.cache.numpy()
    bt = d.block_table.numpy()[0]
    lg, _, _ = oracle.row_logits(q8[0], wp[0], cache, bt, 700)
    perm = np.random.default_rng(2).permutation(cache.shape[0])
    cache2 = np.empty_like(cache)
    cache2[perm] = cache                                           # page p moves to perm[p]
    lg2, _, _ = oracle.row_logits(q8[0], wp[0], cache2, perm[bt].astype(np.int32), 700)
    assert np.array_equal(lg, lg2)
    lg3, _, _ = oracle.row_logits(q8[0], 2.0 * wp[0], cache, bt, 700)
    assert np.array_equal(lg3, 2.0 * lg)
    # a key whose slot is past the row length never influences the earlier logits
    lg4, _, _ = oracle.row_logits(q8[0], wp[0], cache, bt, 650)
    assert np.array_equal(lg4, lg[:650])


# --------------------------------------------------------------------------
# selection
# --------------------------------------------------------------------------

@pytest.mark.parametrize("k", [1, 7, 64])
def test_topk_brute_force_small_rows(k):
    rng = np.random.default_rng(k)
    for length in [0, 1, k - 1, k, k + 1, 150, 300]:
        if length < 0:
            continue
        lg = rng.integers(-20, 20, size=length).astype(np.float64)  # many ties
        out = oracle.topk_row(lg, length, k)
        if length <= k:
            assert list(out) == list(range(length)) + [-1] * (k - length)
        else:
            brute = sorted(range(length), key=lambda i: (-lg[i], i))[:k]
            assert list(out) == brute


def test_causal_identity_for_short_rows():
    # rows with len <= k select every key: exactly [0, len) followed by -1
    # ("vllm.models.glm5next.common.sparse_indexer", _fill_short_decode_causal_indices)
    d = synth.make_decode("tiny")
    lens, _, _ = oracle.expand_rows(d.seq_lens.numpy(), d.decode_lens.numpy(), 1)
    out, _, _, _, _ = oracle.decode_topk(synth.bf16_bits(d.q), d.w.numpy(), d.cache.numpy(),
                                         d.block_table.numpy(), lens, 1, 2048, rows=[0, 1])
    assert list(out[0]) == list(range(1000)) + [-1] * 1048
    assert list(out[1]) == list(range(2048))


def test_decode_topk_rows_are_valid_sets():
    d = synth.make_decode_from_lens([2100, 2500], [1, 1], 1, seed=9)
    lens, _, _ = oracle.expand_rows(d.seq_lens.numpy(), d.decode_lens.numpy(), 1)
    out, lg, _, _, _ = oracle.decode_topk(synth.bf16_bits(d.q), d.w.numpy(), d.cache.numpy(),
                                          d.block_table.numpy(), lens, 1, 2048,
                                          want_logits=True)
    for r in range(2):
        sel = out[r]
        assert len(set(sel.tolist())) == 2048 and sel.min() >= 0 and sel.max() < lens[r]
        kth = np.sort(lg[r])[::-1][2047]
        assert np.all(lg[r][sel] >= kth)
        rest = np.setdiff1d(np.arange(lens[r]), sel)
        assert np.all(lg[r][rest] <= kth)


def _brute_topk(lg, k):
    return sorted(range(len(lg)), key=lambda i: (-lg[i], i))[:k]


def test_decode_topk_two_token_rows_read_their_requests_block_table():
    """next_n = 2: token row b*2 + j reads q row b*2 + j and block-table row b,
    with j < d_b seeing L_b - d_b + j + 1 keys and padded rows none
    ("recipes/.../indexer.py", _prepare_decode_tensors: each token of a request
    reads that request's block table; "vllm.models.glm5next.common.
    sparse_indexer", _decode_topk_seq_lens: padded rows 0). Pinned by the
    numpy restatement of the scores and brute-force sorts, on requests whose
    block tables hold different pages."""
    sl, dl, k = [2300, 2200, 2600], [2, 1, 2], 256
    d = synth.make_decode_from_lens(sl, dl, 2, seed=19)
    bt = d.block_table.numpy()
    assert len(set(bt[0][:36]) & set(bt[1][:35])) == 0            # distinct pages
    lens, _, _ = oracle.expand_rows(np.array(sl), np.array(dl), 2)
    hand = [2299, 2300, 2200, 0, 2599, 2600]
    assert list(lens) == hand
    out, lg, _, _, rows = oracle.decode_topk(synth.bf16_bits(d.q), d.w.numpy(), d.cache.numpy(),
                                             bt, lens, 2, k, want_logits=True)
    q8, _, wp = oracle.quantize_q(synth.bf16_bits(d.q), d.w.numpy())
    cache = d.cache.numpy()
    for r in rows:
        b, L = r // 2, hand[r]
        if L == 0:
            assert list(out[r]) == [-1] * k
            continue
        ref, _ = _dense_reference(q8[r], wp[r], cache, bt[b], L)
        assert np.allclose(lg[r], ref, rtol=1e-12, atol=1e-12)
        # the same q row scored against another request's pages differs
        other, _ = _dense_reference(q8[r], wp[r], cache, bt[(b + 1) % 3], min(L, 2200))
        assert not np.allclose(ref[:len(other)], other)
        assert sorted(out[r].tolist()) == sorted(_brute_topk(lg[r], k))


def test_prefill_topk_routes_queries_to_their_request():
    """Query row i of request r (rows query_start_loc[r] + i) reads request r's
    block table and sees keys [0, L_r - Q_r + 1 + i) ("recipes/.../indexer.py",
    _build_prefill_chunk_metadata_kernel). Pinned by the numpy restatement and
    brute-force sorts; the rows are routed here by walking query_start_loc."""
    sl, ql, k = [300, 517, 90], [3, 5, 2], 64
    p = synth.make_prefill(seed=23, seq_lens=sl, query_lens=ql)
    bt = p.block_table.numpy()
    out, lg, _, _, rows = oracle.prefill_topk(synth.bf16_bits(p.q), p.w.numpy(), p.cache.numpy(),
                                              bt, p.seq_lens.numpy(),
                                              p.query_start_loc.numpy(), k, want_logits=True)
    q8, _, wp = oracle.quantize_q(synth.bf16_bits(p.q), p.w.numpy())
    cache = p.cache.numpy()
    route = []
    for r, (L, Q) in enumerate(zip(sl, ql)):
        for i in range(Q):
            route.append((r, L - Q + 1 + i))
    assert list(rows) == list(range(sum(ql)))
    assert [ln for _, ln in route] == [298, 299, 300, 513, 514, 515, 516, 517, 89, 90]
    for row, (r, L) in enumerate(route):
        ref, _ = _dense_reference(q8[row], wp[row], cache, bt[r], L)
        assert np.allclose(lg[row], ref, rtol=1e-12, atol=1e-12)
        assert sorted(out[row].tolist()) == sorted(_brute_topk(lg[row], k))


# --------------------------------------------------------------------------
# prefill
# --------------------------------------------------------------------------

def _plans():
    for line in _golden_lines("prefill_chunk_plans.txt"):
        _, rest = line.split(" ", 1)
        name, sl, ql, ws, budget, plan = [x.strip() for x in rest.split("|")]
        yield (name, [int(x) for x in sl.split()], [int(x) for x in ql.split()], int(ws),
               int(budget), [tuple(int(v) for v in p.split(":")) for p in plan.split()])


@pytest.mark.parametrize("case", list(_plans()), ids=lambda c: c[0])
def test_prefill_plan_golden(case):
    _, sl, ql, ws, budget, plan = case
    assert oracle.plan_prefill_chunks(sl, ql, ws, budget) == plan


def test_prefill_plan_invariants_random():
    rng = np.random.default_rng(4)
    for _ in range(300):
        n = int(rng.integers(1, 12))
        sl = rng.integers(0, 5000, n)
        ql = np.minimum(rng.integers(0, 3000, n), np.maximum(sl, 0))
        ws = int(rng.integers(1, 20000))
        budget = int(rng.integers(4, 4 * 10 ** 7))
        elems = budget // 4
        plan = oracle.plan_prefill_chunks(sl, ql, ws, budget)
        # chunks cover every request with queries exactly once, in order
        seen_q = {}
        for (r0, r1, a, b) in plan:
            assert 0 <= r0 < r1 <= n and 0 <= a < b
            seen_q.setdefault((r0, r1), []).append((a, b))
        covered = []
        for (r0, r1), pieces in seen_q.items():
            M = int(ql[r0:r1].sum())
            N = int(sl[r0:r1].sum())
            assert pieces[0][0] == 0 and pieces[-1][1] == M
            for (a0, b0), (a1, b1) in zip(pieces, pieces[1:]):
                assert b0 == a1
            if r1 - r0 > 1:
                assert N <= ws and M * N <= elems
            max_q = max(1, elems // N) if N > 0 else M
            assert all(b - a <= max_q for a, b in pieces)
            covered.extend(range(r0, r1))
        with_q = [i for i in range(n)]
        assert sorted(set(covered)) == sorted(set(i for i in covered))
        for i in with_q:
            if any(r0 <= i < r1 for (r0, r1) in seen_q):
                continue
            # a request left out belongs to a chunk with no queries at all
            assert ql[i] == 0


def test_prefill_rows_causal_ranges():
    # query i of a request with seq_len L and query_len Q sees keys [0, L - Q + 1 + i)
    # (_build_prefill_chunk_metadata_kernel: cu_seqlen_ke - cu_seqlen_ks)
    req, ln = oracle.prefill_rows([8, 10, 5], [0, 8, 11, 11])
    assert list(req) == [0] * 8 + [1] * 3
    assert list(ln[:8]) == list(range(1, 9))                      # L == Q: query i sees 0..i
    assert list(ln[8:]) == [8, 9, 10]


def test_fraction_exactness_of_score_scale():
    # scale_s factors out of the head sum because it is >= 0: checked with exact
    # rationals on one key against the unfactored sum.
    k = np.zeros(128, np.uint8)
    k[:4] = [0x38, 0xB8, 0x40, 0x01]
    cache = _one_page_cache([k], [0.375])
    q = torch.zeros(1, 3, 128)
    q[0, 0, :4] = torch.tensor([1.0, 0.5, 0.25, 3.0])
    q[0, 1, :4] = torch.tensor([-1.0, 0.0, 0.5, 0.0])
    q[0, 2, :4] = torch.tensor([0.0, -2.0, 0.0, 1.0])
    w = np.array([[0.5, -0.25, 2.0]], np.float32)
    q8, _, wp = oracle.quantize_q(synth.bf16_bits(q.to(torch.bfloat16)), w)
    lg, _, _ = oracle.row_logits(q8[0], wp[0], cache, np.array([0], np.int32), 1)
    kd = [Fraction(float(v)) for v in oracle.e4m3_decode(k)]
    tot = Fraction(0)
    for h in range(3):
        qd = [Fraction(float(v)) for v in oracle.e4m3_decode(q8[0, h])]
        dot = sum(a * b for a, b in zip(qd, kd))
        tot += Fraction(float(wp[0, h])) * max(Fraction(0.375) * dot, Fraction(0))
    assert abs(Fraction(float(lg[0])) - tot) <= abs(tot) * Fraction(1, 10 ** 15)


# ---------------------------------------------------------------------------
# MXFP4 index keys (GLM5 page: _gather_workspace_shapes, kv_cache_as_quant_view;
# INDEXER page: the use_fp4_indexer_cache gate)
# ---------------------------------------------------------------------------

def _golden_e2m1():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_codes.txt"))
            if l.strip() and not l.startswith("#")]
    return {int(c): float(v) for c, v in rows}


def test_e2m1_decode_matches_golden_table():
    g = _golden_e2m1()
    got = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    for c in range(16):
        assert got[c] == g[c] and np.signbit(got[c]) == np.signbit(g[c]), c


def test_e2m1_encode_round_trips_and_rounds_to_nearest_even():
    g = _golden_e2m1()
    for c in range(16):
        want = c if c != 8 else 8  # -0 keeps its sign bit
        assert int(oracle.e2m1_encode(g[c])) == want, c
    # midpoints (worked by hand): ties go to the even mantissa
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6,
             -0.75: 10, -5.0: 14,
             0.26: 1, 0.74: 1, 1.26: 3, 4.9: 6, 5.1: 7,
             6.0: 7, 7.9: 7, 1e9: 7, -100.0: 15}
    for x, c in cases.items():
        assert int(oracle.e2m1_encode(x)) == c, (x, c)


def test_ue8m0_decode_matches_torch_for_every_code():
    tvals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64)
    got = oracle.ue8m0_decode(np.arange(256, dtype=np.uint8))
    t = tvals.numpy()
    assert np.isnan(got[255]) and np.isnan(t[255])
    assert np.array_equal(got[:255], t[:255])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127


def test_mxfp4_quantize_hand_worked_blocks():
    x = np.zeros((1, 128), np.float32)
    x[0, :6] = [6.0, -3.0, 1.5, 0.75, 0.2, 0.0]     # block 0: amax 6 -> E = 2 - 2 + 127
    x[0, 32] = 0.3                                   # block 1: amax 0.3 -> E = -2 - 2 + 127
    x[0, 33] = -0.1                                  #   0.1 / 2^-4 = 1.6 -> 1.5
    # block 2: all zero -> E = 0, zero codes
    x[0, 96] = 7.9                                   # block 3: amax 7.9 -> E = 127, saturates
    e = oracle.mxfp4_quantize(x)[0]
    assert e[0] == 0xD7 and e[1] == 0x23 and e[2] == 0x00   # (6, -3), (1.5, 1.0), (0, 0)
    assert e[16] == (0xB << 4 | 0x6)                       # (0.3 -> 4.0 * 2^-4, -0.1 -> -1.5 * 2^-4)
    assert list(e[64:68]) == [127, 123, 0, 127]
    assert e[48] == 0x07                                   # 7.9 -> 6 (saturated)
    v = oracle.mxfp4_values(e[None])[0]
    assert v[:6].tolist() == [6.0, -3.0, 1.5, 1.0, 0.0, 0.0]
    assert v[32] == 0.25 and v[33] == -0.09375 and v[96] == 6.0


def test_mxfp4_quantize_error_bound_and_scale_rule():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 128)) * np.exp2(rng.integers(-20, 20, (64, 1)))).astype(np.float32)
    e = oracle.mxfp4_quantize(x)
    v = oracle.mxfp4_values(e)
    for b in range(4):
        blk = x[:, 32 * b:32 * (b + 1)].astype(np.float64)
        amax = np.abs(blk).max(axis=1)
        E = np.floor(np.log2(amax)).astype(int) - 2 + 127
        assert np.array_equal(e[:, 64 + b].astype(int), E)
        X = np.exp2(E - 127.0)[:, None]
        # the block's largest value lands in [4X, 8X): at most 2X from the grid
        # (saturation at 6X), every other value within half a step (<= X)
        assert (np.abs(v[:, 32 * b:32 * (b + 1)] - blk) <= 2 * X).all()
        inside = np.abs(blk) <= 6 * X
        assert (np.abs(v[:, 32 * b:32 * (b + 1)] - blk)[inside] <= X.repeat(32, 1)[inside]).all()


def _mx_cache(rng, pages):
    keys = rng.standard_normal((pages * 64, 128)).astype(np.float32)
    return oracle.mxfp4_quantize(keys).reshape(pages, oracle.MX_PAGE_BYTES), keys


def test_mxfp4_row_logits_hand_computed_key():
    # one head; q8 = code 0x38 (1.0) on d = 0 and 40, 0xB8 (-1.0) on d = 100
    q8 = np.zeros((1, 128), np.uint8)
    q8[0, 0] = 0x38
    q8[0, 40] = 0x38
    q8[0, 100] = 0xB8
    entry = np.zeros(68, np.uint8)
    entry[0] = 0x07            # d = 0: 6.0
    entry[20] = 0x05           # d = 40: 3.0
    entry[50] = 0x0C           # d = 100: -2.0
    entry[64:68] = [126, 128, 127, 125]   # block scales 0.5, 2, 1, 0.25
    cache = np.zeros((2, oracle.MX_PAGE_BYTES), np.uint8)
    slot = 5
    cache[1, slot * 68:(slot + 1) * 68] = entry
    bt = np.array([1], np.int32)
    lg, ta, tb = oracle.row_logits_mxfp4(q8, np.array([0.5]), cache, bt, slot + 1)
    dot = 1.0 * 6.0 * 0.5 + 1.0 * 3.0 * 2.0 + (-1.0) * (-2.0) * 0.25   # 3 + 6 + 0.5
    assert lg[slot] == 0.5 * dot and ta[slot] == 0.5 * dot and tb[slot] == 0.5 * dot
    assert (lg[:slot] == 0.0).all()


def test_mxfp4_row_logits_match_dense_restatement_on_permuted_pages():
    rng = np.random.default_rng(11)
    pages = 6
    cache, _ = _mx_cache(rng, pages)
    q = rng.standard_normal((4, 128)).astype(np.float32)
    q8 = oracle.e4m3_encode(q * 16)
    wp = rng.standard_normal(4)
    bt = rng.permutation(pages).astype(np.int32)
    L = pages * 64 - 17
    lg, ta, tb = oracle.row_logits_mxfp4(q8, wp, cache, bt, L)
    # dense restatement: gather the pages by fancy indexing, decode, matmul
    ent = cache.reshape(pages, 64, 68)[bt].reshape(-1, 68)[:L]
    k = oracle.mxfp4_values(ent)
    dots = oracle.e4m3_decode(q8) @ k.T                   # [H, L]
    want = (wp[:, None] * np.maximum(dots, 0)).sum(0)
    assert np.allclose(lg, want, rtol=1e-12, atol=1e-12)
    # the dot of one head is exact: scaled by 2^(10 - (E_min - 127)) it is an integer
    e_min = int(ent[:, 64:68].min())
    scaled = dots * np.exp2(9 + 1 - (e_min - 127))
    assert np.array_equal(scaled, np.round(scaled))


def test_mxfp4_decode_topk_matches_brute_force():
    rng = np.random.default_rng(12)
    pages = 5
    cache, _ = _mx_cache(rng, pages)
    R, next_n, k = 2, 2, 40
    q = torch.randn(R * next_n, 64, 128, generator=torch.Generator().manual_seed(3))
    qbits = q.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    w = (rng.standard_normal((R * next_n, 64)) / 8).astype(np.float32)
    bt = np.stack([rng.permutation(pages), rng.permutation(pages)]).astype(np.int32)
    lens = np.array([300, 301, 30, 0], np.int32)
    out = oracle.decode_topk_mxfp4(qbits, w, cache, bt, lens, next_n, k)
    q8, _, wp = oracle.quantize_q(qbits, w)
    for r in range(R * next_n):
        L = int(lens[r])
        if L <= k:
            assert out[r].tolist() == list(range(L)) + [-1] * (k - L)
            continue
        lg, _, _ = oracle.row_logits_mxfp4(q8[r], wp[r], cache, bt[r // next_n], L)
        order = sorted(range(L), key=lambda i: (-lg[i], i))
        assert sorted(out[r].tolist()) == sorted(order[:k])


# --------------------------------------------------------------------------
# key-sharded (decode context parallel) decode
# --------------------------------------------------------------------------

def test_dcp_local_len_matches_counting_the_dealt_tokens():
    # INDEXER page, _build_prefill_chunk_metadata_kernel (DCP branch): token t
    # goes to rank (t // I) % W; the closed form must count exactly those.
    for world in (1, 2, 3, 4, 8):
        for inter in (1, 2, 3, 5, 64):
            lens = np.arange(0, 700, 7 if inter > 5 else 1)
            tot = np.zeros_like(lens)
            for r in range(world):
                got = oracle.dcp_local_lens(lens, r, world, inter)
                ref = np.array([int(((np.arange(L) // inter) % world == r).sum()) for L in lens])
                assert np.array_equal(got, ref), (world, inter, r)
                tot += got
            assert np.array_equal(tot, lens)


def test_dcp_local_len_hand_cases():
    # 130 keys, runs of 64 over 2 ranks: rank 0 holds 0..63 and 128..129
    assert oracle.dcp_local_lens([130], 0, 2, 64)[0] == 66
    assert oracle.dcp_local_lens([130], 1, 2, 64)[0] == 64
    # 10 keys, runs of 1 over 4 ranks: 3, 3, 2, 2
    assert [int(oracle.dcp_local_lens([10], r, 4, 1)[0]) for r in range(4)] == [3, 3, 2, 2]


def test_dcp_global_index_inverts_the_dealing():
    for world, inter, L in ((2, 1, 37), (3, 5, 101), (4, 64, 1000), (1, 7, 20)):
        t = np.arange(L)
        owner = (t // inter) % world
        seen = []
        for r in range(world):
            n = int(oracle.dcp_local_lens([L], r, world, inter)[0])
            g = oracle.dcp_global_index(np.arange(n), r, world, inter)
            assert np.array_equal(g, t[owner == r])   # rank r's tokens, in order
            seen.append(g)
        assert np.array_equal(np.sort(np.concatenate(seen)), t)
    assert oracle.dcp_global_index([-1], 1, 2, 64)[0] == -1


def test_topk_row_values_keeps_short_rows_whole():
    rng = np.random.default_rng(11)
    lg = rng.standard_normal(50)
    o, v = oracle.topk_row_values(lg, 50, 64)
    assert np.array_equal(o[:50], np.arange(50)) and np.all(o[50:] == -1)
    assert np.array_equal(v[:50], lg) and np.all(np.isneginf(v[50:]))
    lg = rng.standard_normal(300)
    o, v = oracle.topk_row_values(lg, 300, 64)
    assert np.array_equal(o, np.argsort(-lg, kind="stable")[:64])
    assert np.array_equal(v, lg[o])


def test_merge_candidates_brute_force():
    rng = np.random.default_rng(12)
    for n_per, world, k in ((64, 2, 64), (30, 3, 64), (100, 4, 37)):
        vals = np.round(rng.standard_normal((world, 5, n_per)), 1)   # many ties
        idx = rng.permutation(world * 5 * n_per).reshape(world, 5, n_per).astype(np.int32)
        idx[rng.random(idx.shape) < 0.2] = -1
        vals[idx < 0] = -np.inf
        out, ov = oracle.merge_candidates(vals, idx, k)
        for r in range(5):
            cand = sorted((-vals[w, r, i], idx[w, r, i]) for w in range(world)
                          for i in range(n_per) if idx[w, r, i] >= 0)
            ref = [c[1] for c in cand[:k]] + [-1] * max(0, k - len(cand))
            assert list(out[r]) == ref
            assert np.array_equal(ov[r][:len(cand)], [-c[0] for c in cand[:k]])


@pytest.mark.parametrize("world,inter,next_n", [(1, 1, 1), (2, 1, 1), (3, 64, 2), (4, 5, 1)])
def test_dcp_decode_topk_equals_the_unsharded_topk(world, inter, next_n):
    # every key of a row's top k is in its own rank's top k, so the merge of
    # the ranks' candidates is the unsharded row's top k (same logits)
    k = 96
    seq = np.array([40, 96, 97, 400, 1000, 333], np.int32)
    dl = np.array([1, 2, 1, 2, 2, 1], np.int32) if next_n == 2 else np.ones(6, np.int32)
    inp = synth.make_decode_from_lens(seq, dl, next_n, seed=31 + world)
    qb = synth.bf16_bits(inp.q)
    w = inp.w.numpy()
    rl, _, _ = oracle.expand_rows(seq, dl, next_n)
    shards = [(c.numpy(), b.numpy()) for c, b in synth.shard_decode(inp, world, inter, seed=5)]
    got, gv = oracle.dcp_decode_topk(qb, w, shards, rl, next_n, k, inter)
    ref, lg, _, _, _ = oracle.decode_topk(qb, w, inp.cache.numpy(), inp.block_table.numpy(), rl,
                                          next_n, k, want_logits=True)
    for r in range(rl.shape[0]):
        L = int(rl[r])
        n = min(L, k)
        assert np.all(got[r, n:] == -1) and np.all(np.isneginf(gv[r, n:]))
        assert np.array_equal(gv[r, :n], lg[r][got[r, :n]])        # the unsharded logits
        order = np.lexsort((np.arange(L), -lg[r]))[:n]              # (logit desc, index asc)
        assert np.array_equal(got[r, :n], order)
        assert set(got[r, :n]) == set(ref[r][ref[r] >= 0])



def test_index_key_counts_compress_then_deal():
    # a compressed cache holds entry e for tokens [e * C, e * C + C) once they
    # are all present (L // C entries: the INDEXER page's seq_lens //
    # compress_ratio); the entries are then dealt to ranks like tokens
    for C in (1, 2, 4, 7):
        for world, inter in ((1, 1), (2, 1), (3, 64), (4, 5)):
            lens = np.arange(0, 900)
            for r in range(world):
                got = oracle.index_key_counts(lens, C, r, world, inter)
                ref = np.array([int(((np.arange(L // C) // inter) % world == r).sum())
                                for L in lens])
                assert np.array_equal(got, ref), (C, world, inter, r)
    assert oracle.index_key_counts([10], 4)[0] == 2 and oracle.index_key_counts([3], 4)[0] == 0


@pytest.mark.parametrize("world,inter,ratio", [(1, 1, 4), (2, 1, 1), (2, 64, 4), (3, 5, 2)])
def test_sharded_prefill_equals_the_unsharded_prefill(world, inter, ratio):
    # query i of request r sees (L - Q + 1 + i) // ratio entries; the merge of
    # the ranks' candidates is the unsharded top k over them
    k = 48
    seq = np.array([300, 90, 517], np.int32)
    ql = np.array([5, 90, 7], np.int32)
    ent = seq // ratio                           # entries of the compressed cache
    inp = synth.make_decode_from_lens(ent, np.ones(3, np.int32), 1, seed=44 + ratio)
    qsl = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    pre = synth.make_prefill(seq_lens=seq, query_lens=ql, seed=45)
    qb, w = synth.bf16_bits(pre.q), pre.w.numpy()
    shards = [(c.numpy(), b.numpy()) for c, b in synth.shard_decode(inp, world, inter, seed=6)]
    got, gv = oracle.dcp_prefill_topk(qb, w, shards, seq, qsl, k, inter, ratio)
    req, ln = oracle.prefill_rows(seq, qsl)
    n_ent = ln // ratio
    q8, _, wp = oracle.quantize_q(qb, w)
    for i in range(ln.shape[0]):
        L = int(n_ent[i])
        lg, _, _ = oracle.row_logits(q8[i], wp[i], inp.cache.numpy(),
                                     inp.block_table.numpy()[req[i]], L)
        n = min(L, k)
        order = np.lexsort((np.arange(L), -lg))[:n]
        assert np.array_equal(got[i, :n], order) and np.all(got[i, n:] == -1)
        assert np.array_equal(gv[i, :n], lg[order])


# --------------------------------------------------------------------------
# block / pool selection
# --------------------------------------------------------------------------

def _block_topk_brute(lg, L, B, k, n_init, n_local):
    nb = -(-L // B)
    forced = {b for b in range(nb) if b < n_init or b >= nb - n_local}
    rest = sorted((b for b in range(nb) if b not in forced),
                  key=lambda b: (-max(lg[b * B:min(L, b * B + B)]), b))
    return sorted(forced | set(rest[:k]))


def test_block_topk_brute_force_and_invariants():
    rng = np.random.default_rng(21)
    for L, B, k, ni, nl in [(1, 64, 4, 1, 2), (64, 64, 4, 1, 1), (65, 64, 1, 0, 0), (1000, 64, 5, 1, 2),
                            (1000, 16, 3, 2, 2), (5000, 64, 16, 1, 4), (300, 7, 100, 0, 0),
                            (4096, 64, 64, 0, 0)]:
        lg = np.round(rng.standard_normal(L), 1)           # ties inside and across blocks
        got, n = oracle.block_topk(lg, L, B, k, ni, nl)
        ref = _block_topk_brute(lg, L, B, k, ni, nl)
        assert list(got[:n]) == ref and np.all(got[n:] == -1)
        nb = -(-L // B)
        forced = set(range(min(ni, nb))) | set(range(max(0, nb - nl), nb))
        assert n == len(forced) + min(k, nb - len(forced))   # count
        assert forced <= set(ref)                             # init and local blocks kept


def test_block_topk_hand_case():
    # blocks of 4: [0 1 2 3] [9 0 0 0] [1 1 1 1] [0 0 5 0] [2]: scores 3, 9, 1, 5, 2
    lg = np.array([0, 1, 2, 3, 9, 0, 0, 0, 1, 1, 1, 1, 0, 0, 5, 0, 2], np.float64)
    got, n = oracle.block_topk(lg, 17, 4, 2, 0, 0)
    assert list(got[:n]) == [1, 3]
    got, n = oracle.block_topk(lg, 17, 4, 1, 1, 1)         # block 0 and block 4 forced, then 1
    assert list(got[:n]) == [0, 1, 4]


def test_expand_pools_and_tail():
    # pools of 4 over 10 tokens: complete pools 0, 1; tail 8, 9; pool 2 is the tail
    out, n = oracle.expand_pools(np.array([1, 0]), 10, 4, 16)
    assert list(out[:n]) == [4, 5, 6, 7, 0, 1, 2, 3, 8, 9] and np.all(out[n:] == -1)
    out, n = oracle.expand_pools(np.array([2, -1]), 10, 4, 16)
    assert list(out[:n]) == [8, 9]
    out, n = oracle.expand_pools(np.array([0]), 8, 4, 16)   # no tail
    assert list(out[:n]) == [0, 1, 2, 3]
