"""Seeded synthetic inputs for the sparse-attention indexer.

This module only draws inputs; it holds none of the indexer's arithmetic (no q
quantisation, no scoring, no selection, no row expansion). Both the CUDA
library's tests/benchmark and the CPU oracle consume what it produces.

Workloads (the shapes and distributions of the decode/prefill indexer the pages
describe; the pages measure on no public dataset):

* ``tiny``     4 requests, next_n 1, seq_lens {1000, 2048, 3000, 4096}
* ``decode``   32 requests, next_n 1, seq_lens uniform in [2048, 32768]
* ``mtp``      64 requests, next_n 2, decode_lens uniform in {1, 2},
               seq_lens uniform in [4096, 65536]
* ``long``     128 requests, next_n 1, seq_len 131072, 1% of each request's
               keys shifted by +4 along a query-aligned unit direction
* ``prefill``  4 requests x 8192 queries causally over 8192 keys

Common to all: 64 index heads x head_dim 128; q bf16 ~ N(0, 1); head weights
fp32 ~ N(0, 1) / 8; keys x ~ N(0, 1)^128 stored as fp8 e4m3 codes of
x / scale with the per-token fp32 scale = amax / 448 (the cast is torch's
float8_e4m3fn conversion); 64-token pages laid out as [64 x 128 fp8][64 x fp32]
(8448 bytes); the page pool is sized to the total tokens and every request's
block-table row lists its pages in logical order drawn from a seeded random
permutation of the pool. The heavy-tail direction of request b is the unit
vector along sum_h w[b, h] * q[b, h] (the direction that raises its pre-ReLU
head scores); 1% of the request's token positions (a seeded choice) get +4 times
that vector added before the cast.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

NUM_HEADS = 64
HEAD_DIM = 128
PAGE_TOKENS = 64
PAGE_BYTES = PAGE_TOKENS * (HEAD_DIM + 4)
MX_TOKEN_BYTES = HEAD_DIM // 2 + HEAD_DIM // 32   # packed e2m1 values + ue8m0 block scales
MX_PAGE_BYTES = PAGE_TOKENS * MX_TOKEN_BYTES
SCALE_OFFSET = PAGE_TOKENS * HEAD_DIM
TOPK = 2048
MASTER_SEED = 0x5EED


@dataclasses.dataclass
class Workload:
    name: str
    kind: str                      # "decode" | "prefill"
    num_reqs: int
    next_n: int = 1
    seq_lens: tuple | None = None  # fixed lengths
    seq_range: tuple | None = None  # inclusive uniform range
    decode_len_choices: tuple = (1,)
    heavy_tail_frac: float = 0.0
    query_len: int = 0             # prefill: queries per request (== seq_len here)
    topk: int = TOPK


WORKLOADS = {
    "tiny": Workload("tiny", "decode", 4, 1, seq_lens=(1000, 2048, 3000, 4096)),
    "decode": Workload("decode", "decode", 32, 1, seq_range=(2048, 32768)),
    "mtp": Workload("mtp", "decode", 64, 2, seq_range=(4096, 65536), decode_len_choices=(1, 2)),
    "long": Workload("long", "decode", 128, 1, seq_lens=(131072,) * 128, heavy_tail_frac=0.01),
    "prefill": Workload("prefill", "prefill", 4, 1, seq_lens=(8192,) * 4, query_len=8192),
}


@dataclasses.dataclass
class DecodeInputs:
    q: torch.Tensor            # bf16 [R*next_n, 64, 128]
    w: torch.Tensor            # fp32 [R*next_n, 64]
    cache: torch.Tensor        # uint8 [num_pages, 8448]
    block_table: torch.Tensor  # int32 [R, W]
    seq_lens: torch.Tensor     # int32 [R]
    decode_lens: torch.Tensor  # int32 [R]
    next_n: int
    topk: int

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])


@dataclasses.dataclass
class PrefillInputs:
    q: torch.Tensor                # bf16 [sum q, 64, 128]
    w: torch.Tensor                # fp32 [sum q, 64]
    cache: torch.Tensor            # uint8 [num_pages, 8448]
    block_table: torch.Tensor      # int32 [R, W]
    seq_lens: torch.Tensor         # int32 [R]
    query_lens: torch.Tensor       # int32 [R]
    query_start_loc: torch.Tensor  # int32 [R+1]
    topk: int


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def draw_seq_lens(wl: Workload, seed: int) -> np.ndarray:
    if wl.seq_lens is not None:
        return np.asarray(wl.seq_lens, dtype=np.int32)
    rng = np.random.default_rng(seed)
    lo, hi = wl.seq_range
    return rng.integers(lo, hi + 1, size=wl.num_reqs, dtype=np.int64).astype(np.int32)


def draw_decode_lens(wl: Workload, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed + 1)
    ch = np.asarray(wl.decode_len_choices, dtype=np.int32)
    return ch[rng.integers(0, len(ch), size=wl.num_reqs)]


def page_table(seq_lens: np.ndarray, seed: int, min_width: int = 1):
    """Seeded random permutation of a pool sized to the total tokens. Returns
    (block_table int32 [R, W], num_pages, page_owner int64 [P], page_index int64 [P])
    where page p holds tokens [64*page_index[p], 64*page_index[p]+64) of request
    page_owner[p]. Unused block-table entries are 0."""
    npg = (seq_lens.astype(np.int64) + PAGE_TOKENS - 1) // PAGE_TOKENS
    P = int(npg.sum())
    W = max(int(npg.max()) if len(npg) else 0, min_width)
    rng = np.random.default_rng(seed + 2)
    perm = rng.permutation(P).astype(np.int64)
    bt = np.zeros((len(seq_lens), W), np.int32)
    owner = np.zeros(P, np.int64)
    index = np.zeros(P, np.int64)
    off = 0
    for b, n in enumerate(npg):
        ids = perm[off:off + n]
        bt[b, :n] = ids
        owner[ids] = b
        index[ids] = np.arange(n)
        off += n
    return bt, max(P, 1), owner, index


def fill_cache(cache: torch.Tensor, gen: torch.Generator, page_bias=None, chunk_pages: int = 4096):
    """Writes random keys into every page of ``cache`` (uint8 [P, 8448]).

    page_bias(p0, p1) -> fp32 [p1-p0, 64, 128] additive shift or None."""
    P = cache.shape[0]
    dev = cache.device
    for p0 in range(0, P, chunk_pages):
        p1 = min(P, p0 + chunk_pages)
        x = torch.randn((p1 - p0, PAGE_TOKENS, HEAD_DIM), generator=gen, device=dev,
                        dtype=torch.float32)
        if page_bias is not None:
            b = page_bias(p0, p1)
            if b is not None:
                x += b
        amax = x.abs().amax(dim=-1, keepdim=True)
        scale = amax / 448.0
        k8 = (x / scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
        cache[p0:p1, :SCALE_OFFSET].copy_(k8.view(torch.uint8).reshape(p1 - p0, -1))
        cache[p0:p1, SCALE_OFFSET:].copy_(
            scale.reshape(p1 - p0, PAGE_TOKENS).contiguous().view(torch.uint8))


def make_decode(name_or_wl, seed: int = MASTER_SEED, device="cpu") -> DecodeInputs:
    wl = WORKLOADS[name_or_wl] if isinstance(name_or_wl, str) else name_or_wl
    device = torch.device(device)
    seq_lens = draw_seq_lens(wl, seed)
    decode_lens = (draw_decode_lens(wl, seed) if wl.next_n > 1
                   else np.ones(wl.num_reqs, np.int32))
    return make_decode_from_lens(seq_lens, decode_lens, wl.next_n, seed, device,
                                 wl.heavy_tail_frac, wl.topk)


def make_decode_from_lens(seq_lens, decode_lens, next_n: int, seed: int = MASTER_SEED,
                          device="cpu", heavy_tail_frac: float = 0.0,
                          topk: int = TOPK, bt_min_width: int = 1) -> DecodeInputs:
    device = torch.device(device)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    decode_lens = np.asarray(decode_lens, dtype=np.int32)
    R = len(seq_lens)
    rows = R * next_n
    g = _gen(device, seed * 7919 + 17)
    q = torch.randn((rows, NUM_HEADS, HEAD_DIM), generator=g, device=device).to(torch.bfloat16)
    w = torch.randn((rows, NUM_HEADS), generator=g, device=device) / 8.0
    bt, P, owner, index = page_table(seq_lens, seed, bt_min_width)
    cache = torch.empty((P, PAGE_BYTES), dtype=torch.uint8, device=device)
    bias = None
    if heavy_tail_frac > 0:
        # direction per request from its first token row
        d = (w[::next_n, :, None] * q[::next_n].float()).sum(dim=1)
        u = d / d.norm(dim=-1, keepdim=True)                       # [R, 128]
        rng = np.random.default_rng(seed + 3)
        # biased[p, slot]: token slot of page p gets the shift
        biased = np.zeros((P, PAGE_TOKENS), bool)
        for b in range(R):
            L = int(seq_lens[b])
            nb = int(round(heavy_tail_frac * L))
            pos = rng.choice(L, size=nb, replace=False)
            pg = bt[b, pos // PAGE_TOKENS]
            biased[pg, pos % PAGE_TOKENS] = True
        biased_t = torch.from_numpy(biased).to(device)
        owner_t = torch.from_numpy(owner).to(device)

        def bias(p0, p1):
            m = biased_t[p0:p1].float()[..., None]                 # [n, 64, 1]
            return 4.0 * m * u[owner_t[p0:p1]][:, None, :]

    fill_cache(cache, g, bias)
    return DecodeInputs(q=q, w=w, cache=cache,
                        block_table=torch.from_numpy(bt).to(device),
                        seq_lens=torch.from_numpy(seq_lens).to(device),
                        decode_lens=torch.from_numpy(decode_lens).to(device),
                        next_n=next_n, topk=topk)


def make_decode_mxfp4_from_lens(seq_lens, decode_lens, next_n: int, seed: int = MASTER_SEED,
                                device="cpu", topk: int = TOPK,
                                scale_exponents=(124, 127)) -> DecodeInputs:
    """Decode inputs whose cache holds MXFP4 index keys: pages of 64 entries
    of 68 bytes (64 bytes of packed e2m1 codes, element 2i in the low nibble of
    byte i, then 4 ue8m0 block scales), uint8 [P, 4352]. Every value byte is
    uniform (each e2m1 code equally likely) and every block scale exponent is
    uniform in the inclusive range `scale_exponents`. q, weights and the page
    table are drawn as for the fp8 cache."""
    device = torch.device(device)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    decode_lens = np.asarray(decode_lens, dtype=np.int32)
    rows = len(seq_lens) * next_n
    g = _gen(device, seed * 7919 + 23)
    q = torch.randn((rows, NUM_HEADS, HEAD_DIM), generator=g, device=device).to(torch.bfloat16)
    w = torch.randn((rows, NUM_HEADS), generator=g, device=device) / 8.0
    bt, P, _, _ = page_table(seq_lens, seed)
    cache = torch.empty((P, PAGE_TOKENS, MX_TOKEN_BYTES), dtype=torch.uint8, device=device)
    lo, hi = scale_exponents
    for p0 in range(0, P, 8192):
        p1 = min(P, p0 + 8192)
        cache[p0:p1, :, :HEAD_DIM // 2] = torch.randint(
            0, 256, (p1 - p0, PAGE_TOKENS, HEAD_DIM // 2), generator=g, device=device,
            dtype=torch.int32).to(torch.uint8)
        cache[p0:p1, :, HEAD_DIM // 2:] = torch.randint(
            lo, hi + 1, (p1 - p0, PAGE_TOKENS, HEAD_DIM // 32), generator=g, device=device,
            dtype=torch.int32).to(torch.uint8)
    return DecodeInputs(q=q, w=w, cache=cache.view(P, MX_PAGE_BYTES),
                        block_table=torch.from_numpy(bt).to(device),
                        seq_lens=torch.from_numpy(seq_lens).to(device),
                        decode_lens=torch.from_numpy(decode_lens).to(device),
                        next_n=next_n, topk=topk)


def shard_decode(inp: DecodeInputs, world: int, interleave: int, seed: int = MASTER_SEED):
    """Key-sharded copies of a decode cache: a list over ranks of (cache uint8
    [P_r, 8448], block_table int32 [R, W_r]) on the inputs' device.

    Token t of request b is dealt to rank (t // interleave) % world; a rank
    stores the tokens it is dealt in their order as its local tokens 0, 1, ...
    (the same fp8 codes and scale bytes), on pages of its own seeded random
    permutation. Data placement only: the bytes of each token are copied."""
    dev = inp.cache.device
    lens = inp.seq_lens.cpu().numpy().astype(np.int64)
    bt = inp.block_table.long()
    P0 = inp.cache.shape[0]
    src_v = inp.cache.view(P0, PAGE_BYTES)[:, :SCALE_OFFSET].view(P0, PAGE_TOKENS, HEAD_DIM)
    src_s = inp.cache.view(P0, PAGE_BYTES)[:, SCALE_OFFSET:].view(P0, PAGE_TOKENS, 4)
    shards = []
    for r in range(world):
        toks = [np.nonzero((np.arange(L) // interleave) % world == r)[0] for L in lens]
        local_lens = np.array([len(t) for t in toks], np.int64)
        lbt, P, _, _ = page_table(local_lens.astype(np.int32), seed + 101 * (r + 1))
        out = torch.zeros((P, PAGE_BYTES), dtype=torch.uint8, device=dev)
        dst_v = out[:, :SCALE_OFFSET].view(P, PAGE_TOKENS, HEAD_DIM)
        dst_s = out[:, SCALE_OFFSET:].view(P, PAGE_TOKENS, 4)
        lbt_t = torch.from_numpy(lbt).to(dev).long()
        if local_lens.sum() > 0:
            b = torch.from_numpy(np.repeat(np.arange(len(lens)), local_lens)).to(dev)
            t = torch.from_numpy(np.concatenate(toks)).to(dev)
            j = torch.from_numpy(np.concatenate([np.arange(n) for n in local_lens])).to(dev)
            sp, ss = bt[b, t // PAGE_TOKENS], t % PAGE_TOKENS
            dp, ds = lbt_t[b, j // PAGE_TOKENS], j % PAGE_TOKENS
            dst_v[dp, ds] = src_v[sp, ss]
            dst_s[dp, ds] = src_s[sp, ss]
        shards.append((out, lbt_t.int()))
    return shards


def make_prefill(name_or_wl="prefill", seed: int = MASTER_SEED, device="cpu",
                 seq_lens=None, query_lens=None) -> PrefillInputs:
    wl = WORKLOADS[name_or_wl] if isinstance(name_or_wl, str) else name_or_wl
    device = torch.device(device)
    if seq_lens is None:
        seq_lens = draw_seq_lens(wl, seed)
        query_lens = np.full(wl.num_reqs, wl.query_len, np.int32)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    query_lens = np.asarray(query_lens, dtype=np.int32)
    qsl = np.zeros(len(seq_lens) + 1, np.int32)
    qsl[1:] = np.cumsum(query_lens)
    total_q = int(qsl[-1])
    g = _gen(device, seed * 7919 + 29)
    q = torch.randn((total_q, NUM_HEADS, HEAD_DIM), generator=g, device=device).to(torch.bfloat16)
    w = torch.randn((total_q, NUM_HEADS), generator=g, device=device) / 8.0
    bt, P, _, _ = page_table(seq_lens, seed)
    cache = torch.empty((P, PAGE_BYTES), dtype=torch.uint8, device=device)
    fill_cache(cache, g)
    return PrefillInputs(q=q, w=w, cache=cache, block_table=torch.from_numpy(bt).to(device),
                         seq_lens=torch.from_numpy(seq_lens).to(device),
                         query_lens=torch.from_numpy(query_lens).to(device),
                         query_start_loc=torch.from_numpy(qsl).to(device), topk=wl.topk)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bits of a tensor as numpy uint16 (for the oracle)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
