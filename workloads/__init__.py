"""Seeded synthetic inputs shared by the CUDA path's tests, the oracle's tests
and the benchmark.

This module holds no attention arithmetic: it only describes packs (the
``cu_seqlens`` offsets and the ordered segment list of each sequence) and
draws seeded bf16 tensors.  The pack shapes follow the serving workloads of
"[RFC]: HunyuanImage 3.0 deployment" (classifier-free-guidance pairs of equal
length, concurrent requests at different resolutions, high-resolution edits
with reference images) and the 4K = 16,384-token image of "MiniMax
H3-Image ... 4K in 0.87 s".

Readings where the workload text is silent:
* a request is a text prefix followed by its image segment(s);
* the two CFG branches of a request are two sequences of identical layout;
* the mixed-resolution draws use ``numpy.random.default_rng(seed)``: per
  request ``choice([1024, 2304, 4096, 9216])`` then ``integers(32, 513)``;
* tensors come from ``torch.Generator('cpu').manual_seed(seed)``: ``randn``
  for q [T,Hq,d], then k [T,Hkv,d], then v [T,Hkv,d], rounded fp32 -> bf16
  (round to nearest even); an optional exact power-of-two multiplier
  sharpens q.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Sequence, Tuple

import numpy as np

TEXT = 0
IMAGE = 1


@dataclasses.dataclass
class Pack:
    """A packed batch: per-sequence segment lists plus head geometry."""

    name: str
    seqs: List[List[Tuple[int, int]]]  # per sequence: [(type, length), ...]
    hq: int
    hkv: int
    d: int
    q_mult: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def cu_seqlens(self) -> np.ndarray:
        lens = [sum(n for _, n in s) for s in self.seqs]
        return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)

    @property
    def segments(self) -> np.ndarray:
        """[G, 3] int32: (global start, length, type), in pack order."""
        out = []
        pos = 0
        for s in self.seqs:
            for typ, n in s:
                out.append((pos, n, typ))
                pos += n
        return np.asarray(out, dtype=np.int32).reshape(-1, 3)

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_seqlen(self) -> int:
        cu = self.cu_seqlens
        return int(np.max(np.diff(cu))) if len(cu) > 1 else 0

    def describe(self) -> dict:
        return {"workload": self.name, "num_seqs": len(self.seqs),
                "total_tokens": self.total_tokens, "max_seqlen": self.max_seqlen,
                "hq": self.hq, "hkv": self.hkv, "head_dim": self.d}


def tiny_pack(seed: int = 0) -> Pack:
    """Two sequences: 16 text + 64 image; 24 text + 256 image + 8 text;
    Hq = Hkv = 4, d = 64."""
    return Pack("tiny-2seq-h4-d64",
                [[(TEXT, 16), (IMAGE, 64)], [(TEXT, 24), (IMAGE, 256), (TEXT, 8)]],
                hq=4, hkv=4, d=64, seed=seed)


def cfg_pair(seed: int = 0) -> Pack:
    """One request's CFG pair: 2 x (128 text + 4096 image + 4 text),
    Hq = 32, Hkv = 8, d = 128."""
    seq = [(TEXT, 128), (IMAGE, 4096), (TEXT, 4)]
    return Pack("cfg-pair-2x4228-gqa32-8-d128", [list(seq), list(seq)],
                hq=32, hkv=8, d=128, seed=seed)


def mixed_resolution(seed: int = 0, requests: int = 8) -> Pack:
    """``requests`` concurrent requests x 2 CFG branches; image tokens drawn
    from {1024, 2304, 4096, 9216}, text prefix uniform in [32, 512]."""
    rng = np.random.default_rng(seed)
    seqs = []
    for _ in range(requests):
        n_img = int(rng.choice([1024, 2304, 4096, 9216]))
        n_txt = int(rng.integers(32, 513))
        seq = [(TEXT, n_txt), (IMAGE, n_img)]
        seqs.append(list(seq))
        seqs.append(list(seq))
    return Pack(f"mixed-resolution-{requests}req-x2cfg-gqa32-8-d128", seqs,
                hq=32, hkv=8, d=128, seed=seed)


def highres_edit(seed: int = 0) -> Pack:
    """2 x (256 text + 4096 ref image + 4096 ref image + 16384 target image),
    three distinct image segments per sequence."""
    seq = [(TEXT, 256), (IMAGE, 4096), (IMAGE, 4096), (IMAGE, 16384)]
    return Pack("highres-edit-2x24832-gqa32-8-d128", [list(seq), list(seq)],
                hq=32, hkv=8, d=128, seed=seed)


def skewed(seed: int = 0) -> Pack:
    """1 x (512 text + 16384 image) plus 63 x (U[16,128] text + 256 image);
    q multiplied by 4 to sharpen the softmax."""
    rng = np.random.default_rng(seed)
    txt = rng.integers(16, 129, size=63)
    seqs = [[(TEXT, 512), (IMAGE, 16384)]]
    seqs += [[(TEXT, int(t)), (IMAGE, 256)] for t in txt]
    return Pack("skewed-1x16896+63x-gqa32-8-d128-q4", seqs, hq=32, hkv=8, d=128,
                q_mult=4.0, seed=seed)


CONFIGS = {
    "tiny": tiny_pack,
    "cfg_pair": cfg_pair,
    "mixed_resolution": mixed_resolution,
    "highres_edit": highres_edit,
    "skewed": skewed,
}


def random_pack(rng: np.random.Generator, num_seqs: int, max_len: int,
                hq: int = 4, hkv: int = 2, d: int = 64, allow_empty: bool = True,
                name: str = "random") -> Pack:
    """Random segment structure: alternating and adjacent text/image runs,
    optional empty sequences, lengths up to ``max_len`` per sequence."""
    seqs = []
    for _ in range(num_seqs):
        if allow_empty and rng.random() < 0.1:
            seqs.append([])
            continue
        L = int(rng.integers(1, max_len + 1))
        segs = []
        left = L
        while left > 0:
            n = int(rng.integers(1, max(2, min(left, max_len // 2 + 1)) + 1))
            n = min(n, left)
            segs.append((int(rng.integers(0, 2)), n))
            left -= n
        seqs.append(segs)
    return Pack(name, seqs, hq=hq, hkv=hkv, d=d, seed=int(rng.integers(0, 2**31)))


def make_qkv(pack: Pack, device: str = "cpu"):
    """Seeded bf16 tensors q [T,Hq,d], k [T,Hkv,d], v [T,Hkv,d] on CPU, then
    moved to ``device``."""
    import torch
    T = pack.total_tokens
    g = torch.Generator(device="cpu").manual_seed(pack.seed)
    q = torch.randn(T, pack.hq, pack.d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(T, pack.hkv, pack.d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(T, pack.hkv, pack.d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    if pack.q_mult != 1.0:
        q = q * pack.q_mult  # power of two: exact in bf16
    if device != "cpu":
        q, k, v = q.to(device), k.to(device), v.to(device)
    return q, k, v


def sample_rows(pack: Pack, budget: int, seed: int = 1, tile: int = 128) -> np.ndarray:
    """Deterministic row sample for full-size parity: the first and last row
    of every sequence and segment, rows on both sides of every 128-row tile
    edge of the longest sequences, plus uniform random rows, capped at
    ``budget`` (structural rows first)."""
    cu = pack.cu_seqlens
    segs = pack.segments
    T = int(cu[-1])
    picks: List[int] = []
    for s in range(len(cu) - 1):
        b, e = int(cu[s]), int(cu[s + 1])
        if e > b:
            picks += [b, e - 1]
    for st, n, _ in segs:
        picks += [int(st), int(st + n - 1), min(int(st + n), T - 1)]
    for s in range(len(cu) - 1):
        b, e = int(cu[s]), int(cu[s + 1])
        for t0 in range(b + tile, e, tile):
            picks += [t0 - 1, t0]
    rng = np.random.default_rng(seed)
    structural = list(dict.fromkeys(p for p in picks if 0 <= p < T))
    rng.shuffle(structural)
    structural = structural[: budget // 2]
    n_rand = max(0, budget - len(structural))
    rand = rng.integers(0, T, size=n_rand).tolist() if T > 0 else []
    rows = np.unique(np.asarray(structural + rand, dtype=np.int32))
    return rows[:budget]


def boundary_tile_rows(pack: Pack, budget: int, tile: int = 128) -> np.ndarray:
    """Every row of the 128-row query tiles where the mask changes shape: the
    tile holding each segment's first and last row and each sequence's last
    (ragged) tile, taken sequence by sequence (shortest first, so that every
    kind of sequence is represented) until ``budget`` rows."""
    cu = pack.cu_seqlens
    tiles = []
    for s in range(len(cu) - 1):
        b, e = int(cu[s]), int(cu[s + 1])
        if e == b:
            continue
        starts = {b + ((e - 1 - b) // tile) * tile}
        for st, n, _ in pack.segments:
            st, n = int(st), int(n)
            if b <= st < e:
                starts.add(b + ((st - b) // tile) * tile)
                starts.add(b + ((st + n - 1 - b) // tile) * tile)
        tiles.append((e - b, sorted((t0, min(t0 + tile, e)) for t0 in starts)))
    tiles.sort(key=lambda x: x[0])
    rows: List[int] = []
    for _, ts in tiles:
        for t0, t1 in ts:
            if len(rows) + (t1 - t0) > budget:
                return np.unique(np.asarray(rows, dtype=np.int32))
            rows.extend(range(t0, t1))
    return np.unique(np.asarray(rows, dtype=np.int32))


def seq_segments(pack: Pack) -> np.ndarray:
    """[G, 4] int32 (seq, start, len, type): segments in each sequence's own
    position space."""
    out = []
    for s, seq in enumerate(pack.seqs):
        pos = 0
        for typ, n in seq:
            out.append((s, pos, n, typ))
            pos += n
    return np.asarray(out, dtype=np.int32).reshape(-1, 4)


def prefix_split(pack: Pack):
    """Cached-prefix layout of a pack: per sequence the queries are the tokens
    from its first image segment on (the tokens being generated), the keys
    are the whole sequence (text prefix handed over + image).  Returns
    (q_rows: global token indices of the queries, cu_seqlens_q, q_pos0)."""
    cu = pack.cu_seqlens
    rows, cu_q, q_pos0 = [], [0], []
    for s, seq in enumerate(pack.seqs):
        first_img = 0
        for typ, n in seq:
            if typ == IMAGE:
                break
            first_img += n
        L = int(cu[s + 1] - cu[s])
        first_img = min(first_img, L)
        rows.extend(range(int(cu[s]) + first_img, int(cu[s + 1])))
        cu_q.append(cu_q[-1] + L - first_img)
        q_pos0.append(first_img)
    return np.asarray(rows, dtype=np.int64), np.asarray(cu_q, np.int32), np.asarray(q_pos0, np.int32)


def paged_layout(pack: Pack, rng: np.random.Generator, block: int = 128, spare: int = 3):
    """A shuffled block pool holding every sequence's keys: returns
    (block_table [S, blocks_per_seq] int32, pool_rows: for every pool row the
    global token it holds, or -1)."""
    cu = pack.cu_seqlens
    S = len(cu) - 1
    nblocks = [(int(cu[s + 1] - cu[s]) + block - 1) // block for s in range(S)]
    bps = max(nblocks) if nblocks else 0
    total = sum(nblocks) + spare
    perm = rng.permutation(total)
    table = np.zeros((S, max(bps, 1)), dtype=np.int32)
    pool_rows = -np.ones(total * block, dtype=np.int64)
    k = 0
    for s in range(S):
        for b in range(nblocks[s]):
            pb = int(perm[k]); k += 1
            table[s, b] = pb
            for r in range(block):
                t = int(cu[s]) + b * block + r
                if t < int(cu[s + 1]):
                    pool_rows[pb * block + r] = t
    return table, pool_rows


def key_chunks(pack: Pack, chunk: int):
    """Split every sequence's keys into chunks of ``chunk`` positions (ring
    attention's per-step key blocks).  Returns one (cu_seqlens_k, k_pos0,
    key_rows) per chunk index: key_rows are the global tokens the chunk's
    contiguous key tensor holds, sequence by sequence."""
    cu = pack.cu_seqlens
    S = len(cu) - 1
    L = np.diff(cu).astype(np.int64)
    C = int(-(-int(L.max()) // chunk)) if S and L.max() > 0 else 0
    out = []
    for c in range(C):
        k_pos0 = np.minimum(c * chunk, L).astype(np.int32)
        nk = np.clip(L - c * chunk, 0, chunk)
        cu_k = np.concatenate([[0], np.cumsum(nk)]).astype(np.int32)
        rows = np.concatenate([np.arange(cu[s] + k_pos0[s], cu[s] + k_pos0[s] + nk[s])
                               for s in range(S)]).astype(np.int64)
        out.append((cu_k, k_pos0, rows))
    return out


def quantize_e4m3(x):
    """Per-tensor FP8 E4M3 quantisation of a bf16/fp32 torch tensor: the scale
    maps the tensor's largest magnitude to 448 (E4M3's largest finite
    value); returns (codes uint8 tensor, scale float).  Input preparation for
    the FP8 path; torch's float8_e4m3fn conversion rounds to nearest even."""
    import torch
    amax = float(x.float().abs().max())
    scale = amax / 448.0 if amax > 0 else 1.0
    codes = (x.float() / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale
