"""Seeded synthetic decode workloads (inputs only, no attention arithmetic).

Every input is drawn from a CPU ``torch.Generator`` so that the CUDA path and
the CPU oracle see identical bytes.  bf16 tensors are produced as fp32
standard normals rounded to bf16 (round-to-nearest-even, torch's cast) and
are handed out as ``numpy.uint16`` bit patterns.

Block tables follow the paged-KV picture of the "mini-infer" pages (prajwal7-2002
docs, "Systems Architecture": a fixed physical block pool and a per-request
virtual-to-physical table): a seeded random permutation of the physical block
ids is handed out to the sequences in order, so logically adjacent blocks are
physically scattered.  Unused table entries are -1.

The step is "write then attend": sequence b's new token sits at position
L_b - 1 and is written through ``slot_mapping`` before attention reads it.
With ``q_len`` > 1 (speculative verification, or a chunk of new tokens) the
last q_len positions of each sequence are new: q is [B, q_len, Hq, D] and the
write covers all of them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

BF16_NAN = 0x7FC0  # quiet NaN bit pattern, used to poison never-read pool rows


@dataclasses.dataclass
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    max_blocks: int
    seq_lens: np.ndarray       # [B] int32, includes the token written this step
    block_tables: np.ndarray   # [B, max_blocks] int32, -1 padded
    q: np.ndarray              # [B, Hq, D] uint16 (bf16 bits); [B, q_len, Hq, D] if q_len > 1
    k_cache: np.ndarray        # [num_blocks, bs, Hkv, D] uint16, before this step's write
    v_cache: np.ndarray
    k_new: np.ndarray          # [N, Hkv, D] uint16
    v_new: np.ndarray
    slot_mapping: np.ndarray   # [N] int64
    scale: float
    q_len: int = 1             # new tokens (queries) per sequence
    # FP8 variant: e4m3 codes of the pools (uint8) and the per-pool scales
    k_cache8: Optional[np.ndarray] = None
    v_cache8: Optional[np.ndarray] = None
    k_scale: float = 1.0
    v_scale: float = 1.0
    cascade_blocks: int = 0    # > 0: decode with the first this-many table entries as a shared prefix

    @property
    def fp8(self) -> bool:
        return self.k_cache8 is not None

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def kv_bytes(self) -> int:
        """Bytes of K and V that attention must read (each token once per KV head)."""
        elem = 1 if self.fp8 else 2
        return int(self.seq_lens.astype(np.int64).sum()) * 2 * self.Hkv * self.D * elem

    def unique_kv_bytes(self) -> int:
        """Bytes of K and V in distinct pool rows that attention reads: a block
        shared by several sequences (a prefix-cache hit) counts once."""
        elem = 1 if self.fp8 else 2
        depth = {}   # rows of each physical block read by some sequence (its deepest reader)
        for b in range(self.B):
            L = int(self.seq_lens[b])
            for j in range((L + self.block_size - 1) // self.block_size):
                blk = int(self.block_tables[b, j])
                depth[blk] = max(depth.get(blk, 0), min(self.block_size, L - j * self.block_size))
        return sum(depth.values()) * 2 * self.Hkv * self.D * elem

    def qo_bytes(self) -> int:
        return 2 * self.B * self.q_len * self.Hq * self.D * 2

    def write_bytes(self) -> int:
        """Bytes moved by the cache write: read k_new/v_new (bf16), write them into the pools."""
        n = int((self.slot_mapping >= 0).sum())
        return 2 * n * self.Hkv * self.D * (2 + (1 if self.fp8 else 2))


def _bf16_bits(gen: torch.Generator, shape: Sequence[int]) -> np.ndarray:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def make_workload(name: str, *, B: int, Hq: int, Hkv: int, D: int, block_size: int,
                  seq_lens: Sequence[int], num_blocks: int, seed: int,
                  max_blocks: Optional[int] = None, shared_prefix_blocks: int = 0,
                  scale: Optional[float] = None, poison_unused: bool = False,
                  write_new: bool = True, q_len: int = 1) -> DecodeWorkload:
    """Build one seeded workload.

    ``shared_prefix_blocks`` > 0 makes the first that many table entries of
    every sequence the same physical blocks (prefix-cache reuse).
    ``poison_unused`` fills every pool row that attention must never read
    (rows past L_b in a sequence's last block, and blocks no table uses) with
    bf16 NaN, so that any over-read shows up in the output.
    """
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    gen = torch.Generator().manual_seed(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    assert seq_lens.shape == (B,)
    nbs = [(int(L) + block_size - 1) // block_size for L in seq_lens]
    if max_blocks is None:
        max_blocks = max(1, max(nbs))
    assert max(nbs) <= max_blocks
    perm = torch.randperm(num_blocks, generator=gen).numpy().astype(np.int32)
    tables = np.full((B, max_blocks), -1, dtype=np.int32)
    cursor = shared_prefix_blocks
    shared = perm[:shared_prefix_blocks]
    for b, nb in enumerate(nbs):
        ns = min(nb, shared_prefix_blocks)
        tables[b, :ns] = shared[:ns]
        rest = nb - ns
        if cursor + rest > num_blocks:
            raise ValueError(f"pool of {num_blocks} blocks too small")
        tables[b, ns:nb] = perm[cursor:cursor + rest]
        cursor += rest
    if q_len < 1:
        raise ValueError("q_len must be >= 1")
    q = _bf16_bits(gen, (B, Hq, D) if q_len == 1 else (B, q_len, Hq, D))
    k_cache = _bf16_bits(gen, (num_blocks, block_size, Hkv, D))
    v_cache = _bf16_bits(gen, (num_blocks, block_size, Hkv, D))
    if write_new:
        # token j of sequence b's new ones sits at position L_b - q_len + j
        k_new = _bf16_bits(gen, (B * q_len, Hkv, D))
        v_new = _bf16_bits(gen, (B * q_len, Hkv, D))
        slots = np.full((B * q_len,), -1, dtype=np.int64)
        for b in range(B):
            L = int(seq_lens[b])
            for j in range(q_len):
                t = L - q_len + j
                if t >= 0:
                    slots[b * q_len + j] = int(tables[b, t // block_size]) * block_size + t % block_size
        if len(set(slots[slots >= 0].tolist())) != int((slots >= 0).sum()):
            raise ValueError("new tokens collide on a slot (a shared block is being written)")
    else:
        k_new = np.zeros((0, Hkv, D), np.uint16)
        v_new = np.zeros((0, Hkv, D), np.uint16)
        slots = np.zeros((0,), np.int64)
    if poison_unused:
        live = np.zeros((num_blocks, block_size), dtype=bool)
        for b, L in enumerate(seq_lens):
            for t in range(int(L)):
                live[tables[b, t // block_size], t % block_size] = True
        k_cache[~live] = BF16_NAN
        v_cache[~live] = BF16_NAN
    return DecodeWorkload(name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=block_size,
                          num_blocks=num_blocks, max_blocks=max_blocks, seq_lens=seq_lens,
                          block_tables=tables, q=q, k_cache=k_cache, v_cache=v_cache,
                          k_new=k_new, v_new=v_new, slot_mapping=slots,
                          scale=float(np.float32(1.0 / math.sqrt(D))) if scale is None else scale,
                          q_len=q_len)


def _uniform_lens(seed: int, B: int, lo: int, hi: int) -> list[int]:
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


# The five workload families.  Seeds are 1000 + family id.
def tiny(**kw) -> DecodeWorkload:
    """B=4 sequences of lengths {1, 17, 33, 100}, Hq=4, Hkv=2, D=64, 16-token blocks, 64-block pool."""
    return make_workload("tiny", B=4, Hq=4, Hkv=2, D=64, block_size=16,
                         seq_lens=[1, 17, 33, 100], num_blocks=64, seed=1001, **kw)


def qwen25_1p5b(B: int = 8, **kw) -> DecodeWorkload:
    """Qwen2.5-1.5B-shaped layer: Hq=12, Hkv=2, D=128, bs=16, L ~ U[512, 2048], 4096-block pool."""
    assert B in (1, 8)
    return make_workload(f"qwen2.5-1.5b-B{B}", B=B, Hq=12, Hkv=2, D=128, block_size=16,
                         seq_lens=_uniform_lens(2002 + B, B, 512, 2048), num_blocks=4096,
                         max_blocks=128, seed=1002, **kw)


def qwen25_7b(block_size: int = 16, **kw) -> DecodeWorkload:
    """Qwen2.5-7B-shaped layer: B=8, Hq=28, Hkv=4, D=128, every L=4096; 16-token blocks or 256-token pages."""
    assert block_size in (16, 256)
    nb = 4096 if block_size == 16 else 256
    return make_workload(f"qwen2.5-7b-bs{block_size}", B=8, Hq=28, Hkv=4, D=128,
                         block_size=block_size, seq_lens=[4096] * 8, num_blocks=nb,
                         max_blocks=4096 // block_size, seed=1003, **kw)


def long_context(B: int = 1, L: int = 32768, **kw) -> DecodeWorkload:
    """Flash-decoding stress: B in {1,2}, Hq=28, Hkv=4, D=128, L in {4096, 32768}, bs=16."""
    assert B in (1, 2) and L in (4096, 32768)
    nb_seq = L // 16
    return make_workload(f"long-B{B}-L{L}", B=B, Hq=28, Hkv=4, D=128, block_size=16,
                         seq_lens=[L] * B, num_blocks=2 * B * nb_seq, max_blocks=nb_seq,
                         seed=1004, **kw)


def qwen3_0p6b(B: int = 256, **kw) -> DecodeWorkload:
    """Qwen3-0.6B-shaped high concurrency: B=256, Hq=16, Hkv=8, D=128, bs=16,
    L ~ U[129, 2048], first 8 table entries shared by all sequences, 20480-block pool."""
    return make_workload(f"qwen3-0.6b-B{B}", B=B, Hq=16, Hkv=8, D=128, block_size=16,
                         seq_lens=_uniform_lens(2005, B, 129, 2048), num_blocks=20480,
                         max_blocks=128, shared_prefix_blocks=8, seed=1005, **kw)


def qwen3_long_prefix(B: int = 256, prefix_blocks: int = 128, **kw) -> DecodeWorkload:
    """Qwen3-0.6B-shaped batch behind a long shared prefix (a system prompt held
    once in the prefix cache): B=256, Hq=16, Hkv=8, D=128, bs=16; the first
    prefix_blocks table entries (2048 tokens) are the same blocks for every
    sequence, then each sequence's own U[1, 256] tokens."""
    own = _uniform_lens(2006, B, 1, 256)
    lens = [prefix_blocks * 16 + n for n in own]
    return make_workload(f"qwen3-0.6b-B{B}-prefix{prefix_blocks * 16}", B=B, Hq=16, Hkv=8, D=128,
                         block_size=16, seq_lens=lens, num_blocks=prefix_blocks + B * 16,
                         max_blocks=prefix_blocks + 16, shared_prefix_blocks=prefix_blocks,
                         seed=1006, **kw)


def with_fp8_pools(w: DecodeWorkload) -> DecodeWorkload:
    """FP8 variant of a workload: the same bf16 pools rounded to e4m3 codes by
    torch's float8_e4m3fn cast, with one scale per pool chosen as amax / 448
    (so the codes span the format).  The new-token rows stay bf16."""
    def codes(bits: np.ndarray):
        x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float()
        amax = float(torch.nan_to_num(x, nan=0.0).abs().max())
        scale = float(np.float32(max(amax, 1e-30) / 448.0))
        c = (x / torch.tensor(scale, dtype=torch.float32)).clamp(-448, 448)
        return c.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy(), scale
    w.k_cache8, w.k_scale = codes(w.k_cache)
    w.v_cache8, w.v_scale = codes(w.v_cache)
    w.name = w.name + "-fp8"
    return w


def _cascade(w: DecodeWorkload, n: int) -> DecodeWorkload:
    w.cascade_blocks = n
    w.name = w.name + "-cascade"
    return w


def spec_verify(base: str, q_len: int, **kw) -> DecodeWorkload:
    """Speculative verification on a decode workload: the last q_len positions
    of every sequence are the target model's queries (q_len - 1 drafted tokens
    plus the bonus position), written this step and attended causally."""
    w = WORKLOADS[base](q_len=q_len, **kw)
    w.name = f"{base}-spec{q_len}"
    return w


def prefill_chunk(base: str, q_len: int, **kw) -> DecodeWorkload:
    """Chunked prefill on a decode workload: the last q_len positions of every
    sequence are one chunk of new prompt tokens, written this step and
    attended causally (every base length is at least q_len)."""
    w = WORKLOADS[base](q_len=q_len, **kw)
    assert int(w.seq_lens.min()) >= q_len
    w.name = f"{base}-chunk{q_len}"
    return w


WORKLOADS = {
    "tiny": tiny,
    "qwen2.5-1.5b-B1": lambda **kw: qwen25_1p5b(1, **kw),
    "qwen2.5-1.5b-B8": lambda **kw: qwen25_1p5b(8, **kw),
    "qwen2.5-7b-bs16": lambda **kw: qwen25_7b(16, **kw),
    "qwen2.5-7b-bs256": lambda **kw: qwen25_7b(256, **kw),
    "long-B1-L4096": lambda **kw: long_context(1, 4096, **kw),
    "long-B2-L4096": lambda **kw: long_context(2, 4096, **kw),
    "long-B1-L32768": lambda **kw: long_context(1, 32768, **kw),
    "long-B2-L32768": lambda **kw: long_context(2, 32768, **kw),
    "qwen3-0.6b-B256": lambda **kw: qwen3_0p6b(256, **kw),
}
# multi-query (speculative verification) families: the pages' 1.5B target model
# verifying drafts, and the 7B / Qwen3 layers with four queries per sequence
WORKLOADS.update({
    # the Qwen3 batch decoded as a cascade over its 8 shared prefix blocks
    "qwen3-0.6b-B256-cascade": lambda **kw: _cascade(qwen3_0p6b(256, **kw), 8),
    # FP8 (e4m3) pools: the 7B layer, the long-context stress, the Qwen3 batch
    "qwen2.5-7b-bs16-fp8": lambda **kw: with_fp8_pools(qwen25_7b(16, **kw)),
    "long-B2-L32768-fp8": lambda **kw: with_fp8_pools(long_context(2, 32768, **kw)),
    "qwen3-0.6b-B256-fp8": lambda **kw: with_fp8_pools(qwen3_0p6b(256, **kw)),
    "qwen2.5-1.5b-B8-spec4": lambda **kw: spec_verify("qwen2.5-1.5b-B8", 4, **kw),
    "qwen2.5-7b-bs16-spec4": lambda **kw: spec_verify("qwen2.5-7b-bs16", 4, **kw),
    "qwen3-0.6b-B256-spec4": lambda **kw: spec_verify("qwen3-0.6b-B256", 4, **kw),
    # a long shared prefix (2048 tokens) in front of every sequence, decoded
    # plainly and as a cascade
    "qwen3-0.6b-B256-prefix2048": lambda **kw: qwen3_long_prefix(256, 128, **kw),
    "qwen3-0.6b-B256-prefix2048-cascade": lambda **kw: _cascade(qwen3_long_prefix(256, 128, **kw), 128),
    # a few sequences behind a 16384-token shared prefix (a long shared document)
    "qwen3-0.6b-B8-prefix16384": lambda **kw: qwen3_long_prefix(8, 1024, **kw),
    "qwen3-0.6b-B8-prefix16384-cascade": lambda **kw: _cascade(qwen3_long_prefix(8, 1024, **kw), 1024),
    # parallel samples of one 65536-token document: a prefix larger than L2
    "qwen3-0.6b-B4-prefix65536": lambda **kw: qwen3_long_prefix(4, 4096, **kw),
    "qwen3-0.6b-B4-prefix65536-cascade": lambda **kw: _cascade(qwen3_long_prefix(4, 4096, **kw), 4096),
    # one 512-token chunked-prefill chunk per sequence on the Qwen2.5-1.5B layer
    "qwen2.5-1.5b-B1-chunk512": lambda **kw: prefill_chunk("qwen2.5-1.5b-B1", 512, **kw),
    "qwen2.5-1.5b-B8-chunk512": lambda **kw: prefill_chunk("qwen2.5-1.5b-B8", 512, **kw),
})
