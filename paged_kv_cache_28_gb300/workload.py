"""Seeded synthetic decode batches for paged-KV attention.

This module draws inputs only: sequence lengths, block placement, K/V/Q values
and the block tables / slot mapping that describe them.  It holds none of the
attention or quantisation arithmetic, so both the CUDA path and the CPU oracle
can be fed from it.

The batch shapes follow the traffic described in "appendonly" (rajatmohan.com):
prompt lengths with median 2,400 and p95 about 18,000 tokens ("traffic"),
70B-class attention with 8 KV heads of dimension 128 ("What is actually being
cached"), fixed 16- or 32-token blocks with per-sequence block tables
("Paging"), and a 900-token system prompt shared by many requests ("Prefix
sharing").  The free-list semantics of the allocator follow the worked example
of "KV Cache Engineering for LLM Serving", section 10 (Paging).

Every array is numpy.  Values are drawn with numpy's PCG64 generator, which
gives the same numbers on every platform.  K/V/Q are N(0, 1) rounded to bf16.
FP8 pools hold E4M3 codes drawn as RNE(N(0,1) * 112) clipped to +-448 with
per-(block, head) scales 4/448 * U(0.8, 1.2); 4-bit pools hold codes
clip(rint(N(0,1) * 7/3), -7, 7) with scales 3/7 * U(0.8, 1.2).  These are
random inputs of the right format, not the product's quantiser.
"""
from __future__ import annotations

import dataclasses
import math
import os
from collections import deque

import numpy as np

LOGNORMAL_SIGMA = math.log(18000 / 2400) / 1.6448536269514722   # p95 / median of the traffic


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_to_float(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


class BlockAllocator:
    """FIFO free list of physical block ids.

    allocate(n) takes the n ids at the front of the free list; free(ids) appends
    them at the back in the given order -- the semantics of the worked example in
    "KV Cache Engineering for LLM Serving", section 10.
    """

    def __init__(self, free_ids):
        self.free = deque(int(i) for i in free_ids)

    def allocate(self, n: int) -> list[int]:
        if n > len(self.free):
            raise MemoryError(f"pool exhausted: need {n}, have {len(self.free)}")
        return [self.free.popleft() for _ in range(n)]

    def release(self, ids) -> None:
        self.free.extend(int(i) for i in ids)


@dataclasses.dataclass
class Batch:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    nblocks: int
    max_blocks: int
    kv_dtype: str                      # "bf16", "fp8_e4m3" or "int4"
    seq_lens: np.ndarray               # int32 [B]
    block_tables: np.ndarray           # int32 [B, max_blocks] (unused entries -1)
    slot_mapping: np.ndarray           # int64 [B]: slot of position seq_len-1 (this step's token)
    q: np.ndarray                      # uint16 [B, Hq, D] (bf16 bits)
    k_new: np.ndarray                  # uint16 [B, Hkv, D]
    v_new: np.ndarray                  # uint16 [B, Hkv, D]
    k_pool: np.ndarray | None          # uint16 / uint8 [nblocks, bs, Hkv, D] (int4: D / 2)
    v_pool: np.ndarray | None
    k_scale: np.ndarray | None         # float32 [nblocks, Hkv] (fp8 only)
    v_scale: np.ndarray | None
    sm_scale: float
    seed: int
    shared_prefix_lens: np.ndarray | None = None   # int32 [B]: tokens in blocks shared with others
    prefix_groups: tuple = ()          # ((prefix tokens, [member sequences]), ...) as built

    @property
    def quantized(self) -> bool:
        return self.kv_dtype in ("fp8_e4m3", "int4")

    @property
    def elem_bytes(self) -> float:
        return {"bf16": 2, "fp8_e4m3": 1, "int4": 0.5}[self.kv_dtype]

    @property
    def logical_tokens(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum())

    def unique_kv_tokens(self, window: int = 0) -> int:
        """Distinct (physical block, row) token slots that some sequence reads; with a
        window only the last `window` positions of each sequence count."""
        rows: dict[int, set] = {}
        bs = self.block_size
        for b in range(self.B):
            L = int(self.seq_lens[b])
            first = L - window if (window > 0 and L > window) else 0
            for j in range(first // bs, (L + bs - 1) // bs):
                lo, hi = max(first, j * bs) - j * bs, min(L, (j + 1) * bs) - j * bs
                rows.setdefault(int(self.block_tables[b, j]), set()).update(range(lo, hi))
        return sum(len(r) for r in rows.values())

    def kv_bytes_per_token(self) -> int:
        """K and V of every KV head for one token of one layer."""
        return int(2 * self.Hkv * self.D * self.elem_bytes)

    def scale_bytes_per_block(self) -> int:
        return 2 * self.Hkv * 4 if self.quantized else 0


# --------------------------------------------------------------------------
# value draws
# --------------------------------------------------------------------------

_CHUNK = 1 << 22


def _chunked(rng: np.random.Generator, n: int, fill) -> None:
    """Run fill(child_rng, start, end) over fixed 4M-element chunks in threads.

    Each chunk has its own generator spawned from one draw of `rng`, so the
    result depends only on the seed (not on the thread count)."""
    import concurrent.futures
    ss = np.random.SeedSequence(int(rng.integers(0, 2 ** 63)))
    starts = list(range(0, n, _CHUNK))
    children = ss.spawn(len(starts))
    work = [(np.random.default_rng(c), s, min(n, s + _CHUNK)) for c, s in zip(children, starts)]
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
        list(ex.map(lambda w: fill(*w), work))


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)

    def fill(g, s, e):
        out[s:e] = bf16_bits(g.standard_normal(e - s, dtype=np.float32))

    _chunked(rng, n, fill)
    return out.reshape(shape)


def _int4_codes(rng: np.random.Generator, shape) -> np.ndarray:
    """Packed 4-bit codes: clip(rint(N(0,1) * 7 / 3), -7, 7) + 8 per element, two per byte
    (element 2j in the low nibble); shape's last dim is D / 2."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint8)

    def fill(g, s, e):
        c = np.clip(np.rint(g.standard_normal(2 * (e - s), dtype=np.float32) * np.float32(7 / 3)),
                    -7, 7).astype(np.int16) + 8
        out[s:e] = (c[0::2] | (c[1::2] << 4)).astype(np.uint8)

    _chunked(rng, n, fill)
    return out.reshape(shape)


def _fp8_codes(rng: np.random.Generator, shape) -> np.ndarray:
    import torch  # float8_e4m3fn rounding of the drawn values (input format only)
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint8)

    def fill(g, s, e):
        x = np.clip(g.standard_normal(e - s, dtype=np.float32) * np.float32(112.0), -448, 448)
        out[s:e] = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()

    _chunked(rng, n, fill)
    return out.reshape(shape)


# --------------------------------------------------------------------------
# batch construction
# --------------------------------------------------------------------------

def _layout(rng, seq_lens, bs, max_blocks, pool_factor, prefix_groups=()):
    """Place blocks in a pool: returns (nblocks, block_tables, cow_copies).

    prefix_groups: iterable of (prefix_tokens, [sequence indices]); the full
    blocks of the prefix are one set of physical blocks shared by the group; a
    partial last prefix block is copied into a private block of each sequence
    (copy-on-write), listed in cow_copies as (src_block, dst_block, rows).
    """
    B = len(seq_lens)
    nb = [(int(L) + bs - 1) // bs for L in seq_lens]
    member = {}
    for gi, (plen, seqs) in enumerate(prefix_groups):
        for b in seqs:
            member[b] = gi
    shared_full = [plen // bs for plen, _ in prefix_groups]
    need = sum(shared_full) + sum(1 for plen, _ in prefix_groups if plen % bs)
    for b in range(B):
        need += nb[b] - (shared_full[member[b]] if b in member else 0)
    nblocks = max(1, math.ceil(pool_factor * need))
    alloc = BlockAllocator(rng.permutation(nblocks))
    tables = np.full((B, max_blocks), -1, dtype=np.int32)
    group_blocks = []
    cow = []
    for plen, _ in prefix_groups:
        full = alloc.allocate(plen // bs)
        src_tail = alloc.allocate(1)[0] if plen % bs else None
        group_blocks.append((full, src_tail, plen % bs))
    for b in range(B):
        if b in member:
            full, src_tail, rows = group_blocks[member[b]]
            own = alloc.allocate(nb[b] - len(full))
            tables[b, :len(full)] = full
            tables[b, len(full):nb[b]] = own
            if src_tail is not None:
                cow.append((src_tail, own[0], rows))
        else:
            tables[b, :nb[b]] = alloc.allocate(nb[b])
    return nblocks, tables, cow


def build_batch(name: str, seq_lens, *, Hq: int, Hkv: int, D: int, block_size: int,
                max_blocks: int | None = None, pool_factor: float = 1.2, seed: int = 0,
                kv_dtype: str = "bf16", prefix_groups=(), with_pools: bool = True,
                sm_scale: float | None = None) -> Batch:
    """A decode batch whose position seq_len-1 is this step's new token.

    The pools hold random values at every row (including rows this step will
    overwrite); k_new / v_new are the new token's vectors, to be written at
    slot_mapping by the cache write.  Sequences of length 0 get slot -1.
    """
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = int(seq_lens.size)
    bs = block_size
    if max_blocks is None:
        max_blocks = max(1, int(((seq_lens.max() if B else 1) + bs - 1) // bs))
    nblocks, tables, cow = _layout(rng, seq_lens, bs, max_blocks, pool_factor, prefix_groups)
    slot = np.full(B, -1, dtype=np.int64)
    for b in range(B):
        L = int(seq_lens[b])
        if L > 0:
            slot[b] = int(tables[b, (L - 1) // bs]) * bs + (L - 1) % bs
    q = _normal_bf16(rng, (B, Hq, D))
    k_new = _normal_bf16(rng, (B, Hkv, D))
    v_new = _normal_bf16(rng, (B, Hkv, D))
    k_pool = v_pool = k_scale = v_scale = None
    if with_pools:
        shape = (nblocks, bs, Hkv, D)
        if kv_dtype == "fp8_e4m3":
            k_pool = _fp8_codes(rng, shape)
            v_pool = _fp8_codes(rng, shape)
            k_scale = (np.float32(4.0 / 448.0) *
                       rng.uniform(0.8, 1.2, (nblocks, Hkv)).astype(np.float32))
            v_scale = (np.float32(4.0 / 448.0) *
                       rng.uniform(0.8, 1.2, (nblocks, Hkv)).astype(np.float32))
        elif kv_dtype == "int4":
            shape4 = (nblocks, bs, Hkv, D // 2)
            k_pool = _int4_codes(rng, shape4)
            v_pool = _int4_codes(rng, shape4)
            k_scale = (np.float32(3.0 / 7.0) *
                       rng.uniform(0.8, 1.2, (nblocks, Hkv)).astype(np.float32))
            v_scale = (np.float32(3.0 / 7.0) *
                       rng.uniform(0.8, 1.2, (nblocks, Hkv)).astype(np.float32))
        else:
            k_pool = _normal_bf16(rng, shape)
            v_pool = _normal_bf16(rng, shape)
        for src, dst, rows in cow:
            k_pool[dst, :rows] = k_pool[src, :rows]
            v_pool[dst, :rows] = v_pool[src, :rows]
            if k_scale is not None:
                k_scale[dst] = k_scale[src]
                v_scale[dst] = v_scale[src]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    shared = None
    if prefix_groups:
        shared = np.zeros(B, dtype=np.int32)
        for plen, seqs in prefix_groups:
            for b in seqs:
                shared[b] = (plen // bs) * bs        # the copied tail block is private
    return Batch(name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=bs, nblocks=nblocks,
                 max_blocks=max_blocks, kv_dtype=kv_dtype, seq_lens=seq_lens,
                 block_tables=tables, slot_mapping=slot, q=q, k_new=k_new, v_new=v_new,
                 k_pool=k_pool, v_pool=v_pool, k_scale=k_scale, v_scale=v_scale,
                 sm_scale=float(sm_scale), seed=seed, shared_prefix_lens=shared,
                 prefix_groups=tuple((int(plen), list(seqs)) for plen, seqs in prefix_groups))


def cascade_groups(batch: Batch):
    """The batch's prefix groups as cascade arrays: (group_offsets, group_seqs,
    group_prefix_len) int32, each group's shared length cut down to whole 16-token
    tiles (the copied tail block holds the same values, so it counts as shared)."""
    offsets, seqs, plen = [0], [], []
    for tokens, members in batch.prefix_groups:
        seqs.extend(members)
        offsets.append(len(seqs))
        plen.append((tokens // 16) * 16)
    return (np.asarray(offsets, np.int32), np.asarray(seqs, np.int32),
            np.asarray(plen, np.int32))


def lognormal_lens(rng, n: int, median: float, lo: int, hi: int) -> np.ndarray:
    x = rng.lognormal(math.log(median), LOGNORMAL_SIGMA, n)
    return np.clip(np.rint(x), lo, hi).astype(np.int32)


# --------------------------------------------------------------------------
# the five named workloads
# --------------------------------------------------------------------------

CONFIGS = ("tiny", "llama70b_layer", "prefix_sharing", "long_context", "fp8_mixed",
           "int4_mixed", "code_assistant_turns")


def config_seq_lens(name: str, seed: int):
    """(seq_lens, prefix_groups, shape kwargs) of a named workload."""
    rng = np.random.default_rng(seed + 1000)
    if name == "tiny":
        return (np.array([1, 17, 33, 100], np.int32), (),
                dict(Hq=8, Hkv=2, D=64, block_size=16, max_blocks=8))
    if name == "llama70b_layer":
        return (lognormal_lens(rng, 64, 2400, 1, 32768), (),
                dict(Hq=64, Hkv=8, D=128, block_size=16, max_blocks=2048))
    if name == "prefix_sharing":
        s1 = lognormal_lens(rng, 240, 1500, 1, 32768 - 900)
        s2 = rng.integers(100, 2001, 16).astype(np.int32)
        lens = np.concatenate([900 + s1, 8000 + s2]).astype(np.int32)
        groups = ((900, list(range(240))), (8000, list(range(240, 256))))
        return lens, groups, dict(Hq=64, Hkv=8, D=128, block_size=16, max_blocks=2048)
    if name == "long_context":
        return (np.full(8, 131072, np.int32), (),
                dict(Hq=64, Hkv=8, D=128, block_size=32, max_blocks=4096))
    if name == "code_assistant_turns":
        # 32 repositories, 8 turns each: a turn shares its repository's files (a
        # LogNormal(8000) prefix) with the other turns and adds its own conversation
        # (LogNormal(1500)); the shared KV (~1.4 GB) is far larger than L2
        plen = lognormal_lens(rng, 32, 8000, 2048, 24576)
        sfx = lognormal_lens(rng, 256, 1500, 1, 32768 - 24576)
        lens = np.array([plen[i // 8] + sfx[i] for i in range(256)], np.int32)
        groups = tuple((int(plen[g]), list(range(8 * g, 8 * g + 8))) for g in range(32))
        return lens, groups, dict(Hq=64, Hkv=8, D=128, block_size=16, max_blocks=2048)
    if name in ("fp8_mixed", "int4_mixed"):
        return (rng.integers(1, 4097, 512).astype(np.int32), (),
                dict(Hq=64, Hkv=8, D=128, block_size=16, max_blocks=256,
                     kv_dtype="fp8_e4m3" if name == "fp8_mixed" else "int4"))
    raise KeyError(name)


DEFAULT_SEEDS = {"tiny": 0, "llama70b_layer": 1, "prefix_sharing": 2, "long_context": 3,
                 "fp8_mixed": 4, "int4_mixed": 5, "code_assistant_turns": 6}


def make(name: str, seed: int | None = None, with_pools: bool = True) -> Batch:
    seed = DEFAULT_SEEDS[name] if seed is None else seed
    lens, groups, kw = config_seq_lens(name, seed)
    if name == "tiny":
        kw = dict(kw, pool_factor=64 / 13)      # 13 blocks in a 64-block pool
    return build_batch(name, lens, seed=seed, prefix_groups=groups, with_pools=with_pools, **kw)
