"""Small shared helpers for the tests: building paged caches from dense K/V and
converting between bf16 bit patterns and floats.  No attention or conv
arithmetic lives here."""
from __future__ import annotations

import numpy as np
import torch


def to_bits(x) -> np.ndarray:
    """float array -> bf16 bit patterns (torch's round-to-nearest-even from fp32)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def from_bits(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def paged_cache(k_dense, v_dense, block_size, Hkv, d, perm_seed=None, spare=0):
    """Lay out dense per-sequence K/V (lists of [T_b][Hkv][d] bit arrays) as a paged
    cache [num_blocks][Hkv][block_size][d] plus a block table.  Blocks are handed out
    in order, or in a seeded random order when perm_seed is given.  Unused slots
    get a recognisable filler (bf16 bits 0x3F80 = 1.0)."""
    B = len(k_dense)
    nblk = [(kd.shape[0] + block_size - 1) // block_size for kd in k_dense]
    total = sum(nblk) + spare
    order = np.arange(total)
    if perm_seed is not None:
        order = np.random.default_rng(perm_seed).permutation(total)
    table = np.full((B, max(1, max(nblk))), -1, dtype=np.int32)
    kc = np.full((total, Hkv, block_size, d), 0x3F80, dtype=np.uint16)
    vc = np.full((total, Hkv, block_size, d), 0x3F80, dtype=np.uint16)
    pos = 0
    for b in range(B):
        for i in range(nblk[b]):
            table[b, i] = order[pos]
            pos += 1
        T = k_dense[b].shape[0]
        for j in range(T):
            blk, off = table[b, j // block_size], j % block_size
            kc[blk, :, off, :] = k_dense[b][j]
            vc[blk, :, off, :] = v_dense[b][j]
    return kc, vc, table


def bf16_ulp_diff(a_bits, b_bits) -> np.ndarray:
    """|a - b| in units of the bf16 spacing at max(|a|, |b|), element-wise."""
    a, b = from_bits(a_bits), from_bits(b_bits)
    m = np.maximum(np.abs(a), np.abs(b))
    ulp = np.exp2(np.floor(np.log2(np.maximum(m, 2.0 ** -126))) - 7)
    return np.abs(a - b) / ulp


def compact_cache(k_cache_bits, v_cache_bits, block_table, seqlen_k, seqs, block_size=64):
    """The blocks of the listed sequences only, with a block table renumbered to match
    (so the oracle can run on a few sequences of a large paged cache)."""
    rows, blocks = [], []
    for b in seqs:
        n = (int(seqlen_k[b]) + block_size - 1) // block_size
        ids = np.asarray(block_table[b, :n])
        rows.append(np.arange(len(blocks), len(blocks) + n))
        blocks.extend(ids.tolist())
    idx = np.asarray(blocks)
    table = np.full((len(seqs), max(len(r) for r in rows)), -1, np.int32)
    for i, r in enumerate(rows):
        table[i, :len(r)] = r
    return k_cache_bits[idx], v_cache_bits[idx], table
