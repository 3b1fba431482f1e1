"""Seeded synthetic workloads for the Inkling attention hot path.

This module only draws inputs: shapes, index arrays and random values.  It
holds none of the method's arithmetic, and both the CUDA path's tests/bench
and the oracle consume what it produces.

Workloads (all head_dim 128, paged KV block 64):
  tiny     B=1, 256 new tokens, Hq=8, Hkv=1, d_r=32, rel_extent=64, sliding window 128,
           zero initial conv state.
  swa      one sliding-window prefill layer: B=1, 8192 tokens, Hq=64, Hkv=8, d_r=32,
           rel_extent=512, window 4096, random block table.
  full     one full-attention prefill layer: B=1, 32768 tokens, Hq=64, Hkv=8,
           rel_extent=1024, logits scaled by max(1, ln T / ln 8192).
  decode   MTP-verify decode: 32 sequences x 9 query tokens, key length 32768 each
           (32759 cached + 9 new), full attention with the log scaling,
           rel_extent=1024, random block table, random conv state.
  ragged   mixed prefill: 16 sequences, new lengths uniform in [1024, 16384], cached
           prefix uniform in [0, 4096], window 4096, rel_extent=512.

Value distributions: q, k, v, r and cached K/V ~ N(0, 1) rounded to bf16;
P ~ N(0, 0.02^2) fp32 (its standard deviation is the workload field p_std);
ShortConv weights ~ N(0, 0.5^2) fp32; RMSNorm gains 1 + N(0, 0.1^2) fp32; eps 1e-6.
Carried conv-state rows ~ N(0, 1) bf16 where the sequence has that many earlier
tokens, zero otherwise.  The block table is a seeded permutation of all allocated
blocks; every cache slot starts with random bf16 values so that stray writes are detectable.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List

import numpy as np
import torch

BLOCK_SIZE = 64
HEAD_DIM = 128


@dataclasses.dataclass
class Workload:
    name: str
    Hq: int
    Hkv: int
    q_lens: List[int]
    prefix_lens: List[int]
    d_r: int = 32
    rel_extent: int = 0
    window: int = 0               # 0 = full attention
    log_scale_base: float = 0.0   # 0 = no length-dependent logit scaling
    head_dim: int = HEAD_DIM
    block_size: int = BLOCK_SIZE
    random_block_table: bool = True
    eps: float = 1e-6
    spare_blocks: int = 0
    p_std: float = 0.02           # standard deviation of the relative projection P

    @property
    def B(self) -> int:
        return len(self.q_lens)

    @property
    def N_tok(self) -> int:
        return int(sum(self.q_lens))

    @property
    def seqlen_k(self) -> List[int]:
        return [p + n for p, n in zip(self.prefix_lens, self.q_lens)]

    @property
    def max_blocks(self) -> int:
        return max(1, max((s + self.block_size - 1) // self.block_size for s in self.seqlen_k))

    @property
    def num_blocks(self) -> int:
        return (sum((s + self.block_size - 1) // self.block_size for s in self.seqlen_k)
                + self.spare_blocks)

    def describe(self) -> str:
        kind = "full" if self.window == 0 else f"window {self.window}"
        return (f"{self.name}: B={self.B}, new tokens {self.N_tok}, Hq={self.Hq}, Hkv={self.Hkv}, "
                f"d={self.head_dim}, d_r={self.d_r}, rel_extent={self.rel_extent}, {kind}, "
                f"log-scale base {self.log_scale_base or 'off'}")


def workload(name: str, seed: int = 0) -> Workload:
    """The named workload; ragged lengths are drawn from `seed`."""
    if name == "tiny":
        return Workload("tiny", Hq=8, Hkv=1, q_lens=[256], prefix_lens=[0], d_r=32,
                        rel_extent=64, window=128, random_block_table=False)
    if name == "swa":
        return Workload("swa", Hq=64, Hkv=8, q_lens=[8192], prefix_lens=[0], d_r=32,
                        rel_extent=512, window=4096)
    if name == "full":
        return Workload("full", Hq=64, Hkv=8, q_lens=[32768], prefix_lens=[0], d_r=32,
                        rel_extent=1024, window=0, log_scale_base=8192.0)
    if name == "decode":
        return Workload("decode", Hq=64, Hkv=8, q_lens=[9] * 32, prefix_lens=[32768 - 9] * 32,
                        d_r=32, rel_extent=1024, window=0, log_scale_base=8192.0)
    if name == "ragged":
        rng = np.random.Generator(np.random.Philox(key=[seed, 0x5EED]))
        lens = rng.integers(1024, 16384, size=16, endpoint=True).tolist()
        prefix = rng.integers(0, 4096, size=16, endpoint=True).tolist()
        return Workload("ragged", Hq=64, Hkv=8, q_lens=[int(x) for x in lens],
                        prefix_lens=[int(x) for x in prefix], d_r=32, rel_extent=512, window=4096)
    raise KeyError(name)


def custom(name: str, *, Hq: int, Hkv: int, q_lens, prefix_lens=None, **kw) -> Workload:
    prefix_lens = list(prefix_lens) if prefix_lens is not None else [0] * len(q_lens)
    return Workload(name, Hq=Hq, Hkv=Hkv, q_lens=list(q_lens), prefix_lens=prefix_lens, **kw)


_TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "r": 4, "P": 5, "conv_w_k": 6, "conv_w_v": 7,
               "q_norm_w": 8, "k_norm_w": 9, "conv_state_k": 10, "conv_state_v": 11,
               "k_cache": 12, "v_cache": 13, "perm": 14, "y": 15, "residual": 16,
               "oc_conv_w": 17, "oc_norm_w": 18, "oc_conv_state": 19, "k_cache_e4m3": 20,
               "v_cache_e4m3": 21, "x": 22, "w_qkvr": 23}


def _gen(device, seed: int, tensor: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + _TENSOR_IDS[tensor] * 7919) & 0x7FFF_FFFF_FFFF)
    return g


def _normal(shape, std, device, seed, tensor, dtype):
    g = _gen(device, seed, tensor)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def make_inputs(w: Workload, seed: int = 0, device="cpu", kv_dtype: str = "bf16") -> Dict[str, torch.Tensor]:
    """All inputs of one prologue + attention pass, as torch tensors on `device`.

    Keys: q, k, v [N,Hq,d]/[N,C]/[N,C] bf16; r [N,Hq,d_r] bf16; P [Hq,rel_extent,d_r]
    fp32; conv_w_k, conv_w_v [C,4] fp32; q_norm_w, k_norm_w [d] fp32;
    conv_state_k, conv_state_v [B,3,C] bf16; state_slot [B]; cu_seqlens_q [B+1];
    seqlen_k [B]; block_table [B,max_blocks] (-1 past each sequence's blocks);
    slot_mapping [N]; k_cache, v_cache [num_blocks,Hkv,64,d] bf16, or with kv_dtype "e4m3"
    uint8 E4M3 codes plus k_scale, v_scale [num_blocks,Hkv,64] fp32.
    """
    device = torch.device(device)
    d, C, N, B = w.head_dim, w.Hkv * w.head_dim, w.N_tok, w.B
    bf = torch.bfloat16
    out: Dict[str, torch.Tensor] = {}
    out["q"] = _normal((N, w.Hq, d), 1.0, device, seed, "q", bf)
    out["k"] = _normal((N, C), 1.0, device, seed, "k", bf)
    out["v"] = _normal((N, C), 1.0, device, seed, "v", bf)
    out["r"] = _normal((N, w.Hq, w.d_r), 1.0, device, seed, "r", bf)
    out["P"] = _normal((w.Hq, max(w.rel_extent, 1), w.d_r), w.p_std, device, seed, "P", torch.float32)
    out["conv_w_k"] = _normal((C, 4), 0.5, device, seed, "conv_w_k", torch.float32)
    out["conv_w_v"] = _normal((C, 4), 0.5, device, seed, "conv_w_v", torch.float32)
    out["q_norm_w"] = 1.0 + _normal((d,), 0.1, device, seed, "q_norm_w", torch.float32)
    out["k_norm_w"] = 1.0 + _normal((d,), 0.1, device, seed, "k_norm_w", torch.float32)

    # carried conv state: a row is random where the sequence has a token there
    sk = _normal((B, 3, C), 1.0, device, seed, "conv_state_k", bf)
    sv = _normal((B, 3, C), 1.0, device, seed, "conv_state_v", bf)
    for b, p in enumerate(w.prefix_lens):
        missing = max(0, 3 - p)
        if missing:
            sk[b, :missing] = 0
            sv[b, :missing] = 0
    out["conv_state_k"], out["conv_state_v"] = sk, sv
    out["state_slot"] = torch.arange(B, dtype=torch.int32, device=device)

    cu = np.zeros(B + 1, dtype=np.int64)
    cu[1:] = np.cumsum(w.q_lens)
    out["cu_seqlens_q"] = torch.tensor(cu, dtype=torch.int32, device=device)
    out["seqlen_k"] = torch.tensor(w.seqlen_k, dtype=torch.int32, device=device)

    nb = w.num_blocks
    if w.random_block_table:
        g = _gen("cpu", seed, "perm")
        perm = torch.randperm(nb, generator=g).to(torch.int64).numpy()
    else:
        perm = np.arange(nb, dtype=np.int64)
    table = np.full((B, w.max_blocks), -1, dtype=np.int64)
    pos = 0
    for b, s in enumerate(w.seqlen_k):
        n = (s + w.block_size - 1) // w.block_size
        table[b, :n] = perm[pos:pos + n]
        pos += n
    out["block_table"] = torch.tensor(table, dtype=torch.int32, device=device)
    slots = np.empty(N, dtype=np.int64)
    t = 0
    for b in range(B):
        for i in range(w.q_lens[b]):
            p = w.prefix_lens[b] + i
            slots[t] = table[b, p // w.block_size] * w.block_size + p % w.block_size
            t += 1
    out["slot_mapping"] = torch.tensor(slots, dtype=torch.int32, device=device)
    shape = (nb, w.Hkv, w.block_size, d)
    if kv_dtype == "bf16":
        out["k_cache"] = _normal(shape, 1.0, device, seed, "k_cache", bf)
        out["v_cache"] = _normal(shape, 1.0, device, seed, "v_cache", bf)
    elif kv_dtype == "e4m3":
        # E4M3 codes (held as uint8) of N(0, 1) draws times 128, and row scales 2^-7: the
        # cached rows read back as values of about unit size
        for name in ("k", "v"):
            x = _normal(shape, 128.0, device, seed, f"{name}_cache_e4m3", torch.float32)
            out[f"{name}_cache"] = x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
            out[f"{name}_scale"] = torch.full(shape[:3], 2.0 ** -7, dtype=torch.float32, device=device)
    else:
        raise ValueError(kv_dtype)
    return out


def qkvr_features(w: Workload) -> int:
    """Output features of the qkvr projections: Hq*d + 2*Hkv*d + Hq*d_r."""
    return (w.Hq + 2 * w.Hkv) * w.head_dim + w.Hq * w.d_r


def make_qkvr_inputs(w: Workload, d_model: int, seed: int = 0, device="cpu", kv_dtype: str = "bf16",
                     grid: bool = False) -> Dict[str, torch.Tensor]:
    """Inputs of the qkvr projections with the prologue fused in: make_inputs' tensors with
    q, k, v and r replaced by the hidden states x [N, d_model] bf16 and the projection
    weight w_qkvr [F, d_model] bf16 (nn.Linear layout, rows [q heads | k | v | r heads],
    F = qkvr_features(w)); P, seqlen_k and block_table are kept for the attention after it.

    Default: x ~ N(0, 1) and w_qkvr ~ N(0, 1/d_model), so each projection is about N(0, 1).
    grid=True: x = i/8 and w_qkvr = j/64 with integers i, j uniform in [-8, 8]: every product
    is a multiple of 2^-9 and every partial sum of a row is at most d_model/8 in magnitude,
    so for d_model < 2^18 each sum is exact in fp32 whatever the order of accumulation.
    """
    device = torch.device(device)
    out = make_inputs(w, seed=seed, device=device, kv_dtype=kv_dtype)
    for k in ("q", "k", "v", "r"):
        del out[k]
    N, F = w.N_tok, qkvr_features(w)
    bf = torch.bfloat16
    if grid:
        gx, gw = _gen(device, seed, "x"), _gen(device, seed, "w_qkvr")
        out["x"] = (torch.randint(-8, 9, (N, d_model), generator=gx, device=device).to(torch.float32) / 8).to(bf)
        out["w_qkvr"] = (torch.randint(-8, 9, (F, d_model), generator=gw, device=device).to(torch.float32)
                         / 64).to(bf)
    else:
        out["x"] = _normal((N, d_model), 1.0, device, seed, "x", bf)
        out["w_qkvr"] = _normal((F, d_model), d_model ** -0.5, device, seed, "w_qkvr", bf)
    return out


def make_output_conv_inputs(w: Workload, seed: int = 0, device="cpu", D: int = 0) -> Dict[str, torch.Tensor]:
    """Inputs of the attention-output ShortConv + residual + RMSNorm over the workload's
    new tokens, hidden width D (default Hq * head_dim, the attention output's width).

    Keys: y [N,D] bf16 (stands in for the o_proj output) and residual [N,D] bf16, both
    ~ N(0, 1); conv_w [D,4] fp32 ~ N(0, 0.5^2); norm_w [D] fp32 1 + N(0, 0.1^2);
    conv_state [B,3,D] bf16 ~ N(0, 1) where the sequence has earlier tokens, else zero;
    state_slot [B]; cu_seqlens_q [B+1].
    """
    device = torch.device(device)
    D = D or w.Hq * w.head_dim
    N, B = w.N_tok, w.B
    bf = torch.bfloat16
    out: Dict[str, torch.Tensor] = {}
    out["y"] = _normal((N, D), 1.0, device, seed, "y", bf)
    out["residual"] = _normal((N, D), 1.0, device, seed, "residual", bf)
    out["conv_w"] = _normal((D, 4), 0.5, device, seed, "oc_conv_w", torch.float32)
    out["norm_w"] = 1.0 + _normal((D,), 0.1, device, seed, "oc_norm_w", torch.float32)
    st = _normal((B, 3, D), 1.0, device, seed, "oc_conv_state", bf)
    for b, p in enumerate(w.prefix_lens):
        missing = max(0, 3 - p)
        if missing:
            st[b, :missing] = 0
    out["conv_state"] = st
    out["state_slot"] = torch.arange(B, dtype=torch.int32, device=device)
    cu = np.zeros(B + 1, dtype=np.int64)
    cu[1:] = np.cumsum(w.q_lens)
    out["cu_seqlens_q"] = torch.tensor(cu, dtype=torch.int32, device=device)
    return out


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (any device)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16).to(device)
