"""Pins of the oracle's qkvr projection step (the linears in front of the prologue):
a hand-derived fixture (tests/golden/hand_qkvr.txt) with single roundings at and beside
bf16 ties, numpy's float64 product within half a bf16 ulp, feature selection by unit
rows, exact scaling, and the prologue applied to the projected q, k, v."""
import os

import numpy as np

from helpers import from_bits, to_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_qkvr_hand_golden(oracle_mod):
    W = np.array([[1, 0, 0], [0, 1, 0], [1, 1, 0], [0, 1, -1], [2, 0, 1], [0, 0, 3], [1, 1, 1]], np.float64)
    rows = []
    with open(os.path.join(GOLDEN, "hand_qkvr.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([np.array(part.split(), dtype=np.float64) for part in line.split(";")])
    x = np.stack([r[0] for r in rows])
    y = np.stack([r[1] for r in rows])
    xb = to_bits(x)
    assert np.array_equal(from_bits(xb), x)
    q, k, v, r = oracle_mod.qkvr_projection(xb, to_bits(W), Hq=1, Hkv=1, d=2, d_r=1)
    got = np.concatenate([from_bits(q).reshape(-1, 2), from_bits(k), from_bits(v), from_bits(r).reshape(-1, 1)], 1)
    assert np.array_equal(got, y)


def test_qkvr_matches_float64_product(oracle_mod):
    rng = np.random.default_rng(41)
    Hq, Hkv, d, d_r, D = 4, 2, 8, 4, 40
    x = to_bits(rng.standard_normal((7, D)))
    w = to_bits(0.2 * rng.standard_normal((Hq * d + 2 * Hkv * d + Hq * d_r, D)))
    q, k, v, r = oracle_mod.qkvr_projection(x, w, Hq=Hq, Hkv=Hkv, d=d, d_r=d_r)
    ref = from_bits(x) @ from_bits(w).T
    got = np.concatenate([from_bits(q).reshape(7, -1), from_bits(k), from_bits(v), from_bits(r).reshape(7, -1)], 1)
    half_ulp = 0.5 * np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    assert np.all(np.abs(got - ref) <= half_ulp * (1 + 1e-12))
    # order of the slices: a unit row picks one input feature into one output feature
    w2 = np.zeros((Hq * d + 2 * Hkv * d + Hq * d_r, D))
    w2[Hq * d + 3, 5] = 1.0            # k feature 3 <- x feature 5
    w2[Hq * d + 2 * Hkv * d + 1, 9] = 1.0   # r head 0, feature 1 <- x feature 9
    q, k, v, r = oracle_mod.qkvr_projection(x, to_bits(w2), Hq=Hq, Hkv=Hkv, d=d, d_r=d_r)
    assert np.array_equal(k[:, 3], x[:, 5]) and np.array_equal(r[:, 0, 1], x[:, 9])
    assert not from_bits(q).any() and not from_bits(v).any()
    # exact scaling: x times 4 scales y by 4
    q4, k4, v4, r4 = oracle_mod.qkvr_projection(to_bits(from_bits(x) * 4), w, Hq=Hq, Hkv=Hkv, d=d, d_r=d_r)
    q1, k1, v1, r1 = oracle_mod.qkvr_projection(x, w, Hq=Hq, Hkv=Hkv, d=d, d_r=d_r)
    assert np.array_equal(from_bits(k4), from_bits(k1) * 4) and np.array_equal(from_bits(r4), from_bits(r1) * 4)


def test_qkvr_prologue_is_the_prologue_of_the_projections(oracle_mod):
    rng = np.random.default_rng(42)
    Hq, Hkv, d, d_r, D = 4, 2, 8, 4, 24
    q_lens = [5, 2]
    N = sum(q_lens)
    cu = np.array([0, 5, 7], np.int32)
    x = to_bits(rng.standard_normal((N, D)))
    w = to_bits(0.3 * rng.standard_normal((Hq * d + 2 * Hkv * d + Hq * d_r, D)))
    C = Hkv * d
    common = dict(cu_seqlens_q=cu, Hq=Hq, Hkv=Hkv, d=d, conv_w_k=(0.5 * rng.standard_normal((C, 4))).astype(np.float32),
                  conv_w_v=(0.5 * rng.standard_normal((C, 4))).astype(np.float32),
                  q_norm_w=np.ones(d, np.float32), k_norm_w=np.ones(d, np.float32), eps=1e-6,
                  state_slot=np.array([0, 1], np.int32), conv_state_k=to_bits(rng.standard_normal((2, 3, C))),
                  conv_state_v=to_bits(rng.standard_normal((2, 3, C))), slot_mapping=np.arange(N, dtype=np.int32),
                  block_size=4, k_cache=np.zeros((2, Hkv, 4, d), np.uint16), v_cache=np.zeros((2, Hkv, 4, d), np.uint16))
    out = oracle_mod.qkvr_prologue(x=x, w=w, d_r=d_r, **common)
    q, k, v, r = oracle_mod.qkvr_projection(x, w, Hq=Hq, Hkv=Hkv, d=d, d_r=d_r)
    ref = oracle_mod.prologue(q=q, k=k, v=v, **common)
    for key in ("q_out", "k_cache", "v_cache", "conv_state_k", "conv_state_v"):
        assert np.array_equal(out[key], ref[key]), key
    assert np.array_equal(out["r"], r)
    # the new conv state holds the last 3 projected k rows of each sequence
    assert np.array_equal(out["conv_state_k"][0], k[2:5])
