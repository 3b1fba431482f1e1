"""Pins of the oracle's attention-output ShortConv + residual add + RMSNorm.

Checked against a hand-derived fixture (tests/golden/hand_output_conv.txt), numpy
correlate for the conv, torch rms_norm for the norm over the whole hidden row, exact
special cases (delta filter, zero filter, ties of the residual sum) and invariants of
the definition (state carry, chunking, scale invariance).
"""
import os

import numpy as np
import torch
import torch.nn.functional as F

from helpers import from_bits, to_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _case(rng, q_lens, D=64, state=None, w=None, g=None, eps=1e-6, res_scale=1.0):
    B = len(q_lens)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    N = int(cu[-1])
    if w is None:
        w = (0.5 * rng.standard_normal((D, 4))).astype(np.float32)
    if g is None:
        g = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    if state is None:
        state = to_bits(rng.standard_normal((B + 2, 3, D)))
    return dict(cu_seqlens_q=cu, D=D, y=to_bits(rng.standard_normal((N, D))), conv_w=w,
                state_slot=(np.arange(B, dtype=np.int32) + 2) % (B + 2), conv_state=state,
                residual=to_bits(res_scale * rng.standard_normal((N, D))), norm_w=g, eps=eps)


def _half_ulp(x):
    return 0.5 * np.exp2(np.floor(np.log2(np.maximum(np.abs(x), 1e-30))) - 7)


def test_output_conv_hand_golden(oracle_mod):
    cases = []
    with open(os.path.join(GOLDEN, "hand_output_conv.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                cases.append([np.array([r.split() for r in part.split("|")], dtype=np.float64)
                              for part in line.split(";")])
    w = np.array([[0, 0, 1, 2], [1, 0, 0, 1]], np.float32)
    g = np.array([1, 2], np.float32)
    for state, y, res, h, out, new_state in cases:
        n = y.shape[0]
        got = oracle_mod.output_conv(
            cu_seqlens_q=np.array([0, n], np.int32), D=2, y=to_bits(y), conv_w=w,
            state_slot=np.array([0], np.int32), conv_state=to_bits(state[None]),
            residual=to_bits(res), norm_w=g, eps=0.0)
        assert np.array_equal(from_bits(got["h"]), h)
        assert np.array_equal(got["out"], np.vectorize(oracle_mod.f64_to_bf16_bits)(out).astype(np.uint16))
        assert np.array_equal(from_bits(got["conv_state"][0]), new_state)


def test_output_conv_matches_numpy_correlate(oracle_mod):
    rng = np.random.default_rng(21)
    a = _case(rng, [7, 1, 12, 2], D=24)
    got = oracle_mod.output_conv(**a, want_conv=True)
    cu = a["cu_seqlens_q"]
    for b in range(len(cu) - 1):
        xs = np.concatenate([from_bits(a["conv_state"][a["state_slot"][b]]),
                             from_bits(a["y"][cu[b]:cu[b + 1]])], axis=0)
        for c in range(a["D"]):
            ref = np.correlate(xs[:, c], a["conv_w"][c].astype(np.float64), mode="valid")
            conv = from_bits(got["conv"][cu[b]:cu[b + 1], c])
            assert np.all(np.abs(conv - ref) <= _half_ulp(ref) * (1 + 1e-12) + 1e-300), (b, c)
    # h adds the ROUNDED conv output to the residual and rounds once: the fp32 sum of two
    # bf16 values rounds to the same bf16 as their exact sum (torch rounds fp32 -> bf16)
    s32 = (from_bits(a["residual"]) + from_bits(got["conv"])).astype(np.float32)
    assert np.array_equal(got["h"], to_bits(s32))
    # out is the RMSNorm of the bf16 h over the hidden row
    ref = F.rms_norm(torch.from_numpy(from_bits(got["h"])), (a["D"],),
                     weight=torch.from_numpy(a["norm_w"].astype(np.float64)), eps=a["eps"]).numpy()
    assert np.all(np.abs(from_bits(got["out"]) - ref) <= _half_ulp(ref) * (1 + 1e-9))


def test_delta_filter_zero_residual_is_rms_norm_of_y(oracle_mod):
    rng = np.random.default_rng(22)
    D = 256
    w = np.zeros((D, 4), np.float32)
    w[:, 3] = 1.0
    a = _case(rng, [5, 3], D=D, w=w)
    a["residual"] = np.zeros_like(a["residual"])
    got = oracle_mod.output_conv(**a)
    assert np.array_equal(got["h"], a["y"])
    # the norm runs over the whole hidden row (all D channels), not per head of 128
    ref = F.rms_norm(torch.from_numpy(from_bits(a["y"])), (D,),
                     weight=torch.from_numpy(a["norm_w"].astype(np.float64)), eps=1e-6).numpy()
    assert np.all(np.abs(from_bits(got["out"]) - ref) <= _half_ulp(ref) * (1 + 1e-9))


def test_zero_filter_passes_the_residual(oracle_mod):
    rng = np.random.default_rng(23)
    D = 64
    a = _case(rng, [9], D=D, w=np.zeros((D, 4), np.float32))
    got = oracle_mod.output_conv(**a)
    assert np.array_equal(got["h"], a["residual"])
    ref = F.rms_norm(torch.from_numpy(from_bits(a["residual"])), (D,),
                     weight=torch.from_numpy(a["norm_w"].astype(np.float64)), eps=1e-6).numpy()
    assert np.all(np.abs(from_bits(got["out"]) - ref) <= _half_ulp(ref) * (1 + 1e-9))


def test_residual_sum_rounds_once_to_nearest_even(oracle_mod):
    """h for sums that fall on bf16 ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7
    (even: 1); (1 + 2^-7) + 2^-8 halfway between 1 + 2^-7 and 1 + 2^-6 (even: 1 + 2^-6);
    -(1 + 2^-8) rounds to -1."""
    D = 1
    w = np.array([[0, 0, 0, 1]], np.float32)     # conv = the current token
    y = np.array([[2.0 ** -8], [2.0 ** -8], [-(2.0 ** -8)], [3.0]])
    res = np.array([[1.0], [1 + 2.0 ** -7], [-1.0], [-3.0]])
    got = oracle_mod.output_conv(cu_seqlens_q=np.array([0, 4], np.int32), D=D, y=to_bits(y),
                                 conv_w=w, state_slot=np.array([0], np.int32),
                                 conv_state=np.zeros((1, 3, 1), np.uint16), residual=to_bits(res),
                                 norm_w=np.ones(1, np.float32), eps=0.0)
    assert list(from_bits(got["h"][:, 0])) == [1.0, 1 + 2.0 ** -6, -1.0, 0.0]
    # a single channel normalises to its sign (eps 0); 0 / 0 stays undefined and is not checked
    assert list(from_bits(got["out"][:3, 0])) == [1.0, 1.0, -1.0]


def test_state_carry_short_sequences(oracle_mod):
    rng = np.random.default_rng(24)
    a = _case(rng, [1, 2, 0, 3, 5], D=16)
    got = oracle_mod.output_conv(**a)
    cu = a["cu_seqlens_q"]
    for b in range(5):
        slot = a["state_slot"][b]
        xs = np.concatenate([a["conv_state"][slot], a["y"][cu[b]:cu[b + 1]]], axis=0)
        assert np.array_equal(got["conv_state"][slot], xs[-3:])
    # slots no sequence names are left alone
    used = set(a["state_slot"].tolist())
    for s in range(a["conv_state"].shape[0]):
        if s not in used:
            assert np.array_equal(got["conv_state"][s], a["conv_state"][s])


def test_chunking_invariance(oracle_mod):
    """Splitting a sequence into chunks with the state carried gives identical results."""
    rng = np.random.default_rng(25)
    a = _case(rng, [30], D=16)
    ref = oracle_mod.output_conv(**a)
    state = a["conv_state"].copy()
    hs, outs = [], []
    for lo, hi in ((0, 1), (1, 3), (3, 17), (17, 30)):
        part = dict(a)
        part.update(cu_seqlens_q=np.array([0, hi - lo], np.int32), y=a["y"][lo:hi],
                    residual=a["residual"][lo:hi], conv_state=state)
        got = oracle_mod.output_conv(**part)
        hs.append(got["h"]); outs.append(got["out"]); state = got["conv_state"]
    assert np.array_equal(np.concatenate(hs), ref["h"])
    assert np.array_equal(np.concatenate(outs), ref["out"])
    assert np.array_equal(state, ref["conv_state"])


def test_scale_invariance(oracle_mod):
    """Scaling y, the state and the residual by 8 (exact in bf16) scales h by 8 and leaves
    the normalised output unchanged (eps = 0)."""
    rng = np.random.default_rng(26)
    a = _case(rng, [6, 4], D=32, eps=0.0)
    ref = oracle_mod.output_conv(**a)
    b = dict(a)
    for k in ("y", "residual", "conv_state"):
        b[k] = to_bits(from_bits(a[k]) * 8.0)
    got = oracle_mod.output_conv(**b)
    assert np.array_equal(from_bits(got["h"]), from_bits(ref["h"]) * 8.0)
    assert np.array_equal(got["out"], ref["out"])
