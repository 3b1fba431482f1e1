"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle against a library routine (torch SDPA, torch
rms_norm, numpy correlate), a closed form, a hand-derived fixture in
tests/golden/, or an invariant the method fixes (zero bias is plain causal
attention, a window >= T is full attention, a delta conv filter is the
identity, the bias depends only on i-j).  They are chosen so that a dropped
term, a wrong sign or index, or a transposed operand fails at least one.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from helpers import from_bits, paged_cache, to_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- rounding, lambda

def test_bf16_rounding_matches_torch_on_fp32_values(oracle_mod):
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000),
                        np.array([0.0, -0.0, 1.0, -1.0, 3.3895313892515355e38, 1e-40])])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_mod.f64_to_bf16_bits(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rounding_ties_to_even_and_direct_from_fp64(oracle_mod):
    # exactly halfway between 1 and 1+2^-7: ties to the even significand (1.0)
    assert oracle_mod.f64_to_bf16_bits(1.0 + 2.0 ** -8) == 0x3F80
    # halfway between 1+2^-7 (odd) and 1+2^-6 (even): rounds up to 1+2^-6
    assert oracle_mod.f64_to_bf16_bits(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # just above halfway: an fp32 detour would land on the tie and go down; direct
    # rounding from fp64 must go up to 1+2^-7
    assert oracle_mod.f64_to_bf16_bits(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle_mod.f64_to_bf16_bits(-(1.0 + 2.0 ** -8 + 2.0 ** -40)) == 0xBF81
    assert oracle_mod.f64_to_bf16_bits(1e39) == 0x7F80


def test_log_scale_closed_form(oracle_mod):
    assert oracle_mod.log_scale(32768, 8192) == pytest.approx(15.0 / 13.0, rel=1e-15)
    assert oracle_mod.log_scale(2 ** 20, 8192) == pytest.approx(20.0 / 13.0, rel=1e-15)
    assert oracle_mod.log_scale(8192, 8192) == pytest.approx(1.0, rel=1e-15)
    assert oracle_mod.log_scale(100, 8192) == 1.0
    assert oracle_mod.log_scale(32768, 0) == 1.0


# ---------------------------------------------------------------- prologue

def _prologue_case(rng, q_lens, Hq=4, Hkv=2, d=8, prefix=None, w=None, state=None,
                   gq=None, gk=None, eps=1e-6, block_size=4):
    B = len(q_lens)
    N = sum(q_lens)
    C = Hkv * d
    prefix = prefix or [0] * B
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = to_bits(rng.standard_normal((N, Hq, d)))
    k = to_bits(rng.standard_normal((N, C)))
    v = to_bits(rng.standard_normal((N, C)))
    if w is None:
        w = rng.standard_normal((C, 4)).astype(np.float32) * 0.5
    if state is None:
        state = to_bits(rng.standard_normal((B, 3, C)))
    nblk = [(p + n + block_size - 1) // block_size for p, n in zip(prefix, q_lens)]
    table = np.full((B, max(nblk)), -1, np.int32)
    perm = rng.permutation(sum(nblk) + 2)
    pos = 0
    for b in range(B):
        table[b, :nblk[b]] = perm[pos:pos + nblk[b]]
        pos += nblk[b]
    slots = []
    for b in range(B):
        for i in range(q_lens[b]):
            p = prefix[b] + i
            slots.append(table[b, p // block_size] * block_size + p % block_size)
    nb = sum(nblk) + 2
    kcache = to_bits(rng.standard_normal((nb, Hkv, block_size, d)))
    vcache = to_bits(rng.standard_normal((nb, Hkv, block_size, d)))
    args = dict(cu_seqlens_q=cu, Hq=Hq, Hkv=Hkv, d=d, q=q, k=k, v=v, conv_w_k=w,
                conv_w_v=w[::-1].copy(), q_norm_w=gq if gq is not None else np.ones(d, np.float32),
                k_norm_w=gk if gk is not None else np.ones(d, np.float32), eps=eps,
                state_slot=np.arange(B, dtype=np.int32), conv_state_k=state,
                conv_state_v=state.copy(), slot_mapping=np.array(slots, np.int32),
                block_size=block_size, k_cache=kcache, v_cache=vcache)
    return args


def test_shortconv_hand_golden(oracle_mod):
    rows = []
    with open(os.path.join(GOLDEN, "hand_shortconv.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([np.array(s.split(), dtype=np.float64) for s in line.split(";")])
    for x, y, new_state in rows:
        n = len(x)
        w = np.array([[1, 2, 3, 4]], np.float32)
        args = dict(cu_seqlens_q=np.array([0, n], np.int32), Hq=1, Hkv=1, d=1,
                    q=to_bits(np.ones((n, 1, 1))), k=to_bits(x.reshape(n, 1)),
                    v=to_bits(x.reshape(n, 1)), conv_w_k=w, conv_w_v=w,
                    q_norm_w=np.ones(1, np.float32), k_norm_w=np.ones(1, np.float32), eps=0.0,
                    state_slot=np.array([0], np.int32),
                    conv_state_k=to_bits(np.ones((1, 3, 1))), conv_state_v=to_bits(np.ones((1, 3, 1))),
                    slot_mapping=np.arange(n, dtype=np.int32), block_size=4,
                    k_cache=np.zeros((1, 1, 4, 1), np.uint16), v_cache=np.zeros((1, 1, 4, 1), np.uint16))
        out = oracle_mod.prologue(**args, want_f64=True)
        assert np.array_equal(out["kc_f64"][:, 0], y)
        assert np.array_equal(from_bits(out["vc"][:, 0]), y)
        assert np.array_equal(from_bits(out["conv_state_k"][0, :, 0]), new_state)
        # V is not normalised: the cache holds the conv output itself
        assert np.array_equal(from_bits(out["v_cache"][0, 0, :n, 0]), y)


def test_shortconv_matches_numpy_correlate(oracle_mod):
    rng = np.random.default_rng(2)
    args = _prologue_case(rng, [7, 1, 12], prefix=[5, 0, 2])
    out = oracle_mod.prologue(**args, want_f64=True)
    cu = args["cu_seqlens_q"]
    for name, x, wk, st, key in (("k", args["k"], args["conv_w_k"], args["conv_state_k"], "kc_f64"),
                                  ("v", args["v"], args["conv_w_v"], args["conv_state_v"], "vc_f64")):
        for b in range(len(cu) - 1):
            xs = np.concatenate([from_bits(st[b]), from_bits(x[cu[b]:cu[b + 1]])], axis=0)
            for c in range(xs.shape[1]):
                ref = np.correlate(xs[:, c], wk[c].astype(np.float64), mode="valid")
                assert np.allclose(out[key][cu[b]:cu[b + 1], c], ref, rtol=0, atol=1e-12), (name, b, c)
    # rounded outputs are the nearest bf16 of the fp64 sums
    got = from_bits(out["kc"])
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(out["kc_f64"]), 1e-30))) - 7)
    assert np.all(np.abs(got - out["kc_f64"]) <= 0.5 * ulp + 1e-300)


def test_shortconv_delta_filter_is_identity(oracle_mod):
    rng = np.random.default_rng(3)
    C = 2 * 8
    w = np.zeros((C, 4), np.float32)
    w[:, 3] = 1.0
    args = _prologue_case(rng, [9, 2], prefix=[3, 1], w=w)
    out = oracle_mod.prologue(**args)
    assert np.array_equal(out["kc"], args["k"])
    assert np.array_equal(out["vc"], args["v"])


def test_shortconv_shift_filter_reads_state(oracle_mod):
    rng = np.random.default_rng(4)
    C = 2 * 8
    w = np.zeros((C, 4), np.float32)
    w[:, 0] = 1.0   # the token three back
    args = _prologue_case(rng, [6], w=w)
    out = oracle_mod.prologue(**args)
    expect = np.concatenate([args["conv_state_k"][0], args["k"][:3]], axis=0)
    assert np.array_equal(out["kc"], expect)
    # new state = last three inputs
    assert np.array_equal(out["conv_state_k"][0], args["k"][3:6])


def test_shortconv_state_carry_short_sequences(oracle_mod):
    rng = np.random.default_rng(5)
    args = _prologue_case(rng, [1, 2, 3, 0, 4])
    out = oracle_mod.prologue(**args)
    cu = args["cu_seqlens_q"]
    for b in range(5):
        xs = np.concatenate([args["conv_state_k"][b], args["k"][cu[b]:cu[b + 1]]], axis=0)
        assert np.array_equal(out["conv_state_k"][b], xs[-3:])


def test_shortconv_chunking_invariance(oracle_mod):
    """Splitting a sequence into chunks and carrying the state gives bit-identical
    outputs and final state."""
    rng = np.random.default_rng(6)
    full = _prologue_case(rng, [40])
    ref = oracle_mod.prologue(**full)
    state_k, state_v = full["conv_state_k"].copy(), full["conv_state_v"].copy()
    kcs, vcs = [], []
    for a, b in ((0, 1), (1, 3), (3, 20), (20, 40)):
        args = dict(full)
        args.update(cu_seqlens_q=np.array([0, b - a], np.int32), q=full["q"][a:b],
                    k=full["k"][a:b], v=full["v"][a:b], slot_mapping=full["slot_mapping"][a:b],
                    conv_state_k=state_k, conv_state_v=state_v)
        out = oracle_mod.prologue(**args)
        kcs.append(out["kc"]); vcs.append(out["vc"])
        state_k, state_v = out["conv_state_k"], out["conv_state_v"]
    assert np.array_equal(np.concatenate(kcs), ref["kc"])
    assert np.array_equal(np.concatenate(vcs), ref["vc"])
    assert np.array_equal(state_k, ref["conv_state_k"])
    assert np.array_equal(state_v, ref["conv_state_v"])


def test_rmsnorm_matches_torch_rms_norm(oracle_mod):
    rng = np.random.default_rng(7)
    d = 128
    gq = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    gk = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    args = _prologue_case(rng, [5, 3], Hq=4, Hkv=2, d=d, gq=gq, gk=gk, eps=1e-6)
    out = oracle_mod.prologue(**args)
    qf = torch.from_numpy(from_bits(args["q"]))
    ref_q = F.rms_norm(qf, (d,), weight=torch.from_numpy(gq.astype(np.float64)), eps=1e-6).numpy()
    got_q = from_bits(out["q_out"])
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref_q), 1e-30))) - 7)
    assert np.all(np.abs(got_q - ref_q) <= 0.5 * ulp * (1 + 1e-9))
    # K is normalised after the conv, from the bf16-rounded conv output
    kcf = torch.from_numpy(from_bits(out["kc"]).reshape(-1, 2, d))
    ref_k = F.rms_norm(kcf, (d,), weight=torch.from_numpy(gk.astype(np.float64)), eps=1e-6).numpy()
    slots = args["slot_mapping"]
    got_k = from_bits(out["k_cache"][slots // 4, :, slots % 4, :])
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref_k), 1e-30))) - 7)
    assert np.all(np.abs(got_k - ref_k) <= 0.5 * ulp * (1 + 1e-9))


def test_rmsnorm_unit_gain_unit_rms_and_scale_invariance(oracle_mod):
    rng = np.random.default_rng(8)
    d = 128
    args = _prologue_case(rng, [6], Hq=4, Hkv=2, d=d, eps=0.0)
    out = oracle_mod.prologue(**args)
    y = from_bits(out["q_out"])
    rms = np.sqrt((y ** 2).mean(axis=-1))
    assert np.allclose(rms, 1.0, atol=3e-3)
    args2 = dict(args)
    args2["q"] = to_bits(from_bits(args["q"]) * 8.0)   # exact in bf16
    out2 = oracle_mod.prologue(**args2)
    assert np.array_equal(out2["q_out"], out["q_out"])


def test_kv_write_touches_only_mapped_slots(oracle_mod):
    rng = np.random.default_rng(9)
    args = _prologue_case(rng, [5, 9], prefix=[2, 7])
    out = oracle_mod.prologue(**args)
    slots = args["slot_mapping"]
    mask = np.zeros(args["k_cache"].shape[0] * 4, bool)
    mask[slots] = True
    kc0 = args["k_cache"].transpose(0, 2, 1, 3).reshape(-1, 2, 8)
    kc1 = out["k_cache"].transpose(0, 2, 1, 3).reshape(-1, 2, 8)
    vc1 = out["v_cache"].transpose(0, 2, 1, 3).reshape(-1, 2, 8)
    assert np.array_equal(kc1[~mask], kc0[~mask])
    assert np.array_equal(vc1[slots].reshape(len(slots), -1), out["vc"])


# ---------------------------------------------------------------- attention

def _attn_case(rng, q_lens, prefix, Hq=4, Hkv=2, d=16, d_r=4, rel_extent=0, P=None, r=None,
               block_size=4, perm_seed=None):
    B = len(q_lens)
    T = [p + n for p, n in zip(prefix, q_lens)]
    kd = [to_bits(rng.standard_normal((t, Hkv, d))) for t in T]
    vd = [to_bits(rng.standard_normal((t, Hkv, d))) for t in T]
    kc, vc, table = paged_cache(kd, vd, block_size, Hkv, d, perm_seed=perm_seed, spare=1)
    N = sum(q_lens)
    q = to_bits(rng.standard_normal((N, Hq, d)))
    if r is None:
        r = to_bits(rng.standard_normal((N, Hq, d_r)))
    if P is None:
        P = (0.3 * rng.standard_normal((Hq, d_r, max(rel_extent, 1)))).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    # P is given as the matrices P_h [d_r][distance]; the oracle stores it distance-major
    return dict(cu_seqlens_q=cu, seqlen_k=np.array(T, np.int32), Hq=Hq, Hkv=Hkv, d=d, d_r=d_r,
                rel_extent=rel_extent, window=0, softmax_scale=0.0, log_scale_base=0.0, q=q, r=r,
                P=_stored(P), k_cache=kc, v_cache=vc, block_table=table, block_size=block_size), kd, vd


def _stored(P_math):
    """[Hq][d_r][rel_extent] (the matrices P_h) -> the [Hq][rel_extent][d_r] storage."""
    return np.ascontiguousarray(np.asarray(P_math, np.float32).transpose(0, 2, 1))


def _sdpa_rows(args, kd, vd, bias_fn=None, window=0, lam=1.0):
    """torch SDPA (fp64, math backend) on the dense K/V with an explicit mask; bias_fn(b, h, i, j)
    gives the additive bias before lambda (None = 0)."""
    cu, T = args["cu_seqlens_q"], args["seqlen_k"]
    Hq, Hkv, d = args["Hq"], args["Hkv"], args["d"]
    scale = lam / math.sqrt(d)
    outs = []
    for b in range(len(T)):
        n = cu[b + 1] - cu[b]
        qb = torch.from_numpy(from_bits(args["q"][cu[b]:cu[b + 1]])).permute(1, 0, 2)  # Hq n d
        kb = torch.from_numpy(from_bits(kd[b])).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        vb = torch.from_numpy(from_bits(vd[b])).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        i = torch.arange(T[b] - n, T[b]).view(-1, 1)
        j = torch.arange(T[b]).view(1, -1)
        vis = (j <= i)
        if window:
            vis &= (i - j) < window
        mask = torch.zeros(Hq, n, T[b], dtype=torch.float64)
        if bias_fn is not None:
            for h in range(Hq):
                mask[h] = lam * bias_fn(b, h, i, j)
        mask = mask.masked_fill(~vis, float("-inf"))
        o = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, scale=scale)
        outs.append(o.permute(1, 0, 2).numpy())
    return np.concatenate(outs, axis=0)


def test_attention_hand_golden(oracle_mod):
    with open(os.path.join(GOLDEN, "hand_attention.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    one = to_bits(np.ones((3, 1, 1)))
    zero = np.zeros((3, 1, 1))
    kc, vc, table = paged_cache([to_bits(zero)], [to_bits(np.array([1.0, 2, 4]).reshape(3, 1, 1))],
                                4, 1, 1)
    P = _stored(np.array([[[0.0, math.log(2.0)]]], np.float32))    # P_0 = [[0, ln 2]]
    for case in "ABC":
        sel = [r for r in rows if r[0] == case]
        window, base = int(sel[0][1]), float(sel[0][2])
        out, lse = oracle_mod.attention(cu_seqlens_q=np.array([0, 3], np.int32),
                                        seqlen_k=np.array([3], np.int32), Hq=1, Hkv=1, d=1, d_r=1,
                                        rel_extent=2, window=window, softmax_scale=1.0,
                                        log_scale_base=base, q=one, r=one, P=P, k_cache=kc,
                                        v_cache=vc, block_table=table, block_size=4)
        for r in sel:
            i = int(r[3])
            assert out[i, 0, 0] == pytest.approx(float(r[4]), abs=1e-6), (case, i)
            assert lse[i, 0] == pytest.approx(float(r[5]), abs=1e-6), (case, i)


def test_zero_bias_is_causal_sdpa_with_gqa_and_prefix(oracle_mod):
    rng = np.random.default_rng(10)
    args, kd, vd = _attn_case(rng, [5, 11, 1], [0, 6, 13], rel_extent=0, perm_seed=3)
    out, _ = oracle_mod.attention(**args)
    ref = _sdpa_rows(args, kd, vd)
    assert np.abs(out - ref).max() < 1e-12
    # P = 0 with a non-zero extent gives the same result
    args2 = dict(args, rel_extent=5, P=np.zeros((4, 5, 4), np.float32))
    out2, _ = oracle_mod.attention(**args2)
    assert np.abs(out2 - ref).max() < 1e-12


def test_sliding_window_edge_matches_sdpa(oracle_mod):
    rng = np.random.default_rng(11)
    args, kd, vd = _attn_case(rng, [13, 9], [0, 10])
    for window in (1, 3, 8):
        out, _ = oracle_mod.attention(**dict(args, window=window))
        ref = _sdpa_rows(args, kd, vd, window=window)
        assert np.abs(out - ref).max() < 1e-12, window


def test_window_at_least_T_equals_full(oracle_mod):
    rng = np.random.default_rng(12)
    args, _, _ = _attn_case(rng, [12, 7], [3, 0], rel_extent=6)
    full, lf = oracle_mod.attention(**args)
    wide, lw = oracle_mod.attention(**dict(args, window=15))
    assert np.array_equal(full, wide) and np.array_equal(lf, lw)


@pytest.mark.parametrize("k0", [0, 3])
def test_onehot_feature_bias_is_P_column_additive_mask(oracle_mod, k0):
    """r = e_k0 makes bias[h,i,j] = P[h,k0,i-j] for 0 <= i-j < rel_extent: torch SDPA with
    that additive mask (and lambda on both the scale and the mask) must agree."""
    rng = np.random.default_rng(13 + k0)
    Hq, d_r, E = 4, 4, 6
    q_lens, prefix = [7, 10], [0, 4]
    N = sum(q_lens)
    r = np.zeros((N, Hq, d_r), np.float32)
    r[:, :, k0] = 1.0
    P = (0.7 * rng.standard_normal((Hq, d_r, E))).astype(np.float32)
    args, kd, vd = _attn_case(rng, q_lens, prefix, Hq=Hq, d_r=d_r, rel_extent=E, P=P,
                              r=to_bits(r))

    def bias(b, h, i, j):
        dist = (i - j).numpy()
        val = np.where((dist >= 0) & (dist < E), P[h, k0, np.clip(dist, 0, E - 1)], 0.0)
        return torch.from_numpy(val.astype(np.float64))

    out, _ = oracle_mod.attention(**args)
    ref = _sdpa_rows(args, kd, vd, bias_fn=bias)
    assert np.abs(out - ref).max() < 1e-12
    base = 4.0   # lambda = ln T / ln 4 > 1 for both sequences (T = 7, 14)
    out_l, _ = oracle_mod.attention(**dict(args, log_scale_base=base))
    for b, T in enumerate(args["seqlen_k"]):
        lam = math.log(T) / math.log(base)
        ref_l = _sdpa_rows(args, kd, vd, bias_fn=bias, lam=lam)
        cu = args["cu_seqlens_q"]
        assert np.abs(out_l[cu[b]:cu[b + 1]] - ref_l[cu[b]:cu[b + 1]]).max() < 1e-12


def test_bias_depends_only_on_distance(oracle_mod):
    """The same tokens placed after a prefix of other keys give the same rows once the
    window hides that prefix: the bias is a function of i-j, not of i or j."""
    rng = np.random.default_rng(15)
    Hq, Hkv, d, d_r, E, W = 2, 1, 16, 4, 5, 6
    n, L = 14, 9
    kd = to_bits(rng.standard_normal((n, Hkv, d)))
    vd = to_bits(rng.standard_normal((n, Hkv, d)))
    junk_k = to_bits(rng.standard_normal((L, Hkv, d)))
    junk_v = to_bits(rng.standard_normal((L, Hkv, d)))
    q = to_bits(rng.standard_normal((n, Hq, d)))
    r = to_bits(rng.standard_normal((n, Hq, d_r)))
    P = (0.5 * rng.standard_normal((Hq, d_r, E))).astype(np.float32)
    kc_a, vc_a, tab_a = paged_cache([kd], [vd], 4, Hkv, d)
    kc_b, vc_b, tab_b = paged_cache([np.concatenate([junk_k, kd])], [np.concatenate([junk_v, vd])],
                                    4, Hkv, d, perm_seed=1)
    common = dict(Hq=Hq, Hkv=Hkv, d=d, d_r=d_r, rel_extent=E, window=W, softmax_scale=0.0,
                  log_scale_base=0.0, P=_stored(P), block_size=4)
    oa, la = oracle_mod.attention(cu_seqlens_q=np.array([0, n], np.int32),
                                  seqlen_k=np.array([n], np.int32), q=q, r=r, k_cache=kc_a,
                                  v_cache=vc_a, block_table=tab_a, **common)
    ob, lb = oracle_mod.attention(cu_seqlens_q=np.array([0, n], np.int32),
                                  seqlen_k=np.array([n + L], np.int32), q=q, r=r, k_cache=kc_b,
                                  v_cache=vc_b, block_table=tab_b, **common)
    assert np.abs(oa[W - 1:] - ob[W - 1:]).max() < 1e-13
    assert np.abs(la[W - 1:] - lb[W - 1:]).max() < 1e-13
    # and the rows that do see part of the prefix differ (the prefix is really there)
    assert np.abs(oa[:W - 1] - ob[:W - 1]).max() > 1e-3


def test_constant_P_is_a_row_shift(oracle_mod):
    """P[h,k,delta] = c[h,k] for every delta with rel_extent >= T adds the same bias to every
    visible key of a row: outputs equal the zero-bias ones and lse shifts by lambda*r.c."""
    rng = np.random.default_rng(16)
    Hq, d_r, T = 4, 4, 12
    c = rng.standard_normal((Hq, d_r)).astype(np.float32)
    P = np.repeat(c[:, :, None], T, axis=2).astype(np.float32)
    args, _, _ = _attn_case(rng, [T], [0], Hq=Hq, d_r=d_r, rel_extent=T, P=P)
    base = 3.0
    o1, l1 = oracle_mod.attention(**dict(args, log_scale_base=base))
    o0, l0 = oracle_mod.attention(**dict(args, rel_extent=0, log_scale_base=base))
    assert np.abs(o1 - o0).max() < 1e-12
    lam = math.log(T) / math.log(base)
    shift = lam * np.einsum("nhk,hk->nh", from_bits(args["r"]), c.astype(np.float64))
    assert np.abs((l1 - l0) - shift).max() < 1e-11


def test_rel_extent_one_biases_only_the_diagonal(oracle_mod):
    rng = np.random.default_rng(17)
    args, kd, vd = _attn_case(rng, [9], [2], rel_extent=1)
    r = from_bits(args["r"])
    P = args["P"].transpose(0, 2, 1)          # back to P_h [d_r][distance]

    def bias(b, h, i, j):
        diag = r[:, h, :] @ P[h, :, 0].astype(np.float64)       # [n]
        return torch.from_numpy(np.where((i - j).numpy() == 0, diag[:, None], 0.0))

    out, _ = oracle_mod.attention(**args)
    ref = _sdpa_rows(args, kd, vd, bias_fn=bias)
    assert np.abs(out - ref).max() < 1e-12


def test_gqa_equals_replicated_heads(oracle_mod):
    rng = np.random.default_rng(18)
    Hq, Hkv, d = 4, 2, 16
    args, kd, vd = _attn_case(rng, [6, 5], [1, 8], Hq=Hq, Hkv=Hkv, d=d, rel_extent=4)
    out, lse = oracle_mod.attention(**args)
    kd2 = [np.repeat(k, Hq // Hkv, axis=1) for k in kd]
    vd2 = [np.repeat(v, Hq // Hkv, axis=1) for v in vd]
    kc, vc, table = paged_cache(kd2, vd2, 4, Hq, d)
    out2, lse2 = oracle_mod.attention(**dict(args, Hkv=Hq, k_cache=kc, v_cache=vc, block_table=table))
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_block_table_permutation_invariance(oracle_mod):
    rng = np.random.default_rng(19)
    args, kd, vd = _attn_case(rng, [10, 3], [7, 30], rel_extent=8)
    out, lse = oracle_mod.attention(**args)
    kc, vc, table = paged_cache(kd, vd, 4, 2, 16, perm_seed=42, spare=5)
    out2, lse2 = oracle_mod.attention(**dict(args, k_cache=kc, v_cache=vc, block_table=table))
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_decode_rows_equal_prefill_tail(oracle_mod):
    """Nine query tokens decoded against a cache of T-9 earlier keys equal the last nine
    rows of a prefill of all T tokens."""
    rng = np.random.default_rng(20)
    T = 30
    args, kd, vd = _attn_case(rng, [T], [0], rel_extent=7)
    full, lf = oracle_mod.attention(**dict(args, log_scale_base=5.0))
    dec = dict(args, cu_seqlens_q=np.array([0, 9], np.int32), q=args["q"][T - 9:],
               r=args["r"][T - 9:], log_scale_base=5.0)
    out, lse = oracle_mod.attention(**dec)
    assert np.array_equal(out, full[T - 9:]) and np.array_equal(lse, lf[T - 9:])


def test_row_subset_matches_all_rows(oracle_mod):
    rng = np.random.default_rng(21)
    args, _, _ = _attn_case(rng, [8, 6], [0, 3], rel_extent=3)
    out, lse = oracle_mod.attention(**args)
    rows = np.array([13, 0, 7, 8], np.int32)
    o2, l2 = oracle_mod.attention(**dict(args, rows=rows))
    assert np.array_equal(o2, out[rows]) and np.array_equal(l2, lse[rows])
