"""GPU parity of inkattn_qkvr_prologue (the qkvr projections with the prologue fused into
their epilogue) against the fp64 oracle.

Bars.
- Integer-grid inputs (make_qkvr_inputs(grid=True)): every projection sum is exact in
  fp32 whatever the order of accumulation, so the GPU's projections must equal the
  oracle's correctly rounded ones bit for bit.  Then y (the projections), r, the new conv
  state and the V cache rows are bit-exact (the conv is correctly rounded), q_out and the
  K cache rows within 1 bf16 ulp (RMSNorm in fp32), as for inkattn_prologue.
- Gaussian inputs: each projection is the bf16 rounding (to nearest) of some value within
  delta of the exact sum, delta = 6 sqrt(K) 2^-23 sum_k |x_k w_k|: the probabilistic bound
  on the error of a K-term fp32 sum (Higham and Mary, 2019, lambda = 6) taken with the unit
  roundoff of truncation, 2^-23, so that it holds for either rounding of the partial sums.
  Where the exact sum is far from a bf16 rounding boundary that leaves one value: the
  oracle's.  The prologue's outputs
  are then held to inkattn_prologue's bars against the oracle prologue run on the GPU's
  own projections.
"""
import numpy as np
import pytest
import torch

from helpers import bf16_ulp_diff

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from relative_bias_hybrid_gb300 import build
    build.build()
    from relative_bias_hybrid_gb300 import inputs as gen
    import relative_bias_hybrid_gb300.inkattn as ia
    from relative_bias_hybrid_gb300.step import QkvrStep
    return gen, QkvrStep, oracle_mod, ia


def _run(env, w, d_model, seed=0, grid=True, want_y=True, in_place=False, kv_dtype="bf16"):
    gen, QkvrStep, _, _ = env
    x_cpu = gen.make_qkvr_inputs(w, d_model, seed=seed, device="cpu", grid=grid, kv_dtype=kv_dtype)
    x = {k: v.cuda() for k, v in x_cpu.items()}
    step = QkvrStep(w, x, in_place=in_place, want_y=want_y)
    step.run()
    torch.cuda.synchronize()
    return x_cpu, x, step


def _check_prologue_outputs(env, w, x_cpu, x, step, ref, r_ref):
    """The prologue's outputs of one run against the oracle's dict `ref` (computed on the
    projections the GPU is held to) and r against r_ref."""
    gen, _, _, _ = env
    assert step.device_status() == 0
    assert bf16_ulp_diff(gen.bits(step.q_out), ref["q_out"]).max() <= 1.0
    assert np.array_equal(gen.bits(step.r_out), r_ref)
    assert np.array_equal(gen.bits(step.state_k), ref["conv_state_k"])
    assert np.array_equal(gen.bits(step.state_v), ref["conv_state_v"])
    slots = x_cpu["slot_mapping"].numpy().astype(np.int64)
    blk, off = slots // w.block_size, slots % w.block_size
    kg, vg = gen.bits(x["k_cache"]), gen.bits(x["v_cache"])
    assert bf16_ulp_diff(kg[blk, :, off, :], ref["k_cache"][blk, :, off, :]).max() <= 1.0
    assert np.array_equal(vg[blk, :, off, :], ref["v_cache"][blk, :, off, :])
    untouched = np.ones(kg.shape[0] * w.block_size, bool)
    untouched[slots] = False
    for got, before in ((kg, x_cpu["k_cache"]), (vg, x_cpu["v_cache"])):
        g0 = got.transpose(0, 2, 1, 3).reshape(-1, w.Hkv, w.head_dim)
        b0 = gen.bits(before).transpose(0, 2, 1, 3).reshape(-1, w.Hkv, w.head_dim)
        assert np.array_equal(g0[untouched], b0[untouched])


def _grid_check(env, w, x_cpu, x, step):
    _, _, oracle, _ = env
    ref = oracle.qkvr_prologue_for_inputs(x_cpu, w)
    if step.y_out is not None:
        gen = env[0]
        N = w.N_tok
        y_ref = np.concatenate([ref["q_proj"].reshape(N, -1), ref["k_proj"], ref["v_proj"],
                                ref["r"].reshape(N, -1)], axis=1)
        assert np.array_equal(gen.bits(step.y_out), y_ref)
    _check_prologue_outputs(env, w, x_cpu, x, step, ref, ref["r"])


def _projection_misses(oracle, y_bits, x_bits, w_bits):
    """Indices where y is not the bf16 rounding of a value within delta of the exact
    x . w^T (see the module docstring), for y_bits [n][F] of the rows x_bits [n][K]; also the
    fraction of values that differ from the exactly rounded sum and the largest
    |y - exact| / sum |x w| seen."""
    xf = oracle.bf16_bits_to_f64(x_bits)
    wf = oracle.bf16_bits_to_f64(w_bits)
    exact = xf @ wf.T
    mag = np.abs(xf) @ np.abs(wf).T
    delta = 6.0 * np.sqrt(xf.shape[1]) * 2.0 ** -23 * mag
    # rounding to nearest is monotonic: the roundings of every value in
    # [exact - delta, exact + delta] lie between those of the two ends
    lo = oracle.bf16_bits_to_f64(oracle.round_bf16(exact - delta))
    hi = oracle.bf16_bits_to_f64(oracle.round_bf16(exact + delta))
    y = oracle.bf16_bits_to_f64(y_bits)
    ok = (y >= lo) & (y <= hi)
    mismatch = float((y_bits != oracle.round_bf16(exact)).mean())
    rel = float((np.abs(y - exact) / np.maximum(mag, 1e-300)).max())
    return np.argwhere(~ok), mismatch, rel


@pytest.mark.parametrize("d_model", [512, 200])
def test_grid_ragged_batch(env, d_model):
    """Sequences of 300, 1, 2, 0, 126, 125, 40 and 250 tokens with carried states of every
    length: 11 tiles (an odd count, so one CTA of the last pair has no tile), tiles ending
    at and one past the 125-token boundary, an empty sequence whose state is copied, and
    d_model = 200 with a K tail inside the last 64-column box."""
    gen = env[0]
    w = gen.custom("qkvr-mix", Hq=16, Hkv=2, q_lens=[300, 1, 2, 0, 126, 125, 40, 250],
                   prefix_lens=[0, 5, 1, 7, 2, 100, 0, 3], rel_extent=16)
    _grid_check(env, w, *_run(env, w, d_model, seed=1))


def test_grid_partial_feature_block(env):
    """Hq = 8, Hkv = 1, d_r = 8: F = 1344 features, so the last 256-feature block holds
    64 features of r and 192 past the end; one KV head, so a k block and a v block share
    an item."""
    gen = env[0]
    w = gen.custom("qkvr-odd", Hq=8, Hkv=1, q_lens=[131, 7], prefix_lens=[2, 40], rel_extent=8, d_r=8)
    _grid_check(env, w, *_run(env, w, 256, seed=2))


def test_grid_in_place_state_single_tile(env):
    """Every sequence within one tile (MTP-verify shape): the state may be updated in place."""
    gen = env[0]
    w = gen.custom("qkvr-dec", Hq=16, Hkv=2, q_lens=[9, 9, 1, 125, 3], prefix_lens=[50, 2, 0, 9, 700],
                   rel_extent=16)
    x_cpu, x, step = _run(env, w, 384, seed=3, in_place=True)
    assert step.state_k.data_ptr() == x["conv_state_k"].data_ptr()
    _grid_check(env, w, x_cpu, x, step)


def test_gaussian_projections_and_prologue_on_them(env):
    gen, _, oracle, _ = env
    w = gen.custom("qkvr-g", Hq=16, Hkv=2, q_lens=[260, 5, 130], prefix_lens=[0, 1, 64], rel_extent=16)
    x_cpu, x, step = _run(env, w, 1024, seed=4, grid=False)
    assert step.device_status() == 0
    y = gen.bits(step.y_out)
    bad, mismatch, rel = _projection_misses(oracle, y, gen.bits(x_cpu["x"]), gen.bits(x_cpu["w_qkvr"]))
    assert bad.size == 0, (bad[:10], mismatch, rel)
    assert mismatch < 0.01, mismatch
    N, Qw, C = w.N_tok, w.Hq * w.head_dim, w.Hkv * w.head_dim
    ref = oracle.prologue(cu_seqlens_q=x_cpu["cu_seqlens_q"].numpy(), Hq=w.Hq, Hkv=w.Hkv, d=w.head_dim,
                          q=y[:, :Qw].reshape(N, w.Hq, w.head_dim), k=y[:, Qw:Qw + C], v=y[:, Qw + C:Qw + 2 * C],
                          conv_w_k=x_cpu["conv_w_k"].numpy(), conv_w_v=x_cpu["conv_w_v"].numpy(),
                          q_norm_w=x_cpu["q_norm_w"].numpy(), k_norm_w=x_cpu["k_norm_w"].numpy(), eps=w.eps,
                          state_slot=x_cpu["state_slot"].numpy(), conv_state_k=gen.bits(x_cpu["conv_state_k"]),
                          conv_state_v=gen.bits(x_cpu["conv_state_v"]), slot_mapping=x_cpu["slot_mapping"].numpy(),
                          block_size=w.block_size, k_cache=gen.bits(x_cpu["k_cache"]),
                          v_cache=gen.bits(x_cpu["v_cache"]))
    _check_prologue_outputs(env, w, x_cpu, x, step, ref, y[:, Qw + 2 * C:].reshape(N, w.Hq, w.d_r))


def test_e4m3_cache_rows_are_the_quantised_bf16_rows(env):
    gen, QkvrStep, oracle, _ = env
    w = gen.custom("qkvr-f8", Hq=16, Hkv=2, q_lens=[140, 9], prefix_lens=[0, 100], rel_extent=16)
    xb_cpu, xb, sb = _run(env, w, 256, seed=5, want_y=False)
    x8_cpu, x8, s8 = _run(env, w, 256, seed=5, want_y=False, kv_dtype="e4m3")
    assert sb.device_status() == 0 and s8.device_status() == 0
    assert torch.equal(sb.q_out, s8.q_out) and torch.equal(sb.r_out, s8.r_out)
    assert torch.equal(sb.state_k, s8.state_k) and torch.equal(sb.state_v, s8.state_v)
    slots = x8_cpu["slot_mapping"].numpy().astype(np.int64)
    blk, off = slots // 64, slots % 64
    for name in ("k", "v"):
        rows = gen.bits(xb[f"{name}_cache"])[blk, :, off, :]
        codes, scales = oracle.quantize_rows_e4m3(rows)
        assert np.array_equal(x8[f"{name}_cache"].cpu().numpy()[blk, :, off, :], codes), name
        assert np.array_equal(x8[f"{name}_scale"].cpu().numpy()[blk, :, off], scales), name


def test_bad_slot_is_flagged_and_the_rest_written(env):
    gen, QkvrStep, oracle, ia = env
    w = gen.custom("qkvr-bad", Hq=16, Hkv=2, q_lens=[40], prefix_lens=[0], rel_extent=16)
    x_cpu = gen.make_qkvr_inputs(w, 128, seed=6, grid=True)
    x = {k: v.cuda() for k, v in x_cpu.items()}
    x["slot_mapping"][17] = 1 << 30
    step = QkvrStep(w, x)
    step.run()
    torch.cuda.synchronize()
    assert step.device_status() == ia.INKATTN_ERR_DEVICE_BOUNDS
    ref = oracle.qkvr_prologue_for_inputs(x_cpu, w)
    assert bf16_ulp_diff(gen.bits(step.q_out), ref["q_out"]).max() <= 1.0
    assert np.array_equal(gen.bits(step.state_k), ref["conv_state_k"])


def _window_reference(oracle, gen, w, x_cpu, xb, wb, b, t_lo, t_hi):
    """Oracle outputs for tokens [t_lo, t_hi) of sequence b of a full-size workload: the
    projections of its x rows [t_lo - 3, t_hi), the first three standing in for the conv
    state when t_lo >= 3 (else the sequence's carried state), then the prologue."""
    d = w.head_dim
    s0 = int(x_cpu["cu_seqlens_q"][b])
    a = max(0, t_lo - 3)
    q, k, v, r = oracle.qkvr_projection(xb[s0 + a:s0 + t_hi], wb, Hq=w.Hq, Hkv=w.Hkv, d=d, d_r=w.d_r)
    h = t_lo - a
    slot = int(x_cpu["state_slot"][b])
    st_k = gen.bits(x_cpu["conv_state_k"])[slot:slot + 1].copy()
    st_v = gen.bits(x_cpu["conv_state_v"])[slot:slot + 1].copy()
    if t_lo >= 3:
        st_k[0], st_v[0] = k[:3], v[:3]
    n = t_hi - t_lo
    sm = x_cpu["slot_mapping"].numpy()[s0 + t_lo:s0 + t_hi]
    ref = oracle.prologue(cu_seqlens_q=np.array([0, n], np.int32), Hq=w.Hq, Hkv=w.Hkv, d=d, q=q[h:], k=k[h:],
                          v=v[h:], conv_w_k=x_cpu["conv_w_k"].numpy(), conv_w_v=x_cpu["conv_w_v"].numpy(),
                          q_norm_w=x_cpu["q_norm_w"].numpy(), k_norm_w=x_cpu["k_norm_w"].numpy(), eps=w.eps,
                          state_slot=np.array([0], np.int32), conv_state_k=st_k, conv_state_v=st_v,
                          slot_mapping=sm, block_size=w.block_size,
                          k_cache=np.zeros((w.num_blocks, w.Hkv, w.block_size, d), np.uint16),
                          v_cache=np.zeros((w.num_blocks, w.Hkv, w.block_size, d), np.uint16))
    return ref, r[h:], sm, slot


def _windows(w):
    """(sequence, first token, end) windows: a sequence's start (the carried state), the
    edges of its 125-token tiles, its middle and its end (the new state)."""
    out = []
    for b in ([0] if w.B == 1 else [0, w.B // 2, w.B - 1]):
        n = w.q_lens[b]
        out += [(b, lo, hi) for lo, hi in ((0, 6), (122, 130), (247, 253), (n // 2, n // 2 + 3), (n - 5, n))
                if 0 <= lo < hi <= n]
    return out


@pytest.mark.parametrize("name", ["swa", "full", "ragged"])
def test_full_size_layer_grid_sampled(env, name):
    """The prefill workloads at full size (d_model 8192, F 12288) in the launch configuration
    the bench times: token windows at a sequence's start, across tile edges, in the middle
    and at the end are checked against the oracle, and the new state against the
    projections of the last three tokens."""
    gen, _, oracle, _ = env
    w = gen.workload(name)
    x_cpu, x, step = _run(env, w, 8192, seed=7, want_y=False)
    assert step.device_status() == 0
    xb, wb = gen.bits(x_cpu["x"]), gen.bits(x_cpu["w_qkvr"])
    kg, vg = gen.bits(x["k_cache"]), gen.bits(x["v_cache"])
    q_out, r_out = gen.bits(step.q_out), gen.bits(step.r_out)
    state_k, state_v = gen.bits(step.state_k), gen.bits(step.state_v)
    for b, t_lo, t_hi in _windows(w):
        s0 = int(x_cpu["cu_seqlens_q"][b])
        ref, r_ref, sm, slot = _window_reference(oracle, gen, w, x_cpu, xb, wb, b, t_lo, t_hi)
        where = (name, b, t_lo, t_hi)
        assert bf16_ulp_diff(q_out[s0 + t_lo:s0 + t_hi], ref["q_out"]).max() <= 1.0, where
        assert np.array_equal(r_out[s0 + t_lo:s0 + t_hi], r_ref), where
        blk, off = sm // 64, sm % 64
        assert bf16_ulp_diff(kg[blk, :, off, :], ref["k_cache"][blk, :, off, :]).max() <= 1.0, where
        assert np.array_equal(vg[blk, :, off, :], ref["v_cache"][blk, :, off, :]), where
        if t_hi == w.q_lens[b]:
            assert np.array_equal(state_k[slot], ref["conv_state_k"][0]), where
            assert np.array_equal(state_v[slot], ref["conv_state_v"][0]), where


def test_full_size_gaussian_projections_sampled(env):
    """The K = 8192 projections of Gaussian inputs at full size, on sampled rows."""
    gen, _, oracle, _ = env
    w = gen.workload("swa")
    x_cpu, x, step = _run(env, w, 8192, seed=8, grid=False, want_y=True)
    assert step.device_status() == 0
    rows = np.array([0, 1, 2, 124, 125, 126, 3000, 8191])
    y = gen.bits(step.y_out)[rows]
    bad, mismatch, rel = _projection_misses(oracle, y, gen.bits(x_cpu["x"])[rows], gen.bits(x_cpu["w_qkvr"]))
    assert bad.size == 0, (bad[:10], mismatch, rel)
    assert mismatch < 0.02, mismatch
