"""GPU parity of the E4M3 (FP8) KV cache: the prologue's quantised cache write, and the
decode and the prefill over such a cache.

Bars: the prologue's codes and row scales are bit-exact against the oracle's quantisation
of the very bf16 rows the bf16 prologue writes (the quantisation is an integer decision
taken in exact power-of-two arithmetic on both sides); its queries and conv state equal
the bf16 run's.  The decode reads code * scale exactly (f16 holds every such value of the
prologue's rows), so it is held to the bf16 path's bar against the oracle run on the
dequantised cache: max-abs <= 1e-2, mean-abs <= 1e-3, |dLSE| <= 2e-3.  The prefill expands
the blocks it reads into a bf16 copy (exact) and runs the bf16 prefill on it: the copy is
checked bit for bit, the outputs at the same bar."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 1e-2, 1e-3, 2e-3


@pytest.fixture(scope="module")
def env(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from relative_bias_hybrid_gb300 import build
    build.build()
    from relative_bias_hybrid_gb300 import inputs as gen
    import relative_bias_hybrid_gb300.inkattn as ia
    from relative_bias_hybrid_gb300.step import AttentionStep
    return gen, AttentionStep, oracle_mod, ia


def _dequant_bits(oracle, gen, codes, scales):
    """The cache the decode reads, as bf16 bits (code * scale is a bf16 value, exactly)."""
    vals = oracle.dequantize_e4m3(codes, scales)
    t = torch.from_numpy(vals).to(torch.bfloat16)
    assert np.array_equal(t.double().numpy(), vals, equal_nan=True)
    return gen.bits(t)


def _compare(out, lse, o_ref, lse_ref, what, lse_tol=LSE_ABS):
    err = np.abs(out - o_ref)
    assert np.isfinite(out).all(), what
    assert err.max() <= MAX_ABS, (what, err.max(), err.mean())
    assert err.mean() <= MEAN_ABS, (what, err.mean())
    d = np.abs(lse - lse_ref)
    assert (d <= lse_tol).all(), (what, d.max())


def _run(env, w, seed, splits=0):
    gen, AttentionStep, _, _ = env
    x = gen.make_inputs(w, seed=seed, device="cuda", kv_dtype="e4m3")
    x_before = {k: v.clone() for k, v in x.items()}
    step = AttentionStep(w, x, mode="decode", num_splits=splits, out_dtype=torch.float32)
    step.run()
    torch.cuda.synchronize()
    return x_before, x, step


def _check(env, w, x, step, lse_tol=LSE_ABS):
    gen, _, oracle, _ = env
    assert step.device_status() == 0
    kc = _dequant_bits(oracle, gen, x["k_cache"].cpu().numpy(), x["k_scale"].cpu().numpy())
    vc = _dequant_bits(oracle, gen, x["v_cache"].cpu().numpy(), x["v_scale"].cpu().numpy())
    xs = {k: x[k].cpu() for k in ("cu_seqlens_q", "seqlen_k", "r", "P", "block_table")}
    o_ref, lse_ref = oracle.attention_for_inputs(xs, w, gen.bits(step.q_out), kc, vc)
    _compare(step.out.float().cpu().numpy(), step.lse.cpu().numpy(), o_ref, lse_ref, w.name, lse_tol)


def test_prologue_writes_quantised_rows(env):
    gen, AttentionStep, oracle, _ = env
    w = gen.custom("pro8", Hq=16, Hkv=2, q_lens=[9, 40, 3, 1], prefix_lens=[100, 0, 1, 70], rel_extent=64)
    xb = gen.make_inputs(w, seed=3, device="cuda")
    x8 = gen.make_inputs(w, seed=3, device="cuda", kv_dtype="e4m3")
    before = {k: x8[k].clone() for k in ("k_cache", "v_cache", "k_scale", "v_scale")}
    sb, s8 = AttentionStep(w, xb, mode="prefill"), AttentionStep(w, x8, mode="decode")
    sb.run_prologue()
    s8.run_prologue()
    torch.cuda.synchronize()
    assert sb.device_status() == 0 and s8.device_status() == 0
    assert torch.equal(sb.q_out, s8.q_out)
    assert torch.equal(xb["conv_state_k"], x8["conv_state_k"]) and torch.equal(xb["conv_state_v"], x8["conv_state_v"])
    slots = x8["slot_mapping"].cpu().numpy().astype(np.int64)
    blk, off = slots // 64, slots % 64
    for name in ("k", "v"):
        rows = gen.bits(xb[f"{name}_cache"])[blk, :, off, :]                 # [N][Hkv][128] bf16
        codes, scales = oracle.quantize_rows_e4m3(rows)
        got = x8[f"{name}_cache"].cpu().numpy()
        gs = x8[f"{name}_scale"].cpu().numpy()
        assert np.array_equal(got[blk, :, off, :], codes), name
        assert np.array_equal(gs[blk, :, off], scales), name
        # rows no token maps to are untouched
        keep = np.ones(got.shape[0] * 64, bool)
        keep[slots] = False
        g0 = got.transpose(0, 2, 1, 3).reshape(-1, w.Hkv, 128)
        b0 = before[f"{name}_cache"].cpu().numpy().transpose(0, 2, 1, 3).reshape(-1, w.Hkv, 128)
        assert np.array_equal(g0[keep], b0[keep])
        s0 = gs.transpose(0, 2, 1).reshape(-1, w.Hkv)
        sb0 = before[f"{name}_scale"].cpu().numpy().transpose(0, 2, 1).reshape(-1, w.Hkv)
        assert np.array_equal(s0[keep], sb0[keep])


@pytest.mark.parametrize("splits", [1, 0, 3])
def test_decode_e4m3_small(env, splits):
    gen = env[0]
    w = gen.custom("dec8", Hq=16, Hkv=2, q_lens=[9, 9, 4, 1], prefix_lens=[700, 40, 1500, 3000],
                   rel_extent=200, log_scale_base=256.0)
    x_before, x, step = _run(env, w, seed=4, splits=splits)
    _check(env, w, x, step)


def test_decode_e4m3_at_the_row_limit_with_window(env):
    gen = env[0]
    w = gen.custom("dec8-rows", Hq=32, Hkv=2, q_lens=[8, 8], prefix_lens=[1000, 2989], rel_extent=300,
                   window=1024)
    _check(env, w, *_run(env, w, seed=8, splits=3)[1:])


def test_decode_e4m3_strong_bias_mtp_shape(env):
    """The MTP-verify shape on three sequences with P ~ N(0, 0.5); the LSE bar adds the
    bound of the bias tables' fp16 rounding of P, as for the bf16 cache."""
    gen = env[0]
    from test_gpu_attention import _decode_table_lse_bound
    w = gen.custom("dec8-strong", Hq=64, Hkv=8, q_lens=[9, 9, 9], prefix_lens=[32759] * 3, rel_extent=1024,
                   log_scale_base=8192.0, p_std=0.5)
    x_before, x, step = _run(env, w, seed=19)
    xc = {k: x_before[k].cpu() for k in ("r", "P", "cu_seqlens_q")}
    _check(env, w, x, step, lse_tol=LSE_ABS + _decode_table_lse_bound(w, xc))


def test_decode_e4m3_full_size_sampled(env):
    """The MTP-verify workload with an E4M3 cache (32 x 9 queries, 32768 keys each), in the
    launch configuration the bench times: three sequences against the oracle."""
    gen, AttentionStep, oracle, _ = env
    w = gen.workload("decode")
    x_before, x, step = _run(env, w, seed=2)
    assert step.device_status() == 0
    seqs = [0, 17, 31]
    bt = x["block_table"].cpu().numpy()
    sk = x["seqlen_k"].cpu().numpy()
    blocks = np.concatenate([bt[b, :(sk[b] + 63) // 64] for b in seqs]).astype(np.int64)
    idx = torch.as_tensor(blocks, device="cuda")
    kc = _dequant_bits(oracle, gen, x["k_cache"].index_select(0, idx).cpu().numpy(),
                       x["k_scale"].index_select(0, idx).cpu().numpy())
    vc = _dequant_bits(oracle, gen, x["v_cache"].index_select(0, idx).cpu().numpy(),
                       x["v_scale"].index_select(0, idx).cpu().numpy())
    table = np.full((3, bt.shape[1]), -1, np.int32)
    pos = 0
    for i, b in enumerate(seqs):
        n = (sk[b] + 63) // 64
        table[i, :n] = np.arange(pos, pos + n)
        pos += n
    rows = np.concatenate([np.arange(b * 9, b * 9 + 9) for b in seqs])
    ridx = torch.as_tensor(rows.astype(np.int64), device="cuda")
    sub = gen.custom("dec8-3", Hq=64, Hkv=8, q_lens=[9] * 3, prefix_lens=[32759] * 3, rel_extent=1024,
                     log_scale_base=8192.0)
    xs = {"cu_seqlens_q": torch.tensor([0, 9, 18, 27], dtype=torch.int32),
          "seqlen_k": torch.tensor([32768] * 3, dtype=torch.int32),
          "r": x["r"].index_select(0, ridx).cpu(), "P": x["P"].cpu(), "block_table": torch.from_numpy(table)}
    o_ref, lse_ref = oracle.attention_for_inputs(xs, sub, gen.bits(step.q_out)[rows], kc, vc)
    _compare(step.out.index_select(0, ridx).float().cpu().numpy(), step.lse.index_select(0, ridx).cpu().numpy(),
             o_ref, lse_ref, "decode e4m3")


def test_decode_e4m3_bad_scale_is_flagged(env):
    gen, AttentionStep, _, ia = env
    w = gen.custom("dec8-bad", Hq=16, Hkv=2, q_lens=[9], prefix_lens=[500], rel_extent=64)
    x = gen.make_inputs(w, seed=5, device="cuda", kv_dtype="e4m3")
    blk = int(x["block_table"][0, 2].item())
    x["k_scale"][blk, 1, 7] = 1e30                 # a row inside the sequence
    step = AttentionStep(w, x, mode="decode", num_splits=1, out_dtype=torch.float32)
    step.run()
    torch.cuda.synchronize()
    assert step.device_status() == ia.INKATTN_ERR_DEVICE_BOUNDS
    assert torch.isfinite(step.out).all()


def test_nan_codes_past_sequence_end_are_ignored(env):
    """NaN codes and scales in every cache row past a sequence's end inside its last block:
    those rows are read as zeros and masked, and no bounds error is flagged."""
    gen, AttentionStep, _, _ = env
    w = gen.custom("dec8-nan", Hq=16, Hkv=2, q_lens=[9, 4], prefix_lens=[291, 1000], rel_extent=100)
    x = gen.make_inputs(w, seed=7, device="cuda", kv_dtype="e4m3")
    bt = x["block_table"].cpu().numpy()
    for b, T in enumerate(w.seqlen_k):
        if T % 64:
            last = int(bt[b, (T - 1) // 64])
            for name in ("k", "v"):
                x[f"{name}_cache"][last, :, T % 64:, :] = 0x7F
                x[f"{name}_scale"][last, :, T % 64:] = float("nan")
    step = AttentionStep(w, x, mode="decode", num_splits=1, out_dtype=torch.float32)
    step.run()
    torch.cuda.synchronize()
    assert step.device_status() == 0
    _check(env, w, x, step)


def test_decode_e4m3_noalloc_is_bit_identical(env):
    gen, AttentionStep, _, ia = env
    w = gen.custom("dec8-na", Hq=16, Hkv=2, q_lens=[9, 9], prefix_lens=[2000, 700], rel_extent=128)
    x = gen.make_inputs(w, seed=9, device="cuda", kv_dtype="e4m3")
    step = AttentionStep(w, x, mode="decode", num_splits=3, out_dtype=torch.float32)
    step.run()
    torch.cuda.synchronize()
    ref = step.out.clone()
    step.out.zero_()
    ia.inkattn_decode_noalloc(step.attn, 3)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    assert torch.equal(step.out, ref)


# ---------------------------------------------------------------- prefill over an E4M3 cache

def _prefill_e4m3(env, w, seed):
    gen, AttentionStep, _, _ = env
    x = gen.make_inputs(w, seed=seed, device="cuda", kv_dtype="e4m3")
    step = AttentionStep(w, x, mode="prefill", out_dtype=torch.float32)
    step.run()
    torch.cuda.synchronize()
    return x, step


def _check_prefill_rows(env, w, x, step, rows=None, lse_tol=LSE_ABS):
    """The prefill's rows against the oracle on the dequantised cache (after the prologue
    wrote the new tokens' rows), at the bf16 bars."""
    gen, _, oracle, _ = env
    assert step.device_status() == 0
    kc = _dequant_bits(oracle, gen, x["k_cache"].cpu().numpy(), x["k_scale"].cpu().numpy())
    vc = _dequant_bits(oracle, gen, x["v_cache"].cpu().numpy(), x["v_scale"].cpu().numpy())
    xs = {k: x[k].cpu() for k in ("cu_seqlens_q", "seqlen_k", "r", "P", "block_table")}
    o_ref, lse_ref = oracle.attention_for_inputs(xs, w, gen.bits(step.q_out), kc, vc, rows=rows)
    out, lse = step.out.float().cpu().numpy(), step.lse.cpu().numpy()
    if rows is not None:
        out, lse = out[rows], lse[rows]
    _compare(out, lse, o_ref, lse_ref, w.name, lse_tol)


@pytest.mark.parametrize("case", ["window_strong_bias", "full_lambda"])
def test_prefill_e4m3_small(env, case):
    """Prefill over an E4M3 cache: ragged sequences with prefixes, several band tiles, the
    strong bias (P ~ N(0, 0.5)) with a window, and a full layer with log scaling."""
    gen = env[0]
    if case == "window_strong_bias":
        w = gen.custom(case, Hq=8, Hkv=2, q_lens=[700, 130, 3], prefix_lens=[0, 200, 61], window=400,
                       rel_extent=600, p_std=0.5)
    else:
        w = gen.custom(case, Hq=16, Hkv=2, q_lens=[300, 260], prefix_lens=[900, 0], rel_extent=256,
                       log_scale_base=256.0)
    _check_prefill_rows(env, w, *_prefill_e4m3(env, w, seed=11))


def test_prefill_e4m3_copy_is_the_dequantised_cache(env):
    """The workspace copy: for each block a sequence reads, code * scale bit for bit (rows past
    the sequence's end zero), and the copy's block table (-1 past each sequence's blocks)."""
    gen, _, oracle, _ = env
    w = gen.custom("copy8", Hq=8, Hkv=2, q_lens=[70, 5], prefix_lens=[100, 250], rel_extent=64)
    x, step = _prefill_e4m3(env, w, seed=12)
    assert step.device_status() == 0
    mb = x["block_table"].shape[1]
    per = w.B * mb * w.Hkv * 64 * 128 * 2
    ws = step.workspace
    pad = (per + 255) // 256 * 256
    k16 = gen.bits(ws[:per].view(torch.bfloat16)).reshape(w.B * mb, w.Hkv, 64, 128)
    v16 = gen.bits(ws[pad:pad + per].view(torch.bfloat16)).reshape(w.B * mb, w.Hkv, 64, 128)
    table = ws[2 * pad:2 * pad + w.B * mb * 4].view(torch.int32).cpu().numpy().reshape(w.B, mb)
    bt = x["block_table"].cpu().numpy()
    for b, T in enumerate(w.seqlen_k):
        n = (T + 63) // 64
        assert np.array_equal(table[b, :n], b * mb + np.arange(n))
        assert (table[b, n:] == -1).all()
        for j in range(n):
            phys = int(bt[b, j])
            rows = min(64, T - 64 * j)
            for got, name in ((k16, "k"), (v16, "v")):
                want = oracle.dequantize_e4m3(x[f"{name}_cache"][phys].cpu().numpy(),
                                              x[f"{name}_scale"][phys].cpu().numpy())
                g = got[b * mb + j]
                assert np.array_equal(g[:, :rows].view(np.uint16), gen.bits(torch.from_numpy(want[:, :rows]).to(torch.bfloat16))), (b, j, name)
                assert not g[:, rows:].any(), (b, j, name)


def test_prefill_e4m3_full_layer_sampled(env):
    """The full layer (32768 tokens, rel_extent 1024, log scaling) over an E4M3 cache, in the
    launch configuration the bench times, on one row of every 128-row tile and the edges."""
    gen = env[0]
    from test_gpu_attention import _one_row_per_tile
    w = gen.workload("full")
    x, step = _prefill_e4m3(env, w, seed=13)
    _check_prefill_rows(env, w, x, step, rows=_one_row_per_tile(w))


def test_prefill_e4m3_bad_scale_is_flagged(env):
    gen, AttentionStep, _, ia = env
    w = gen.custom("pre8-bad", Hq=8, Hkv=2, q_lens=[100], prefix_lens=[200], rel_extent=64)
    x = gen.make_inputs(w, seed=14, device="cuda", kv_dtype="e4m3")
    blk = int(x["block_table"][0, 1].item())
    x["v_scale"][blk, 0, 5] = float("inf")          # a row the prologue does not rewrite
    step = AttentionStep(w, x, mode="prefill", out_dtype=torch.float32)
    step.run()
    torch.cuda.synchronize()
    assert step.device_status() == ia.INKATTN_ERR_DEVICE_BOUNDS
    assert torch.isfinite(step.out).all()
