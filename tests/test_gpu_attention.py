"""GPU parity of inkattn_prefill / inkattn_decode + inkattn_combine against the fp64
oracle, on the same bf16 queries and caches the GPU prologue produced (so the attention
error is isolated).  Bar: max-abs <= 1e-2 and mean-abs <= 1e-3 on the outputs, and
|lse - lse_ref| <= 2e-3.  Full-size workloads are checked on sampled rows (all heads),
chosen to include tile edges, window and rel_extent edges and sequence ends.

The bar is checked on fp32 outputs (out_dtype = f32): a bf16 output adds its own
rounding, up to half a bf16 ulp (0.0078 for |o| in [2, 4), 0.0156 above 4), which alone
can exceed 1e-2.  A separate test pins the bf16 output to the fp32 one rounded once."""
import numpy as np
import pytest
import torch

from helpers import compact_cache

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 1e-2, 1e-3, 2e-3


@pytest.fixture(scope="module")
def env(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from relative_bias_hybrid_gb300 import build
    build.build()
    from relative_bias_hybrid_gb300 import inputs as gen
    from relative_bias_hybrid_gb300.step import AttentionStep
    return gen, AttentionStep, oracle_mod


def _run(env, w, mode="prefill", seed=0, device_inputs=False, num_splits=0, out_dtype=torch.float32):
    gen, AttentionStep, _ = env
    if device_inputs:
        x = gen.make_inputs(w, seed=seed, device="cuda")
        x_cpu = None
    else:
        x_cpu = gen.make_inputs(w, seed=seed, device="cpu")
        x = {k: v.cuda() for k, v in x_cpu.items()}
    step = AttentionStep(w, x, mode=mode, num_splits=num_splits, out_dtype=out_dtype)
    step.run()
    torch.cuda.synchronize()
    assert step.device_status() == 0
    return x_cpu, x, step


def _compare(out, lse, o_ref, lse_ref, what, lse_tol=LSE_ABS):
    err = np.abs(out - o_ref)
    assert np.isfinite(out).all(), what
    where = np.unravel_index(int(np.argmax(err)), err.shape)
    assert err.max() <= MAX_ABS, (what, err.max(), "at", where, "ref", o_ref[where], "mean", err.mean())
    assert err.mean() <= MEAN_ABS, (what, err.mean())
    if lse is not None:
        d = np.abs(lse - lse_ref)
        assert (d <= lse_tol).all(), (what, d.max(), np.max(d - lse_tol))


def _check_all_rows(env, w, x_cpu, x, step, lse_tol=LSE_ABS):
    gen, _, oracle = env
    o_ref, lse_ref = oracle.attention_for_inputs(x_cpu, w, gen.bits(step.q_out), gen.bits(x["k_cache"]),
                                                 gen.bits(x["v_cache"]))
    _compare(step.out.float().cpu().numpy(), step.lse.cpu().numpy(), o_ref, lse_ref, w.name, lse_tol)


def _decode_table_lse_bound(w, x_cpu):
    """The decode's bias tables multiply r by P rounded to fp16 (11 significant bits, relative
    error <= 2^-11 per element), so a logit moves by at most lam * 2^-11 * sum_e |r_e P_e|, and
    the LSE by no more than the largest such move over the row's biased keys.  Per (row, head)."""
    r = np.abs(x_cpu["r"].float().numpy().astype(np.float64))          # [N][Hq][d_r]
    P = np.abs(x_cpu["P"].numpy().astype(np.float64))                  # [Hq][rel_extent][d_r]
    cu = x_cpu["cu_seqlens_q"].numpy()
    bound = np.zeros((w.N_tok, w.Hq))
    for b in range(w.B):
        T = w.seqlen_k[b]
        lam = max(1.0, np.log(T) / np.log(w.log_scale_base)) if w.log_scale_base > 1 else 1.0
        for t in range(cu[b], cu[b + 1]):
            i = w.prefix_lens[b] + t - cu[b]
            lim = min(w.rel_extent, i + 1)
            s = np.einsum("he,hde->hd", r[t], P[:, :lim])                # [Hq][distances]
            bound[t] = lam * 2.0 ** -11 * s.max(axis=1)
    return bound


def _sample_rows(w, extra=()):
    rows = set(extra)
    start = 0
    for b, n in enumerate(w.q_lens):
        pre = w.prefix_lens[b]
        for t in (0, 1, 63, 64, 127, 128, 129, n // 2, n - 129, n - 128, n - 2, n - 1):
            if 0 <= t < n:
                rows.add(start + t)
        for edge in (w.window, w.rel_extent):         # positions where a window / extent edge lands
            for dt in (-1, 0, 1):
                t = edge + dt - pre
                if edge and 0 <= t < n:
                    rows.add(start + t)
        start += n
    return np.array(sorted(rows), np.int32)


def _check_rows(env, w, x, step, rows):
    """Oracle on sampled rows; only the tensors the oracle needs are copied to the host."""
    gen, _, oracle = env
    x_cpu = {k: x[k].cpu() for k in ("cu_seqlens_q", "seqlen_k", "r", "P", "block_table")}
    o_ref, lse_ref = oracle.attention_for_inputs(x_cpu, w, gen.bits(step.q_out), gen.bits(x["k_cache"]),
                                                 gen.bits(x["v_cache"]), rows=rows)
    idx = torch.as_tensor(rows.astype(np.int64), device="cuda")
    out = step.out.index_select(0, idx).float().cpu().numpy()
    lse = step.lse.index_select(0, idx).cpu().numpy()
    _compare(out, lse, o_ref, lse_ref, w.name)


# ---------------------------------------------------------------- prefill

def test_prefill_tiny_all_rows(env):
    gen = env[0]
    w = gen.workload("tiny")
    _check_all_rows(env, w, *_run(env, w))


@pytest.mark.parametrize("case", ["swa_ragged", "full_logscale", "no_bias", "no_bias_window", "extent_past_T",
                                  "gqa4", "gqa3_unpaired", "mha", "empty_sequence"])
def test_prefill_small_mixed(env, case):
    gen = env[0]
    kw = dict(Hq=8, Hkv=2, q_lens=[200, 77, 300, 1], prefix_lens=[0, 150, 37, 9])
    if case == "swa_ragged":
        w = gen.custom(case, window=100, rel_extent=70, **kw)
    elif case == "full_logscale":
        w = gen.custom(case, window=0, rel_extent=130, log_scale_base=64.0, **kw)
    elif case == "no_bias":
        w = gen.custom(case, window=0, rel_extent=0, **kw)
    elif case == "no_bias_window":
        # two query tiles per CTA with different key ranges at both window edges
        w = gen.custom(case, Hq=8, Hkv=2, q_lens=[700, 129, 256], prefix_lens=[30, 0, 500], window=200,
                       rel_extent=0)
    elif case == "extent_past_T":
        w = gen.custom(case, window=0, rel_extent=600, **kw)
    elif case == "gqa4":
        w = gen.custom(case, Hq=16, Hkv=4, q_lens=[257, 129], prefix_lens=[64, 0], window=192,
                       rel_extent=96, d_r=32)
    elif case == "gqa3_unpaired":
        # odd group size: head pairs do not share a KV head, so no CTA pairing
        w = gen.custom(case, Hq=6, Hkv=2, q_lens=[300, 45], prefix_lens=[20, 0], window=0,
                       rel_extent=200)
    elif case == "mha":
        w = gen.custom(case, Hq=3, Hkv=3, q_lens=[190, 260], prefix_lens=[0, 70], window=128,
                       rel_extent=50)
    else:
        # a sequence with no new tokens between two others (its cached prefix stays unread)
        w = gen.custom(case, Hq=8, Hkv=2, q_lens=[130, 0, 129], prefix_lens=[5, 64, 0],
                       window=0, rel_extent=100)
    _check_all_rows(env, w, *_run(env, w, seed=11))


def _one_row_per_tile(w, seed=5):
    """One row in every 128-row query tile of every sequence (at a seeded offset within the
    tile), plus the edges of _sample_rows."""
    rng = np.random.default_rng(seed)
    rows = set(_sample_rows(w).tolist())
    start = 0
    for n in w.q_lens:
        for t0 in range(0, n, 128):
            rows.add(start + t0 + int(rng.integers(0, min(128, n - t0))))
        start += n
    return np.array(sorted(rows), np.int32)


@pytest.mark.parametrize("name", ["swa", "full", "ragged", "full_nobias"])
def test_prefill_full_size_sampled(env, name):
    import dataclasses
    gen = env[0]
    w = gen.workload(name.replace("_nobias", ""))
    if name.endswith("_nobias"):
        w = dataclasses.replace(w, name=name, rel_extent=0)
    _, x, step = _run(env, w, device_inputs=True, seed=1)
    rows = _one_row_per_tile(w) if name.startswith("full") else _sample_rows(w)
    _check_rows(env, w, x, step, rows)


@pytest.mark.parametrize("case", ["swa_window", "full_lambda", "gqa3_unpaired_lambda"])
def test_prefill_strong_bias(env, case):
    """P ~ N(0, 0.5): the bias (std ~2.8 logits) outweighs q.k / sqrt(d) (std ~1), so an
    error in the band (a wrong shear, distance, extent edge or precision) moves the output
    well past the bar on every row.  Every case spans five or more band tiles."""
    gen = env[0]
    if case == "swa_window":
        w = gen.custom(case, Hq=8, Hkv=2, q_lens=[700, 530], prefix_lens=[0, 200], window=400,
                       rel_extent=600, p_std=0.5)
    elif case == "full_lambda":
        w = gen.custom(case, Hq=8, Hkv=2, q_lens=[900, 300], prefix_lens=[0, 650], window=0,
                       rel_extent=700, log_scale_base=128.0, p_std=0.5)
    else:
        w = gen.custom(case, Hq=6, Hkv=2, q_lens=[640], prefix_lens=[100], window=0, rel_extent=640,
                       log_scale_base=64.0, p_std=0.5)
    _check_all_rows(env, w, *_run(env, w, seed=17))


# ---------------------------------------------------------------- decode

@pytest.mark.parametrize("splits", [1, 0, 2, 3, 7])
def test_decode_small(env, splits):
    gen = env[0]
    w = gen.custom("dec", Hq=16, Hkv=2, q_lens=[9, 9, 4, 1], prefix_lens=[700, 40, 1500, 3000],
                   rel_extent=200, log_scale_base=256.0)
    _check_all_rows(env, w, *_run(env, w, mode="decode", seed=4, num_splits=splits))


@pytest.mark.parametrize("Hq,Hkv,ql", [(32, 2, 8), (16, 2, 16)])
def test_decode_at_the_row_limit(env, Hq, Hkv, ql):
    """(token, query head) rows of a KV head at their limit of 128 (the MMA's M, every TMEM
    lane and every bias-table row in use), with uneven prefixes and 3 splits."""
    gen = env[0]
    w = gen.custom("dec-rows", Hq=Hq, Hkv=Hkv, q_lens=[ql, ql], prefix_lens=[1000, 2989], rel_extent=300,
                   log_scale_base=256.0)
    assert (Hq // Hkv) * ql == 128
    _check_all_rows(env, w, *_run(env, w, mode="decode", seed=8, num_splits=3))


def test_decode_sliding_window(env):
    gen = env[0]
    w = gen.custom("dec-swa", Hq=64, Hkv=8, q_lens=[9, 9], prefix_lens=[5000, 300], rel_extent=512,
                   window=1024)
    _check_all_rows(env, w, *_run(env, w, mode="decode", seed=6, num_splits=4))


@pytest.mark.parametrize("splits", [0, 1, 2])
def test_decode_strong_bias_mtp_shape(env, splits):
    """The MTP-verify shape (9 queries, key length 32768, Hq 64, Hkv 8, rel_extent 1024,
    lambda = 15/13) on three sequences with P ~ N(0, 0.5): the bias tables decide the output.
    The outputs are held to the bar; the LSE to the bar plus the bound of the tables' fp16
    rounding of P (see _decode_table_lse_bound)."""
    gen = env[0]
    w = gen.custom("dec-strong", Hq=64, Hkv=8, q_lens=[9, 9, 9], prefix_lens=[32759] * 3, rel_extent=1024,
                   log_scale_base=8192.0, p_std=0.5)
    x_cpu, x, step = _run(env, w, mode="decode", seed=19, num_splits=splits)
    if splits == 0:
        assert step.num_splits > 1          # three sequences: the heuristic splits the keys
    _check_all_rows(env, w, x_cpu, x, step, lse_tol=LSE_ABS + _decode_table_lse_bound(w, x_cpu))


def test_decode_full_size_sampled(env):
    """The MTP-verify workload (32 x 9 queries, KV 32768): three sequences against the
    oracle; all sequences agree between the heuristic's split count and another one (4
    splits and the combine when the heuristic streams each sequence whole)."""
    gen, AttentionStep, oracle = env
    w = gen.workload("decode")
    x = gen.make_inputs(w, seed=2, device="cuda")
    snap = {k: x[k].clone() for k in ("k_cache", "v_cache", "conv_state_k", "conv_state_v")}
    step = AttentionStep(w, x, mode="decode", out_dtype=torch.float32)
    other = 4 if step.num_splits == 1 else 1
    step.run()
    torch.cuda.synchronize()
    assert step.device_status() == 0
    seqs = [0, 17, 31]
    bt = x["block_table"].cpu().numpy()
    sk = x["seqlen_k"].cpu().numpy()
    blocks = np.concatenate([bt[b, :(sk[b] + 63) // 64] for b in seqs])
    idx = torch.as_tensor(blocks.astype(np.int64), device="cuda")
    kc = gen.bits(x["k_cache"].index_select(0, idx))
    vc = gen.bits(x["v_cache"].index_select(0, idx))
    table = np.full((3, bt.shape[1]), -1, np.int32)
    pos = 0
    for i, b in enumerate(seqs):
        n = (sk[b] + 63) // 64
        table[i, :n] = np.arange(pos, pos + n)
        pos += n
    rows = np.concatenate([np.arange(b * 9, b * 9 + 9) for b in seqs])
    q = gen.bits(step.q_out)[rows]
    sub = gen.custom("dec3", Hq=64, Hkv=8, q_lens=[9] * 3, prefix_lens=[32759] * 3, rel_extent=1024,
                     log_scale_base=8192.0)
    xs = {"cu_seqlens_q": torch.tensor([0, 9, 18, 27], dtype=torch.int32),
          "seqlen_k": torch.tensor([32768] * 3, dtype=torch.int32),
          "r": x["r"][torch.as_tensor(rows.astype(np.int64), device="cuda")].cpu(),
          "P": x["P"].cpu(), "block_table": torch.from_numpy(table)}
    o_ref, lse_ref = oracle.attention_for_inputs(xs, sub, q, kc, vc)
    ridx = torch.as_tensor(rows.astype(np.int64), device="cuda")
    _compare(step.out.index_select(0, ridx).float().cpu().numpy(),
             step.lse.index_select(0, ridx).cpu().numpy(), o_ref, lse_ref, "decode")
    # same caches and conv state, another split count: every sequence agrees
    out_h = step.out.float().clone()
    for k, v in snap.items():
        x[k].copy_(v)
    one = AttentionStep(w, x, mode="decode", num_splits=other, out_dtype=torch.float32)
    one.run()
    torch.cuda.synchronize()
    diff = (one.out.float() - out_h).abs()
    assert diff.max().item() <= MAX_ABS and diff.mean().item() <= MEAN_ABS


def test_decode_equals_prefill_tail(env):
    """Decoding the last 9 tokens against the cache equals the last 9 rows of a prefill."""
    gen, AttentionStep, _ = env
    T = 1000
    wp = gen.custom("pre", Hq=16, Hkv=2, q_lens=[T], prefix_lens=[0], rel_extent=300,
                    log_scale_base=128.0)
    x_cpu = gen.make_inputs(wp, seed=12, device="cpu")
    x = {k: v.cuda() for k, v in x_cpu.items()}
    pre = AttentionStep(wp, x, mode="prefill", out_dtype=torch.float32)
    pre.run()
    wd = gen.custom("dec", Hq=16, Hkv=2, q_lens=[9], prefix_lens=[T - 9], rel_extent=300,
                    log_scale_base=128.0)
    xd = dict(x)
    xd["r"] = x["r"][T - 9:].contiguous()
    xd["cu_seqlens_q"] = torch.tensor([0, 9], dtype=torch.int32, device="cuda")
    dec_q = pre.q_out[T - 9:].contiguous()
    import relative_bias_hybrid_gb300.inkattn as ia
    out = torch.empty(dec_q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(dec_q.shape[:2], dtype=torch.float32, device="cuda")
    p = ia.attn_params(q=dec_q, k_cache=x["k_cache"], v_cache=x["v_cache"], cu_seqlens_q=xd["cu_seqlens_q"],
                       seqlen_k=x["seqlen_k"], block_table=x["block_table"], out=out, max_seqlen_q=9,
                       max_seqlen_k=T, r=xd["r"], P=x["P"], rel_extent=300, log_scale_base=128.0, lse=lse)
    for S in (1, 4):
        nb = ia.inkattn_decode_workspace_bytes(p, S)
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
        ia.inkattn_decode(p, S, ws)
        ia.inkattn_combine(p, S, ws)
        torch.cuda.synchronize()
        assert (out.float() - pre.out[T - 9:].float()).abs().max().item() <= 1e-2
        assert (lse - pre.lse[T - 9:]).abs().max().item() <= 2e-3


def test_bad_block_id_is_flagged(env):
    gen, AttentionStep, _ = env
    w = gen.custom("badblk", Hq=8, Hkv=2, q_lens=[100], prefix_lens=[50], rel_extent=20)
    x_cpu = gen.make_inputs(w, seed=13, device="cpu")
    x_cpu["block_table"][0, 1] = 10 ** 6
    x = {k: v.cuda() for k, v in x_cpu.items()}
    step = AttentionStep(w, x, mode="prefill")
    step.run()
    torch.cuda.synchronize()
    assert step.device_status() == 5


def test_malformed_batch_is_flagged_by_the_prefill(env):
    # in a batch of several sequences, one whose cu_seqlens_q entries run backwards (and the
    # next, which then has more rows than keys) is flagged and skipped; the others are still
    # computed
    gen, AttentionStep, oracle = env
    w = gen.custom("badcu", Hq=8, Hkv=2, q_lens=[600, 60, 140], prefix_lens=[0, 30, 0], rel_extent=90)
    x_cpu = gen.make_inputs(w, seed=17, device="cpu")
    x = {k: v.cuda() for k, v in x_cpu.items()}
    step = AttentionStep(w, x, mode="prefill")
    step.run_prologue()
    torch.cuda.synchronize()
    assert step.device_status() == 0
    x["cu_seqlens_q"][2] = 550            # sequence 1: [600, 550); sequence 2: 250 rows, 140 keys
    step.run_attention()
    torch.cuda.synchronize()
    assert step.device_status() == 5
    # sequence 0 is intact
    rows = np.arange(0, 600, 7, dtype=np.int32)
    x_ref = {k: x_cpu[k] for k in ("seqlen_k", "r", "P", "block_table")}
    x_ref["cu_seqlens_q"] = x_cpu["cu_seqlens_q"]
    o_ref, lse_ref = oracle.attention_for_inputs(x_ref, w, gen.bits(step.q_out), gen.bits(x["k_cache"]),
                                                 gen.bits(x["v_cache"]), rows=rows)
    idx = torch.as_tensor(rows.astype(np.int64), device="cuda")
    _compare(step.out.index_select(0, idx).float().cpu().numpy(), step.lse.index_select(0, idx).cpu().numpy(),
             o_ref, lse_ref, w.name)


@pytest.mark.parametrize("mode,splits", [("prefill", 0), ("decode", 1), ("decode", 4)])
def test_bf16_output_is_the_fp32_output_rounded_once(env, mode, splits):
    gen, AttentionStep, _ = env
    import relative_bias_hybrid_gb300.inkattn as ia
    if mode == "prefill":
        w = gen.custom("rnd", Hq=8, Hkv=2, q_lens=[300, 129], prefix_lens=[0, 40], rel_extent=90,
                       window=200)
    else:
        w = gen.custom("rnd", Hq=16, Hkv=2, q_lens=[9, 7], prefix_lens=[900, 2000], rel_extent=300,
                       log_scale_base=512.0)
    x = gen.make_inputs(w, seed=14, device="cuda")
    step = AttentionStep(w, x, mode=mode, num_splits=splits, out_dtype=torch.float32)
    step.run_prologue()
    step.run_attention()
    out_bf = torch.empty(step.out.shape, dtype=torch.bfloat16, device="cuda")
    p = ia.attn_params(q=step.q_out, k_cache=x["k_cache"], v_cache=x["v_cache"],
                       cu_seqlens_q=x["cu_seqlens_q"], seqlen_k=x["seqlen_k"],
                       block_table=x["block_table"], out=out_bf, max_seqlen_q=max(w.q_lens),
                       max_seqlen_k=max(w.seqlen_k), r=x["r"], P=x["P"], rel_extent=w.rel_extent,
                       window=w.window, log_scale_base=w.log_scale_base)
    if mode == "prefill":
        ia.inkattn_prefill(p)
    else:
        ia.inkattn_decode(p, step.num_splits, step.workspace)
        ia.inkattn_combine(p, step.num_splits, step.workspace)
    torch.cuda.synchronize()
    assert torch.equal(out_bf.view(torch.int16), step.out.to(torch.bfloat16).view(torch.int16))


# ---------------------------------------------------------------- poisoned cache tails

def _poison_tails(x):
    """NaN into every K and V slot past a sequence's end inside its last cache block."""
    nan = torch.tensor(float("nan"), dtype=x["k_cache"].dtype, device=x["k_cache"].device)
    table = x["block_table"].cpu()
    for b, T in enumerate(x["seqlen_k"].cpu().tolist()):
        for pos in range(T, (T + 63) // 64 * 64):
            blk = int(table[b, pos // 64])
            x["k_cache"][blk, :, pos % 64, :] = nan
            x["v_cache"][blk, :, pos % 64, :] = nan


@pytest.mark.parametrize("mode,rel_extent", [("prefill", 150), ("prefill", 0), ("decode", 200)])
def test_nan_past_sequence_end_is_ignored(env, mode, rel_extent):
    """Keys past a sequence's end inside its last loaded block are masked; their V rows are
    zeroed before P V, so NaN there (0 * NaN = NaN otherwise) leaves the output finite and
    equal to the oracle's, which reads only the valid keys."""
    gen, AttentionStep, _ = env
    if mode == "decode":
        w = gen.custom("nan-tail-dec", Hq=16, Hkv=2, q_lens=[9, 4], prefix_lens=[900, 2000],
                       rel_extent=rel_extent, log_scale_base=256.0)
    else:
        w = gen.custom("nan-tail", Hq=8, Hkv=2, q_lens=[301, 140], prefix_lens=[20, 3], window=200,
                       rel_extent=rel_extent)
    x_cpu = gen.make_inputs(w, seed=31, device="cpu")
    x = {k: v.cuda() for k, v in x_cpu.items()}
    assert all(T % 64 != 0 for T in x_cpu["seqlen_k"].tolist())
    step = AttentionStep(w, x, mode=mode, out_dtype=torch.float32)
    step.run_prologue()
    _poison_tails(x)
    step.run_attention()
    torch.cuda.synchronize()
    assert step.device_status() == 0
    _check_all_rows(env, w, x_cpu, x, step)


@pytest.mark.parametrize("where", ["pageable", "pinned"])
def test_cache_outside_this_gpu_is_rejected(env, where):
    """The TMA-read tensors must be device memory of the current device: a cache in host
    memory (pageable or pinned) is rejected with INVALID_ARG and nothing is launched."""
    gen, AttentionStep, _ = env
    import relative_bias_hybrid_gb300.inkattn as ia
    w = gen.custom("hostptr", Hq=8, Hkv=2, q_lens=[9], prefix_lens=[100], rel_extent=50)
    x = gen.make_inputs(w, seed=3, device="cuda")
    host = x["k_cache"].cpu()
    if where == "pinned":
        host = host.pin_memory()
    out = torch.full((w.N_tok, w.Hq, 128), 7.0, dtype=torch.float32, device="cuda")
    p = ia.attn_params(q=x["q"], k_cache=host, v_cache=x["v_cache"], cu_seqlens_q=x["cu_seqlens_q"],
                       seqlen_k=x["seqlen_k"], block_table=x["block_table"], out=out, max_seqlen_q=9,
                       max_seqlen_k=max(w.seqlen_k), r=x["r"], P=x["P"], rel_extent=w.rel_extent)
    assert ia.inkattn_prefill(p, raise_on_error=False) == ia.INKATTN_ERR_INVALID_ARG
    assert ia.inkattn_decode(p, 1, None, raise_on_error=False) == ia.INKATTN_ERR_INVALID_ARG
    assert ia.inkattn_decode_noalloc(p, 0, raise_on_error=False) == ia.INKATTN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())                  # nothing was written
    p.k_cache = x["k_cache"].data_ptr()               # the same call on device memory runs
    assert ia.inkattn_prefill(p, raise_on_error=False) == ia.INKATTN_OK
    torch.cuda.synchronize()
