"""GPU parity of inkattn_prologue against the fp64 oracle.

Bars: conv state and untouched cache bytes bit-exact; q_out, normed K and conv'd V
within 1 bf16 ulp of the oracle's correctly rounded values; a delta conv filter makes
the V cache a bit-exact scatter of v (pure slot indexing)."""
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
    from relative_bias_hybrid_gb300.step import AttentionStep
    return gen, AttentionStep, oracle_mod


def _run(env, w, x_cpu=None, seed=0):
    gen, AttentionStep, _ = env
    x_cpu = x_cpu if x_cpu is not None else gen.make_inputs(w, seed=seed, device="cpu")
    x = {k: v.cuda() for k, v in x_cpu.items()}
    step = AttentionStep(w, x, mode="prefill")
    step.run_prologue()
    torch.cuda.synchronize()
    return x_cpu, x, step


def _check(env, w, x_cpu, x, step):
    gen, _, oracle = env
    assert step.device_status() == 0
    ref = oracle.prologue_for_inputs(x_cpu, w)
    assert bf16_ulp_diff(gen.bits(step.q_out), ref["q_out"]).max() <= 1.0
    assert np.array_equal(gen.bits(x["conv_state_k"]), ref["conv_state_k"])
    assert np.array_equal(gen.bits(x["conv_state_v"]), ref["conv_state_v"])
    slots = x_cpu["slot_mapping"].numpy().astype(np.int64)
    blk, off = slots // w.block_size, slots % w.block_size
    kg, vg = gen.bits(x["k_cache"]), gen.bits(x["v_cache"])
    assert bf16_ulp_diff(kg[blk, :, off, :], ref["k_cache"][blk, :, off, :]).max() <= 1.0
    assert bf16_ulp_diff(vg[blk, :, off, :], ref["v_cache"][blk, :, off, :]).max() <= 1.0
    untouched = np.ones(kg.shape[0] * w.block_size, bool)
    untouched[slots] = False
    k0 = gen.bits(x_cpu["k_cache"]).transpose(0, 2, 1, 3).reshape(-1, w.Hkv, w.head_dim)
    v0 = gen.bits(x_cpu["v_cache"]).transpose(0, 2, 1, 3).reshape(-1, w.Hkv, w.head_dim)
    assert np.array_equal(kg.transpose(0, 2, 1, 3).reshape(-1, w.Hkv, w.head_dim)[untouched], k0[untouched])
    assert np.array_equal(vg.transpose(0, 2, 1, 3).reshape(-1, w.Hkv, w.head_dim)[untouched], v0[untouched])


def test_prologue_tiny(env):
    gen = env[0]
    w = gen.workload("tiny")
    _check(env, w, *_run(env, w))


def test_weights_at_4_byte_alignment(env):
    # the fp32 conv weights and gains need only 4-byte alignment: each passed 4 bytes past a
    # 16-byte boundary
    gen, AttentionStep, _ = env
    w = gen.workload("tiny")
    x_cpu = gen.make_inputs(w, seed=3, device="cpu")
    x = {k: v.cuda() for k, v in x_cpu.items()}
    for name in ("conv_w_k", "conv_w_v", "q_norm_w", "k_norm_w"):
        t = x[name]
        buf = torch.zeros(t.numel() + 4, dtype=t.dtype, device=t.device)
        view = buf[1:1 + t.numel()].view(t.shape)
        view.copy_(t)
        assert view.data_ptr() % 16 == 4
        x[name] = view
    step = AttentionStep(w, x, mode="prefill")
    step.run_prologue()
    torch.cuda.synchronize()
    _check(env, w, x_cpu, x, step)


def test_prologue_ragged_short_sequences(env):
    gen = env[0]
    w = gen.custom("mix", Hq=8, Hkv=2, q_lens=[1, 2, 3, 0, 17, 40, 5, 64],
                   prefix_lens=[0, 1, 2, 5, 0, 3, 100, 7], rel_extent=16)
    _check(env, w, *_run(env, w, seed=3))


@pytest.mark.parametrize("name", ["swa", "full"])
def test_prologue_layer_full_size(env, name):
    """One prefill layer at full size (8192 / 32768 tokens): the two K/V group sizes the
    launch picks (32 tokens on the short grid, 64 on the long one)."""
    gen = env[0]
    w = gen.workload(name)
    _check(env, w, *_run(env, w, seed=1))


def test_prologue_many_sequences_uneven_tiles(env):
    """Long enough that K/V groups of 64 tokens are used, with sequence lengths that end
    inside a group and inside a query tile, and a carried state on every sequence."""
    gen = env[0]
    w = gen.custom("many", Hq=8, Hkv=2, q_lens=[1000, 77, 4097, 63, 2048, 5, 3001, 130] * 2,
                   prefix_lens=[0, 3, 50, 2, 7, 1, 900, 4] * 2)
    _check(env, w, *_run(env, w, seed=4))


def test_prologue_decode_shape(env):
    gen = env[0]
    w = gen.custom("dec", Hq=64, Hkv=8, q_lens=[9] * 6, prefix_lens=[100, 1, 2, 0, 77, 5000])
    _check(env, w, *_run(env, w, seed=2))


def test_delta_filter_makes_v_cache_an_exact_scatter(env):
    gen = env[0]
    w = gen.custom("delta", Hq=8, Hkv=2, q_lens=[33, 5], prefix_lens=[4, 0])
    x_cpu = gen.make_inputs(w, seed=5, device="cpu")
    x_cpu["conv_w_v"].zero_()
    x_cpu["conv_w_v"][:, 3] = 1.0
    _, x, step = _run(env, w, x_cpu=x_cpu)
    slots = x_cpu["slot_mapping"].numpy().astype(np.int64)
    vg = gen.bits(x["v_cache"])[slots // 64, :, slots % 64, :]
    assert np.array_equal(vg.reshape(len(slots), -1), gen.bits(x_cpu["v"]))


def test_chunked_prologue_equals_whole(env):
    """Two calls over a split sequence, carrying the conv state, write the same cache
    bytes and leave the same state as one call."""
    gen, AttentionStep, _ = env
    w = gen.custom("whole", Hq=8, Hkv=2, q_lens=[50], prefix_lens=[0])
    x_cpu = gen.make_inputs(w, seed=7, device="cpu")
    _, xa, _ = _run(env, w, x_cpu=x_cpu)
    xb = {k: v.cuda() for k, v in x_cpu.items()}
    for lo, hi in ((0, 2), (2, 21), (21, 50)):
        wc = gen.custom("chunk", Hq=8, Hkv=2, q_lens=[hi - lo], prefix_lens=[lo])
        xc = dict(xb)
        for key in ("q", "k", "v", "slot_mapping"):
            xc[key] = xb[key][lo:hi].contiguous()
        xc["cu_seqlens_q"] = torch.tensor([0, hi - lo], dtype=torch.int32, device="cuda")
        xc["seqlen_k"] = torch.tensor([hi], dtype=torch.int32, device="cuda")
        step = AttentionStep(wc, xc, mode="prefill")
        step.run_prologue()
    torch.cuda.synchronize()
    for key in ("k_cache", "v_cache", "conv_state_k", "conv_state_v"):
        assert torch.equal(xa[key].view(torch.int16), xb[key].view(torch.int16)), key


def test_out_of_range_slot_is_flagged_not_written(env):
    gen = env[0]
    w = gen.custom("bad", Hq=8, Hkv=2, q_lens=[10], prefix_lens=[0])
    x_cpu = gen.make_inputs(w, seed=9, device="cpu")
    good = x_cpu["slot_mapping"].clone()
    x_cpu["slot_mapping"][4] = x_cpu["k_cache"].shape[0] * 64 + 3      # past the cache
    x_cpu2 = {k: v.clone() for k, v in x_cpu.items()}
    _, x, step = _run(env, w, x_cpu=x_cpu)
    assert step.device_status() == 5
    # every other token was written as usual
    x_cpu2["slot_mapping"] = good
    _, x_ok, _ = _run(env, w, x_cpu=x_cpu2)
    g = good.numpy().astype(np.int64)
    keep = np.arange(10) != 4
    kg = gen.bits(x["k_cache"])[g // 64, :, g % 64, :][keep]
    kr = gen.bits(x_ok["k_cache"])[g // 64, :, g % 64, :][keep]
    assert np.array_equal(kg, kr)
