"""inkattn_decode_noalloc: decode for callers that cannot allocate device memory where
they decode (plugin hosts that own all device memory and hand over only inputs and
outputs, serving loops that must not allocate on the hot path).

With the same split count it runs the same kernels as inkattn_decode + inkattn_combine
with a workspace the caller allocated, so its output and LSE must be bit-identical to
theirs, on two calls in a row (the static buffer keeps the previous call's contents).
This file is collected last on purpose."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from relative_bias_hybrid_gb300 import build
    build.build()
    from relative_bias_hybrid_gb300 import inputs as gen
    from relative_bias_hybrid_gb300 import inkattn as ia
    from relative_bias_hybrid_gb300.step import AttentionStep
    return gen, ia, AttentionStep


def _noalloc_matches_workspace_decode(env, w, splits, expect_splits, seed):
    gen, ia, AttentionStep = env
    x = gen.make_inputs(w, seed=seed, device="cuda")
    ref = AttentionStep(w, x, mode="decode", num_splits=expect_splits, out_dtype=torch.float32)
    ref.run_prologue()                        # fills the cache for the new tokens once
    ref.run_attention()                       # existing entry points, torch-allocated workspace
    torch.cuda.synchronize()
    assert ref.device_status() == 0
    if expect_splits > 1:
        assert ref.workspace is not None      # the split partials do go through scratch memory
    out2 = torch.empty_like(ref.out)
    lse2 = torch.empty_like(ref.lse)
    p = ia.attn_params(q=ref.q_out, k_cache=x["k_cache"], v_cache=x["v_cache"],
                       cu_seqlens_q=x["cu_seqlens_q"], seqlen_k=x["seqlen_k"],
                       block_table=x["block_table"], out=out2, max_seqlen_q=max(w.q_lens),
                       max_seqlen_k=max(w.seqlen_k), r=x["r"], P=x["P"], rel_extent=w.rel_extent,
                       log_scale_base=w.log_scale_base, lse=lse2, dev_status=ref.status)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):                         # two calls in a row share the static buffer
        out2.fill_(float("nan"))
        lse2.fill_(float("nan"))
        rc = ia.lib().inkattn_decode_noalloc(ctypes.byref(p), splits, ctypes.c_void_p(stream))
        assert rc == ia.INKATTN_OK, ia.status_string(rc)
        torch.cuda.synchronize()
        assert ref.device_status() == 0
        assert torch.equal(out2.view(torch.int32), ref.out.view(torch.int32))
        assert torch.equal(lse2.view(torch.int32), ref.lse.view(torch.int32))


@pytest.mark.parametrize("splits", [5, 0])
def test_noalloc_decode_matches_workspace_decode(env, splits):
    gen, ia, AttentionStep = env
    w = gen.custom("noalloc", Hq=64, Hkv=8, q_lens=[9, 9, 5], prefix_lens=[3000, 700, 6000],
                   rel_extent=1024, log_scale_base=8192.0)
    expect = splits
    if splits == 0:
        x = gen.make_inputs(w, seed=21, device="cuda")
        probe = AttentionStep(w, x, mode="decode")
        expect = probe.num_splits
        assert expect > 1
        assert ia.inkattn_decode_workspace_bytes(probe.attn, expect) <= ia.DECODE_NOALLOC_MAX_BYTES
    _noalloc_matches_workspace_decode(env, w, splits, expect, seed=21)


def test_noalloc_lowers_the_heuristic_split_count_to_fit(env):
    """39 sequences x 9 queries over 16384 keys: the heuristic picks more splits than the
    static buffer holds, and the call takes the largest count below it that fits."""
    gen, ia, AttentionStep = env
    w = gen.custom("noalloc-big", Hq=64, Hkv=8, q_lens=[9] * 39, prefix_lens=[16384 - 9] * 39,
                   rel_extent=1024, log_scale_base=8192.0)
    x = gen.make_inputs(w, seed=23, device="cuda")
    probe = AttentionStep(w, x, mode="decode")
    S = probe.num_splits
    assert ia.inkattn_decode_workspace_bytes(probe.attn, S) > ia.DECODE_NOALLOC_MAX_BYTES
    while S > 1 and ia.inkattn_decode_workspace_bytes(probe.attn, S) > ia.DECODE_NOALLOC_MAX_BYTES:
        S -= 1
    assert S > 1
    del probe, x
    _noalloc_matches_workspace_decode(env, w, 0, S, seed=23)


def test_noalloc_rejects_partials_beyond_its_buffer(env):
    gen, ia, AttentionStep = env
    w = gen.custom("big", Hq=64, Hkv=8, q_lens=[9] * 64, prefix_lens=[2000] * 64, rel_extent=64)
    x = gen.make_inputs(w, seed=22, device="cuda")
    step = AttentionStep(w, x, mode="decode", num_splits=1)
    need = ia.inkattn_decode_workspace_bytes(step.attn, 8)
    assert need > ia.DECODE_NOALLOC_MAX_BYTES
    rc = ia.inkattn_decode_noalloc(step.attn, 8, raise_on_error=False)
    assert rc == ia.INKATTN_ERR_INVALID_ARG
