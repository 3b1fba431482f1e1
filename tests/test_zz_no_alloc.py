"""inkattn_decode_noalloc: decode for callers that cannot allocate device memory where
they decode (host functions enqueued on a stream, plugin hosts that own all device
memory, serving loops that must not allocate on the hot path).

It must give the same result as inkattn_decode + inkattn_combine with a workspace the
caller allocated, on two calls in a row (the static buffer keeps the previous call's
contents).  This file is collected last on purpose."""
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


@pytest.mark.parametrize("splits", [5, 0])
def test_noalloc_decode_matches_workspace_decode(env, splits):
    gen, ia, AttentionStep = env
    w = gen.custom("noalloc", Hq=64, Hkv=8, q_lens=[9, 9, 5], prefix_lens=[3000, 700, 6000],
                   rel_extent=1024, log_scale_base=8192.0)
    x = gen.make_inputs(w, seed=21, device="cuda")
    ref = AttentionStep(w, x, mode="decode", num_splits=splits)
    ref.run_prologue()                        # fills the cache for the new tokens once
    ref.run_attention()                       # existing entry points, torch-allocated workspace
    torch.cuda.synchronize()
    assert ref.device_status() == 0
    if splits:
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
        assert torch.isfinite(out2.float()).all()
        assert (out2.float() - ref.out.float()).abs().max().item() <= 1e-2
        assert (lse2 - ref.lse).abs().max().item() <= 2e-3


def test_noalloc_rejects_partials_beyond_its_buffer(env):
    gen, ia, AttentionStep = env
    w = gen.custom("big", Hq=64, Hkv=8, q_lens=[9] * 64, prefix_lens=[2000] * 64, rel_extent=64)
    x = gen.make_inputs(w, seed=22, device="cuda")
    step = AttentionStep(w, x, mode="decode", num_splits=1)
    need = ia.inkattn_decode_workspace_bytes(step.attn, 8)
    assert need > ia.DECODE_NOALLOC_MAX_BYTES
    rc = ia.inkattn_decode_noalloc(step.attn, 8, raise_on_error=False)
    assert rc == ia.INKATTN_ERR_INVALID_ARG
