"""The C-ABI calls issue only stream-ordered work, so a whole step (prologue, then prefill,
or decode and combine), and the qkvr projections with the prologue fused in, can be captured
into a CUDA graph and replayed: the replay must write exactly what the same calls wrote
when issued directly (same inputs, same state)."""
import pytest
import torch

pytestmark = pytest.mark.gpu

_STATE = ("conv_state_k", "conv_state_v", "k_cache", "v_cache")


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from relative_bias_hybrid_gb300 import build
    build.build()
    from relative_bias_hybrid_gb300 import inputs as gen
    from relative_bias_hybrid_gb300.step import AttentionStep
    return gen, AttentionStep


@pytest.mark.parametrize("mode,splits", [("prefill", 0), ("prefill_nobias", 0), ("decode", 1), ("decode", 3),
                                         ("decode_e4m3", 3)])
def test_step_replays_from_a_cuda_graph(env, mode, splits):
    gen, AttentionStep = env
    kv = "e4m3" if mode.endswith("e4m3") else "bf16"
    mode = mode.replace("_e4m3", "")
    if mode == "decode":
        w = gen.custom("graph-dec", Hq=16, Hkv=2, q_lens=[9, 4], prefix_lens=[900, 2000], rel_extent=200,
                       log_scale_base=256.0)
    else:
        w = gen.custom("graph-pre", Hq=8, Hkv=2, q_lens=[300, 140], prefix_lens=[20, 0], window=200,
                       rel_extent=0 if mode == "prefill_nobias" else 150)
    x = gen.make_inputs(w, seed=21, device="cuda", kv_dtype=kv)
    state = _STATE + (("k_scale", "v_scale") if kv == "e4m3" else ())
    saved = {k: x[k].clone() for k in state}
    step = AttentionStep(w, x, mode="decode" if mode == "decode" else "prefill", num_splits=splits)

    step.run()
    torch.cuda.synchronize()
    direct = {"out": step.out.clone(), "lse": step.lse.clone(), **{k: x[k].clone() for k in state}}
    assert int(step.status.item()) == 0

    for k in state:
        x[k].copy_(saved[k])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run()
    # capturing records the work without running it; start the replay from the same state
    for k in state:
        x[k].copy_(saved[k])
    step.out.zero_()
    step.lse.zero_()
    graph.replay()
    torch.cuda.synchronize()

    assert int(step.status.item()) == 0
    assert torch.equal(step.out, direct["out"])
    assert torch.equal(step.lse, direct["lse"])
    for k in state:
        assert torch.equal(x[k], direct[k]), k


def test_qkvr_replays_from_a_cuda_graph(env):
    """The qkvr projections with the prologue fused in (persistent CTA-pair kernel),
    captured and replayed: q, r, the cache rows and the new conv state as issued directly."""
    gen, _ = env
    from relative_bias_hybrid_gb300.step import QkvrStep
    w = gen.custom("graph-qkvr", Hq=16, Hkv=2, q_lens=[300, 9, 140], prefix_lens=[0, 40, 2], rel_extent=16)
    x = gen.make_qkvr_inputs(w, 256, seed=22, device="cuda")
    saved = {k: x[k].clone() for k in ("k_cache", "v_cache")}
    step = QkvrStep(w, x)
    step.run()
    torch.cuda.synchronize()
    assert step.device_status() == 0
    direct = {"q": step.q_out.clone(), "r": step.r_out.clone(), "sk": step.state_k.clone(),
              "sv": step.state_v.clone(), **{k: x[k].clone() for k in saved}}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run()
    for k in saved:
        x[k].copy_(saved[k])
    for t in (step.q_out, step.r_out, step.state_k, step.state_v):
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert step.device_status() == 0
    assert torch.equal(step.q_out, direct["q"]) and torch.equal(step.r_out, direct["r"])
    assert torch.equal(step.state_k, direct["sk"]) and torch.equal(step.state_v, direct["sv"])
    for k in saved:
        assert torch.equal(x[k], direct[k]), k
