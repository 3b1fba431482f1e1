"""GPU parity of inkattn_output_conv against the fp64 oracle.

Bars: the new residual stream h and the conv state bit-exact (both are correctly
rounded values of exact sums); out within 1 bf16 ulp (its sum of squares is taken in
fp32 on the device); slots no sequence names untouched."""

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
    return gen, ia, oracle_mod


def _run(env, w, D=0, seed=0, inplace=False, x_cpu=None, spare_slots=0):
    """Draws the inputs on the device (or takes x_cpu), keeps a host copy of them as they
    were before the call, runs inkattn_output_conv and returns both."""
    gen, ia, _ = env
    if x_cpu is not None:
        x = {k: v.cuda() for k, v in x_cpu.items()}
    else:
        x = gen.make_output_conv_inputs(w, seed=seed, D=D, device="cuda")
    if spare_slots:
        # extra state slots nobody names, placed first: sequences use slots spare.. spare+B-1
        _, _, Dx = x["conv_state"].shape
        extra = torch.full((spare_slots, 3, Dx), 1.5, dtype=torch.bfloat16, device="cuda")
        x["conv_state"] = torch.cat([extra, x["conv_state"]])
        x["state_slot"] = x["state_slot"] + spare_slots
    x_cpu = {k: v.cpu() for k, v in x.items()}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    h = x["residual"] if inplace else torch.empty_like(x["y"])
    out = torch.empty_like(x["y"])
    max_q = max(w.q_lens) if w.q_lens else 0
    p = ia.output_conv_params(y=x["y"], conv_w=x["conv_w"], norm_w=x["norm_w"],
                              cu_seqlens_q=x["cu_seqlens_q"], state_slot=x["state_slot"],
                              conv_state=x["conv_state"], residual=x["residual"], h_out=h, out=out,
                              max_seqlen_q=max_q, eps=w.eps, dev_status=status)
    ia.inkattn_output_conv(p)
    torch.cuda.synchronize()
    return x_cpu, x, h, out, int(status.item())


def _check(env, w, x_cpu, x, h, out, status, seqs=None):
    gen, _, oracle = env
    assert status == 0
    cu = x_cpu["cu_seqlens_q"].numpy()
    if seqs is None:
        seqs = list(range(len(cu) - 1))
    # sequences are independent: run the oracle on the listed ones only
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in seqs]).astype(np.int64)
    lens = [int(cu[b + 1] - cu[b]) for b in seqs]
    sub_cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    slots = x_cpu["state_slot"].numpy()[seqs]
    ref = oracle.output_conv(cu_seqlens_q=sub_cu, D=x_cpu["y"].shape[1], y=gen.bits(x_cpu["y"])[rows],
                             conv_w=x_cpu["conv_w"].numpy(), state_slot=slots,
                             conv_state=gen.bits(x_cpu["conv_state"]),
                             residual=gen.bits(x_cpu["residual"])[rows],
                             norm_w=x_cpu["norm_w"].numpy(), eps=w.eps)
    assert np.array_equal(gen.bits(h)[rows], ref["h"])
    assert bf16_ulp_diff(gen.bits(out)[rows], ref["out"]).max() <= 1.0
    st = gen.bits(x["conv_state"])
    assert np.array_equal(st[slots], ref["conv_state"][slots])
    return st


def test_output_conv_tiny(env):
    gen = env[0]
    w = gen.workload("tiny")                 # D = 8 x 128 = 1024, zero carried state
    _check(env, w, *_run(env, w))


def test_output_conv_short_and_ragged_sequences_with_state(env):
    """Sequences of 0..3 tokens (the new state mixes carried rows and new ones), lengths
    around the 16-token tile and several tiles, random carried state."""
    gen = env[0]
    w = gen.custom("oc_ragged", Hq=64, Hkv=8, q_lens=[1, 2, 3, 0, 4, 15, 16, 17, 33, 100],
                   prefix_lens=[5, 1, 2, 7, 0, 3, 9, 0, 40, 2])
    x_cpu, x, h, out, status = _run(env, w, seed=3, spare_slots=2)
    st = _check(env, w, x_cpu, x, h, out, status)
    # the two unnamed slots are untouched; the empty sequence keeps its state
    assert np.array_equal(st[:2], gen.bits(x_cpu["conv_state"][:2]))
    empty = int(x_cpu["state_slot"][3])
    assert np.array_equal(st[empty], gen.bits(x_cpu["conv_state"][empty]))


@pytest.mark.parametrize("D", [8, 24, 1032, 4096, 16392, 32768])
def test_output_conv_hidden_widths(env, D):
    """One group of 8 channels; a width whose groups leave most threads of the last pass
    idle; the widest allowed."""
    gen = env[0]
    w = gen.custom("oc_width", Hq=8, Hkv=1, q_lens=[37, 5], prefix_lens=[0, 2])
    _check(env, w, *_run(env, w, D=D, seed=D))


def test_output_conv_in_place_residual(env):
    gen = env[0]
    w = gen.custom("oc_inplace", Hq=64, Hkv=8, q_lens=[50, 7], prefix_lens=[3, 0])
    x_cpu, x, h, out, status = _run(env, w, seed=5, inplace=True)
    assert h.data_ptr() == x["residual"].data_ptr()
    _check(env, w, x_cpu, x, h, out, status)


def test_output_conv_delta_filter_zero_residual(env):
    """A delta filter and a zero residual make h a bit-exact copy of y (pure indexing)."""
    gen = env[0]
    w = gen.custom("oc_delta", Hq=64, Hkv=8, q_lens=[40, 3], prefix_lens=[10, 0])
    x_cpu = gen.make_output_conv_inputs(w, seed=6, device="cpu")
    x_cpu["conv_w"] = torch.zeros_like(x_cpu["conv_w"])
    x_cpu["conv_w"][:, 3] = 1.0
    x_cpu["residual"] = torch.zeros_like(x_cpu["residual"])
    x_cpu, x, h, out, status = _run(env, w, x_cpu=x_cpu)
    assert status == 0
    assert torch.equal(h.cpu(), x_cpu["y"])
    _check(env, w, x_cpu, x, h, out, status)


def test_output_conv_bad_state_slot_reports_bounds(env):
    gen, ia, _ = env
    w = gen.custom("oc_bad", Hq=8, Hkv=1, q_lens=[20, 20], prefix_lens=[0, 0])
    x_cpu = gen.make_output_conv_inputs(w, seed=7, device="cpu")
    x_cpu["state_slot"] = torch.tensor([0, 5], dtype=torch.int32)   # 2 slots exist
    x_cpu, x, h, out, status = _run(env, w, x_cpu=x_cpu)
    assert status == ia.INKATTN_ERR_DEVICE_BOUNDS
    # the valid sequence was still processed
    _check(env, w, x_cpu, x, h, out, 0, seqs=[0])


@pytest.mark.parametrize("name", ["swa", "decode"])
def test_output_conv_full_size(env, name):
    """The launch the bench times (D = 8192), on the whole SWA layer and the MTP-verify
    decode batch."""
    gen = env[0]
    w = gen.workload(name)
    _check(env, w, *_run(env, w))


def test_output_conv_ragged_batch_sampled(env):
    """The ragged mixed prefill batch (158k tokens, D = 8192): every sequence runs on the
    GPU, the oracle checks four of them whole."""
    gen = env[0]
    w = gen.workload("ragged")
    _check(env, w, *_run(env, w), seqs=[0, 5, 11, 15])


def test_conv_rounding_hard_cases(env):
    """Conv sums whose fp32 evaluation lands on or next to a bf16 rounding boundary, or
    cancels: the kernel's fast path must hand each of them to its error-free evaluation
    and store the correctly rounded value (h bit-exact with a zero residual).  Per channel,
    taps w and carried rows x (oldest first), with y = 0 for the one new token:
      1 + 2^-8 + 2^-30 (just above a tie: rounds up), 1 + 2^-8 - 2^-30 (just below: down),
      1 + 2^-8 (an exact tie: even, 1), (1 + 2^-23) * 1.5 - 1.5 (cancellation, 1.5 * 2^-23),
      a sum whose terms cancel to 2^-40, and their negatives."""
    gen, ia, _ = env
    cases = [
        ([1.0, 2.0 ** -8, 2.0 ** -30, 0.0], [1.0, 1.0, 1.0]),
        ([1.0, 2.0 ** -8, -(2.0 ** -30), 0.0], [1.0, 1.0, 1.0]),
        ([1.0, 2.0 ** -8, 0.0, 0.0], [1.0, 1.0, 1.0]),
        ([1.0 + 2.0 ** -23, -1.0, 0.0, 0.0], [1.5, 1.5, 0.0]),
        ([3.0, -1.0, 2.0 ** -40, 0.0], [1.0, 3.0, 1.0]),
        ([0.1, 0.2, 0.3, 0.0], [-3.0, 1.5, 0.5]),
    ]
    cases += [([-w for w in ws], xs) for ws, xs in cases]
    D = 8 * ((len(cases) + 7) // 8)
    w = gen.custom("oc_hard", Hq=1, Hkv=1, q_lens=[1], prefix_lens=[3])
    x_cpu = gen.make_output_conv_inputs(w, seed=1, D=D, device="cpu")
    conv_w = torch.zeros(D, 4)
    state = torch.zeros(1, 3, D)
    for c, (ws, xs) in enumerate(cases):
        conv_w[c] = torch.tensor(ws, dtype=torch.float64).float()
        state[0, :, c] = torch.tensor(xs)
    x_cpu["conv_w"] = conv_w
    x_cpu["conv_state"] = state.to(torch.bfloat16)
    assert torch.equal(x_cpu["conv_state"].float(), state)         # the rows are bf16 values
    x_cpu["y"] = torch.zeros_like(x_cpu["y"])
    x_cpu["residual"] = torch.zeros_like(x_cpu["residual"])
    x_cpu, x, h, out, status = _run(env, w, x_cpu=x_cpu)
    _check(env, w, x_cpu, x, h, out, status)
