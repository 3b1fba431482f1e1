"""Host-side logic of bench.py: the algorithmic work counts (closed forms for the
workloads), and the one-GPU rule (a multi-GPU request is refused before any GPU work)."""
import pytest

import bench
from relative_bias_hybrid_gb300 import inputs as gen


def test_sliding_window_pair_count_closed_form():
    w = gen.workload("swa")
    # sum_{i<8192} min(i+1, 4096) = 4096*4097/2 + 4096*4096
    assert bench.visible_pairs(w) == 4096 * 4097 // 2 + 4096 * 4096 == 25_167_872
    assert bench.biased_pairs(w) == 512 * 513 // 2 + (8192 - 512) * 512
    assert bench.attention_flops(w) == pytest.approx(8.247e11 + 1.664e10, rel=2e-3)


def test_full_layer_pair_count_closed_form():
    w = gen.workload("full")
    assert bench.visible_pairs(w) == 32768 * 32769 // 2 == 536_887_296
    # biased pairs: sum_i min(i + 1, 1024) = 1024*1025/2 + (32768 - 1024) * 1024
    assert bench.biased_pairs(w) == 1024 * 1025 // 2 + (32768 - 1024) * 1024
    assert bench.attention_flops(w) == pytest.approx(1.7593e13 + 1.353e11, rel=1e-3)


def test_decode_bytes_and_prologue_bytes():
    w = gen.workload("decode")
    # K+V of 32 sequences x 8 KV heads x 32768 keys x 128 x bf16 = 4 GiB, plus small terms
    assert bench.decode_bytes(w) == pytest.approx(4.314e9, rel=1e-3)
    s = gen.workload("swa")
    assert bench.prologue_bytes(s) == 40_964 * 8192 + 2 * 2 * 3 * 1024 * 2


def test_ragged_workload_is_seeded_and_in_range():
    a, b = gen.workload("ragged"), gen.workload("ragged")
    assert a.q_lens == b.q_lens and a.prefix_lens == b.prefix_lens and a.B == 16
    assert all(1024 <= n <= 16384 for n in a.q_lens) and all(0 <= p <= 4096 for p in a.prefix_lens)


@pytest.mark.parametrize("argv,env", [(["--gpus", "2"], {}), (["--gpus", "8"], {}),
                                      ([], {"WORLD_SIZE": "2", "RANK": "0"})])
def test_more_than_one_gpu_is_refused_before_any_gpu_work(monkeypatch, argv, env):
    for k, v in env.items():
        monkeypatch.setenv(k, v)

    def no_gpu(*a, **k):
        raise AssertionError("the GPU arm ran")

    monkeypatch.setattr(bench, "run_gpu", no_gpu)
    assert bench.main(argv) == 2


def test_qkvr_flop_count_and_grid_inputs_are_exact_in_fp32():
    """The bench's qkvr FLOP count, and the claim the GPU parity tests rest on: with the
    integer-grid inputs every projection sum is exact in fp32 whatever the order of the
    additions (checked on sampled rows of the full-width weight against float64, summing in
    the natural order, in reverse and pairwise)."""
    import numpy as np
    import torch
    import bench
    from relative_bias_hybrid_gb300 import inputs as gen
    w = gen.workload("swa")
    assert bench.qkvr_flops(w, 8192) == 2.0 * 8192 * 12288 * 8192
    small = gen.custom("g", Hq=16, Hkv=2, q_lens=[5], prefix_lens=[0], rel_extent=16)
    x = gen.make_qkvr_inputs(small, 8192, seed=3, grid=True)
    xf = x["x"].to(torch.float64).numpy()
    wf = x["w_qkvr"].to(torch.float64).numpy()[::97]
    exact = xf @ wf.T
    prod = (xf[:, None, :] * wf[None, :, :]).astype(np.float32)       # exact in fp32 (multiples of 2^-9)
    assert np.array_equal(prod.astype(np.float64), xf[:, None, :] * wf[None, :, :])
    fwd = np.zeros(exact.shape, np.float32)
    for k in range(prod.shape[2]):
        fwd += prod[:, :, k]
    rev = np.zeros(exact.shape, np.float32)
    for k in reversed(range(prod.shape[2])):
        rev += prod[:, :, k]
    pair = prod
    while pair.shape[2] > 1:
        pair = pair[:, :, 0::2] + pair[:, :, 1::2]
    for got in (fwd, rev, pair[:, :, 0]):
        assert np.array_equal(got.astype(np.float64), exact)
