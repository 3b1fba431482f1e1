"""The failure path of the bounded device waits, made to run on purpose without any fault:
in a child process with INKATTN_TEST_WITHHOLD_ARRIVAL=1 and INKATTN_TEST_WAIT_LIMIT_US=2000,
the attention kernels' softmax withholds its first arrival on the barrier that the MMA warp
waits on before P V.  That wait runs out after 2 ms; the kernel must record
INKATTN_ERR_DEVICE_TIMEOUT in dev_status, drain the copies and MMAs it issued, release TMEM
and return, leaving the CUDA context usable.  Covered: the relative-bias prefill with CTA
pairs (K/V multicast) and without, the prefill without bias, and the decode over a bf16
and over an E4M3 cache (the latter with its converter warps between the copies and the
MMAs); and the qkvr projections (CTA pairs), where one epilogue warp of each odd CTA
withholds its first accumulator release, so the even CTA's MMA warp gives up, and both
CTAs of every pair wind down (the pair's copies and commits drained, TMEM released by
both)."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import torch
from relative_bias_hybrid_gb300 import inputs as gen
from relative_bias_hybrid_gb300.step import AttentionStep
cases = {
    "prefill_pairs": (gen.custom("t1", Hq=8, Hkv=2, q_lens=[300, 140], prefix_lens=[0, 90], rel_extent=100), "prefill"),
    "prefill_unpaired": (gen.custom("t2", Hq=6, Hkv=2, q_lens=[300], prefix_lens=[0], rel_extent=100), "prefill"),
    "prefill_no_bias": (gen.custom("t3", Hq=8, Hkv=2, q_lens=[600], prefix_lens=[0], rel_extent=0), "prefill"),
    "decode": (gen.custom("t4", Hq=16, Hkv=2, q_lens=[9, 4], prefix_lens=[2000, 700], rel_extent=200), "decode"),
    "decode_e4m3": (gen.custom("t5", Hq=16, Hkv=2, q_lens=[9, 4], prefix_lens=[2000, 700], rel_extent=200), "decode"),
}
res = {}
for name, (w, mode) in cases.items():
    x = gen.make_inputs(w, seed=3, device="cuda", kv_dtype="e4m3" if name.endswith("e4m3") else "bf16")
    st = AttentionStep(w, x, mode=mode, num_splits=1 if mode == "decode" else 0)
    st.run_prologue()                 # no bounded waits in the prologue
    torch.cuda.synchronize()
    assert st.device_status() == 0
    t0 = time.time()
    st.run_attention()
    torch.cuda.synchronize()
    res[name] = {"status": st.device_status(), "seconds": time.time() - t0}
from relative_bias_hybrid_gb300.step import QkvrStep
# enough items that every cluster of the persistent grid takes at least three
wq = gen.custom("t6", Hq=16, Hkv=2, q_lens=[12000, 300], prefix_lens=[0, 5], rel_extent=16)
xq = gen.make_qkvr_inputs(wq, 128, seed=3, device="cuda", grid=True)
sq = QkvrStep(wq, xq)
t0 = time.time()
sq.run()
torch.cuda.synchronize()
res["qkvr"] = {"status": sq.device_status(), "seconds": time.time() - t0}
res["context_usable"] = torch.arange(1000, device="cuda", dtype=torch.float32).sum().item() == 499500.0
print("RESULT " + json.dumps(res))
"""


@pytest.fixture(scope="module")
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from relative_bias_hybrid_gb300 import build
    build.build()


def test_withheld_arrival_times_out_cleanly(built):
    env = dict(os.environ, INKATTN_TEST_WITHHOLD_ARRIVAL="1", INKATTN_TEST_WAIT_LIMIT_US="2000")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])
    assert res.pop("context_usable") is True
    for name, v in res.items():
        assert v["status"] == 4, (name, v)          # INKATTN_ERR_DEVICE_TIMEOUT
        assert v["seconds"] < 10.0, (name, v)


def test_without_the_setting_nothing_is_withheld(built):
    """The same child without the environment variables: every status stays 0."""
    env = {k: v for k, v in os.environ.items() if not k.startswith("INKATTN_TEST_")}
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    res = json.loads([l for l in r.stdout.splitlines() if l.startswith("RESULT ")][-1][len("RESULT "):])
    assert res.pop("context_usable") is True
    for name, v in res.items():
        assert v["status"] == 0, (name, v)
