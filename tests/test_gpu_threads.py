"""Concurrent host threads: a fresh process starts four threads that, each
on its own CUDA stream, make their first calls of every kernel family at
the same time (the per-device setup of each kernel is then raced), and the
results must equal those of the same calls made one after another."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import sys, threading
sys.path.insert(0, sys.argv[1])
import torch
import rl_nvfp4_quantize_gb300 as nvq
from rl_nvfp4_quantize_gb300 import synth

dev = torch.device("cuda", 0)
w = synth.expert_weights(2, 256, 512, seed=1, device=dev)
x = synth.activations(300, 512, seed=2, device=dev)
counts = [120, 180]
torch.cuda.synchronize()

def work(out, stream):
    with torch.cuda.stream(stream):
        q = nvq.nvfp4_quantize_dual(w, four_over_six=True, stream=stream)
        n = nvq.nf4_quantize(w, stream=stream)
        m = nvq.mxfp8_quantize(w, columnwise=True, stream=stream)
        a = nvq.act_quantize_per_token(x, four_over_six=True, stream=stream)
        dy = x[:, :256].contiguous()
        g = nvq.nvfp4_dgrad(dy, counts, q["codes_row"], q["scales_row"], q["tensor_scale"], stream=stream)
        y = nvq.nf4_routed_linear(x, counts, n["codes"], n["absmax"], stream=stream)
        stream.synchronize()
        out.append([q["codes_row"], q["codes_col"], q["scales_col"], n["codes"], m["codes_col"],
                    m["scales_row"], a["codes"], g, y])

results = [[] for _ in range(4)]
threads = [threading.Thread(target=work, args=(results[i], torch.cuda.Stream(dev))) for i in range(4)]
for t in threads:
    t.start()
for t in threads:
    t.join()
ref = []
work(ref, torch.cuda.Stream(dev))
for r in results:
    assert len(r) == 1, "a thread failed"
    for a, b in zip(r[0], ref[0]):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), "results differ"
print("threads ok")
"""


def test_concurrent_first_calls():
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
