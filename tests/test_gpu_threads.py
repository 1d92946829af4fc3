"""The C ABI from several host threads at once: calls are stateless and
thread-safe (each thread brings its own stream, workspace and outputs).  A
fresh process runs the first calls of four threads concurrently -- so the
per-device lazy set-up (kernel attributes, occupancy, the tensor-map encoder
lookup) races -- mixing bf16 decode (CTA pairs), FP8 decode (1-byte path)
and multi-token decode, and every result must equal, bit for bit, the same
call made alone afterwards (a fixed split plan is deterministic)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import sys, threading
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import mla_decode_attention_paged_gb300 as mla
from mla_decode_attention_paged_gb300 import workloads as W

mla.load_library(build_if_missing=True)
dev = torch.device("cuda", 0)
g = W.generator(77)
B, H, P = 3, 16, 64
lens = torch.tensor([700, 129, 1500], dtype=torch.int32)
table, npg = W.draw_page_table(lens, P, True, g)
bf = W.draw_bf16((npg, P, 576), 1.0, g).to(dev)
codes, sc = W.draw_fp8_cache(npg, P, g)
codes, sc = codes.to(dev), sc.to(dev)
WK, WV = W.draw_bf16((H, 128, 512), 0.02, g).to(dev), W.draw_bf16((H, 128, 512), 0.02, g).to(dev)
qn, qp = W.draw_bf16((B, H, 128), 1.0, g).to(dev), W.draw_bf16((B, H, 64), 1.0, g).to(dev)
qn2, qp2 = W.draw_bf16((B, 2, H, 128), 1.0, g).to(dev), W.draw_bf16((B, 2, H, 64), 1.0, g).to(dev)
table, lens = table.to(dev), lens.to(dev)
scale = 1.0 / np.sqrt(192.0)

def run(kind, stream):
    with torch.cuda.stream(stream):
        if kind == 0:
            d = mla.dims(H, P)
            return mla.decode(d, qn, qp, bf, None, table, lens, WK, WV, scale, num_splits=5, stream=stream)
        if kind == 1:
            d = mla.dims(H, P, fp8=True)
            return mla.decode(d, qn, qp, codes, sc, table, lens, WK, WV, scale, num_splits=5, stream=stream)
        d = mla.dims(H, P)
        return mla.decode_multi(d, qn2, qp2, bf, None, table, lens, WK, WV, scale, num_splits=5, stream=stream)

results, errors = {}, []
start = threading.Barrier(4)

def worker(i):
    try:
        s = torch.cuda.Stream(device=dev)
        start.wait()
        outs = [run((i + k) % 3, s) for k in range(6)]
        s.synchronize()
        results[i] = [(((i + k) % 3), o.clone(), l.clone()) for k, (o, l) in enumerate(outs)]
    except Exception as e:  # reported below
        errors.append(repr(e))

threads = [threading.Thread(target=worker, args=(i,)) for i in range(4)]
for t in threads: t.start()
for t in threads: t.join()
assert not errors, errors
torch.cuda.synchronize()
ref = {}
for kind in range(3):
    s = torch.cuda.current_stream()
    o, l = run(kind, s)
    torch.cuda.synchronize()
    ref[kind] = (o, l)
n = 0
for i, lst in results.items():
    for kind, o, l in lst:
        assert torch.equal(o, ref[kind][0]) and torch.equal(l, ref[kind][1]), (i, kind)
        n += 1
print("ok", n)
'''


def test_concurrent_first_calls_from_four_threads(cuda_lib):
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-4000:])
    assert r.stdout.strip().splitlines()[-1] == "ok 24"
