"""Determinism gate across processes and workloads ("cake_gdn: deterministic
chunked GDN training kernels", Validation of the round-13 kernels: many shapes,
repeated runs, hashed forward and backward outputs; "[Cake 1/13] gdn: ...", Tests:
repeats in a new process and on a side stream).

For the three fwd+bwd workloads of the method's configurations (4 x 4096, the
32K varlen pack, one 65536-token sequence with 64 value heads) every output of
fwd + bwd is hashed (SHA-256 of its bytes).  Within this process the hashes of
two runs on the default stream and one on a side stream must agree; a second
Python process computes the same hashes from scratch and must agree too.
"""
import hashlib
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORKLOADS = ("fb_4x4096", "fb_32k_varlen", "fb_65536_long")


def _hash_outputs(out):
    return {k: hashlib.sha256(v.contiguous().view(torch.uint8).cpu().numpy().tobytes()).hexdigest()
            for k, v in sorted(out.items()) if v is not None}


def workload_hashes(names, side_stream=True):
    """{workload: [hashes of each run]} of fwd + bwd through the C ABI: two runs on
    the current stream and (side_stream) one on a side stream."""
    from chunked_gated_delta_06_gb300 import workloads as W
    from gpu_helpers import run_chunk_raw
    res = {}
    for name in names:
        wl = W.CHUNK_CONFIGS[name]()
        runs = [_hash_outputs(run_chunk_raw(wl, torch)) for _ in range(2)]
        if side_stream:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                runs.append(_hash_outputs(run_chunk_raw(wl, torch)))
            s.synchronize()
        res[name] = runs
        del wl
    return res


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_gated_delta_06_gb300 import build
    build.build()


def test_fwd_bwd_hashes_agree_across_runs_streams_and_processes():
    here = workload_hashes(WORKLOADS)
    for name, runs in here.items():
        for i, r in enumerate(runs[1:], 1):
            assert r == runs[0], (name, i, [k for k in r if r[k] != runs[0][k]])
    code = ("import json, sys; sys.path[:0] = [%r, %r]; "
            "import test_gpu_determinism as t; "
            "print('HASHES ' + json.dumps(t.workload_hashes(%r, side_stream=False)))"
            % (os.path.join(ROOT, "tests"), ROOT, list(WORKLOADS)))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=1200,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    line = [x for x in r.stdout.splitlines() if x.startswith("HASHES ")][-1]
    there = json.loads(line[len("HASHES "):])
    for name in WORKLOADS:
        for i, h in enumerate(there[name]):
            assert h == here[name][0], (name, "other process", i,
                                        [k for k in h if h[k] != here[name][0][k]])
