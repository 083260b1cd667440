"""Failure detection on the GPU without a fault: a bounded device wait that
runs out must end the kernel with the workspace error set, and the context
must stay usable.

A failure-path build of the library (-DSPEC_TEST_HOOKS, waits limited to
50 ms) can drop the first job one combiner would post, so that the waits
depending on it (the producer's mailbox poll, the consumers' queue wait, the
combiner's arrival wait) never complete.  Every one of them is bounded: it
gives up, raises the CTA's abort flag and the workspace error word, and
every role loop leaves; the kernel returns.  The test runs in a child
process (its own CUDA context and its own copy of the library), checks the
error word, then runs the same call with the hook off on the same context
and requires the normal result.
"""
import json
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import ctypes, json, sys, time
    sys.path.insert(0, sys.argv[2])
    import torch
    import speculative_decoding_draft_sampling_gb300 as sv
    from speculative_decoding_draft_sampling_gb300 import _build
    import workloads
    lib = _build.build(force=True, extra_flags=["-DSPEC_TEST_HOOKS", "-DSPEC_WAIT_LIMIT_NS=50000000ull"],
                       out=sys.argv[1])
    sv.LIB_PATH = lib
    sv._lib = None
    L = sv.lib()
    L.spec_test_drop_first_post.argtypes = [ctypes.c_int]
    L.spec_test_drop_first_post.restype = ctypes.c_int
    dev = torch.device("cuda", 0)
    w = workloads.make_chain("dflash", device=dev, B=8, V=5003)
    args = (w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k)
    ref = sv.verify_chain(*args)
    torch.cuda.synchronize()
    e0 = sv.workspace_error(ref.ws)
    assert L.spec_test_drop_first_post(1) == 0
    t0 = time.perf_counter()
    bad = sv.verify_chain(*args)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    e1 = sv.workspace_error(bad.ws)
    assert L.spec_test_drop_first_post(0) == 0
    again = sv.verify_chain(*args)
    torch.cuda.synchronize()
    e2 = sv.workspace_error(again.ws)
    same = bool(torch.equal(again.tokens, ref.tokens) and torch.equal(again.num_accepted, ref.num_accepted)
                and torch.equal(again.status, ref.status))
    print(json.dumps(dict(e0=e0, e1=e1, e2=e2, same=same, seconds=dt)))
""")


def test_bounded_wait_runs_out_and_reports(tmp_path):
    script = tmp_path / "child.py"
    script.write_text(CHILD)
    r = subprocess.run([sys.executable, str(script), str(tmp_path / "libspecverify_hooks.so"), ROOT],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    res = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    assert res["e0"] == 0
    assert res["e1"] & 1, res              # SPEC_WS_ERR_WAIT: a wait gave up
    assert res["seconds"] < 30.0, res     # the kernel returned after its waits ran out
    assert res["e2"] == 0 and res["same"], res
