"""spec_verify_greedy_static: greedy verification for callers that cannot
allocate device memory when they verify (host callbacks, allocator-free
runtimes, plugins given raw buffers by an engine that owns all allocation).

The entry point takes its scratch space from a fixed array the library
reserves in device memory.  This test calls it through the C ABI, twice in a
row on different batches (the shared array keeps the previous call's
contents), and checks each result against spec_verify_greedy with its own
caller-provided workspace; greedy verification is exact, so the results must
be identical.  It lives in a file of its own, collected last, and builds and
loads the library itself, so it also runs alone in a fresh process."""
import ctypes

import pytest
import torch

import speculative_decoding_draft_sampling_gb300 as sv
import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _static_fn():
    sv.build()
    lib = sv.lib()
    f = lib.spec_verify_greedy_static
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [P, i32, i64, i64, P, i32, i32, i32, P, P, P, P, P, P]
    f.restype = ctypes.c_int
    return lib, f


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_static(f, lg, draft):
    B, K = draft.shape
    V = lg.shape[-1]
    tok = torch.full((B, K + 1), -7, dtype=torch.int32, device=DEV)
    n = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    st = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    ldt = 0 if lg.dtype == torch.float32 else 1
    rc = f(_p(lg), ldt, lg.stride(0), lg.stride(1), _p(draft), B, K, V, None, None,
           _p(tok), _p(n), _p(st), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, tok, n, st


def test_static_workspace_matches_caller_workspace_twice():
    lib, f = _static_fn()
    batches = []
    for seed, over in ((11, dict(B=48, V=50021)), (12, dict(B=20, K=5, V=12345))):
        w = workloads.make_chain("eagle3", device=DEV, seed=seed, **over)
        am = torch.argmax(w.logits[:, :w.K].float(), dim=-1).to(torch.int32)
        mix = torch.where(torch.rand(am.shape, device=DEV) < 0.7, am, w.draft).contiguous()
        batches.append((w.logits, mix))
    for lg, draft in batches:                       # two calls in a row
        rc, tok, n, st = _call_static(f, lg, draft)
        assert rc == 0, lib.spec_last_error()
        ref = sv.verify_greedy(lg, draft)           # caller-provided workspace
        torch.cuda.synchronize()
        assert torch.equal(tok, ref.tokens)
        assert torch.equal(n, ref.num_accepted)
        assert torch.equal(st, ref.status)


def test_static_workspace_limits():
    lib, f = _static_fn()
    # greedy scratch is a fixed control block: every batch within the
    # library's shape limits fits the 64 KiB array
    assert lib.spec_verify_greedy_workspace_size(1 << 20, 8, 151936) <= (64 << 10)
    # shapes beyond those limits are refused before any device work
    lg = torch.zeros((1, 1, 64), device=DEV)
    d = torch.zeros((1, 1), dtype=torch.int32, device=DEV)
    rc = f(_p(lg), 0, 0, 64, _p(d), 1, 4097, 64, None, None, _p(d), _p(d), _p(d), None)
    assert rc == 2
    assert b"K > 4096" in lib.spec_last_error()
    rc = f(_p(lg), 0, 0, 64, _p(d), 1, 1, 0, None, None, _p(d), _p(d), _p(d), None)
    assert rc == 1
