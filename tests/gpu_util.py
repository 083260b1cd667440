"""Helpers shared by the GPU parity tests: host copies for the oracle, the
oracle run over request chunks on every host core, and decision /
probability comparison with the near-tie rule.

Tolerances (fixed here, from the arithmetic): decisions (accepted count,
committed tokens, status bits) must be identical unless the oracle flags a
near-tie (|u - p/q| <= 1e-6 at an examined position, or the sample's target
within 1e-6 of a CDF boundary); probabilities and normalisers in `diag`
within 1e-5 relative (fp32 accumulation on the GPU against float64).  The
number of requests excused by a near-tie is itself bounded by every test
(near-ties occur with probability ~1e-6 per decision, so more than a couple
means the flags, not the kernel, decide the comparison).
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle

DIAG_RTOL = 1e-5


def max_near(B):
    """Requests a comparison of B requests may excuse as near-ties."""
    return max(2, B // 100)


def host(t: torch.Tensor) -> np.ndarray:
    """A host copy in the oracle's input format (bf16 as raw uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def run_chunks(fn, B, chunk=None):
    """fn(lo, hi) -> dict of per-request arrays, run over request chunks on
    the host cores (the oracle's ctypes calls release the GIL); the chunks'
    results are concatenated in request order."""
    if B == 0:
        return fn(0, 0)
    workers = max(1, min(os.cpu_count() or 1, 32))
    chunk = chunk or max(1, -(-B // (4 * workers)))
    spans = [(lo, min(B, lo + chunk)) for lo in range(0, B, chunk)]
    with ThreadPoolExecutor(max_workers=workers) as ex:
        parts = list(ex.map(lambda s: fn(*s), spans))
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}


def oracle_chain(w, idx=None, **kw):
    lg, q, d, u = w.logits, w.q, w.draft, w.uniforms
    if idx is not None:
        lg, q, d, u = lg[idx], q[idx], d[idx], u[idx]
    return oracle.verify_chain(host(lg), host(q), host(d), host(u), w.temperature, w.top_k, **kw)


def oracle_chain_all(w):
    """The oracle over every request of a dense chain workload."""
    lg, q, d, u = host(w.logits), host(w.q), host(w.draft), host(w.uniforms)
    return run_chunks(lambda a, b: oracle.verify_chain(lg[a:b], q[a:b], d[a:b], u[a:b], w.temperature, w.top_k),
                      w.B)


def compare_chain(res, ref, K, check_diag=True):
    """Returns (mismatches outside near-ties, mismatches at near-ties)."""
    tok = res.tokens.cpu().numpy()
    n = res.num_accepted.cpu().numpy()
    st = res.status.cpu().numpy()
    dg = res.diag.cpu().numpy() if (check_diag and res.diag is not None) else None
    bad, near = [], 0
    for b in range(tok.shape[0]):
        same = (n[b] == ref["num_accepted"][b] and (tok[b] == ref["tokens"][b]).all()
                and st[b] == ref["status"][b])
        if not same:
            if ref["near_tie"][b] != 0:
                near += 1
            else:
                bad.append(b)
            continue
        if dg is not None:
            rows = ref["rows_read"][b]
            for i in range(rows):
                want = ref["diag"][b, i]
                got = dg[b, i].astype(np.float64)
                if np.isnan(want).all():
                    continue
                for j in range(4):
                    if not np.isclose(got[j], want[j], rtol=DIAG_RTOL, atol=1e-30):
                        bad.append((b, i, j, float(got[j]), float(want[j])))
    return bad, near


def assert_chain_parity(res, ref, K, check_diag=True, draft=None):
    """Every request compared; near-ties counted and bounded; a request
    excused by a near-tie must still be a valid outcome."""
    bad, near = compare_chain(res, ref, K, check_diag)
    assert not bad, bad[:5]
    B = res.tokens.shape[0]
    assert near <= max_near(B), (near, B)
    if draft is not None:
        tok = res.tokens.cpu().numpy()
        n = res.num_accepted.cpu().numpy()
        d = draft.cpu().numpy()
        for b in range(B):
            assert (tok[b, :n[b]] == d[b, :n[b]]).all()
            assert (tok[b, n[b] + 1:] == -1).all()
    return near


def compare_exact(res_tokens, res_n, ref):
    tok = res_tokens.cpu().numpy()
    n = res_n.cpu().numpy()
    assert np.array_equal(n, ref["num_accepted"]), (n, ref["num_accepted"])
    assert np.array_equal(tok, ref["tokens"])
