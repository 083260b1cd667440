"""Helpers shared by the GPU parity tests: host copies for the oracle and
decision / probability comparison with the near-tie rule.

Tolerances (fixed here, from the arithmetic): decisions (accepted count,
committed tokens, status bits) must be identical unless the oracle flags a
near-tie (|u - p/q| <= 1e-6 at an examined position, or the sample's target
within 1e-6 of a CDF boundary); probabilities and normalisers in `diag`
within 1e-5 relative (fp32 accumulation on the GPU against float64).
"""
import numpy as np
import torch

import oracle

DIAG_RTOL = 1e-5


def host(t: torch.Tensor) -> np.ndarray:
    """A host copy in the oracle's input format (bf16 as raw uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def oracle_chain(w, idx=None, **kw):
    lg, q, d, u = w.logits, w.q, w.draft, w.uniforms
    if idx is not None:
        lg, q, d, u = lg[idx], q[idx], d[idx], u[idx]
    return oracle.verify_chain(host(lg), host(q), host(d), host(u), w.temperature, w.top_k, **kw)


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


def compare_exact(res_tokens, res_n, ref):
    tok = res_tokens.cpu().numpy()
    n = res_n.cpu().numpy()
    assert np.array_equal(n, ref["num_accepted"]), (n, ref["num_accepted"])
    assert np.array_equal(tok, ref["tokens"])
