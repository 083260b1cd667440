"""Float64 CPU oracle for batched speculative-sampling verification.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may import this
package.  It shares no code with the CUDA library in
``speculative_decoding_draft_sampling_gb300``; the only thing both sides see
is the seeded input generator in ``workloads``.

The arithmetic lives in ``spec_oracle.c`` (plain C99, double precision,
scalar loops, compiled with ``-ffp-contract=off``).  This module compiles it
with gcc on first use and wraps each function for numpy arrays.

Source page: "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
(Speculative decoding for LLMs: Medusa, MTP, EAGLE, DFlash, DDTree and
DSpark), chzhyang.github.io -- §1 (acceptance rule, residual and bonus
samples, greedy consistency), §5 (DDTree Q(u) and best-first heap, tree
walk; DSpark s_j and expected advance).

Parity pins live in ``tests/test_oracle_pins.py``; none of the oracle's
functions is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIBDIR = os.path.join(_HERE, "lib")
_LIB = os.path.join(_LIBDIR, "libspec_oracle.so")
_lock = threading.Lock()
_lib = None

ST_BAD_ROW, ST_Q_ZERO, ST_R_ZERO, ST_BAD_TOKEN, ST_BAD_K = 1, 2, 4, 8, 16
ST_TREE_FULL, ST_BAD_NODE = 32, 64
NEAR_TIE_SAMPLE_BIT = 1 << 31
MAX_BUDGET = 256   # ranks are stored in one byte per depth


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C99, no fused multiply-add)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC),
                                              os.path.getmtime(os.path.join(_HERE, "spec_oracle.h")))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
            lib.oracle_verify_chain.argtypes = [P, i32, i64, i64, P, i64, i64, P, P,
                                                i32, i32, i32, f32, i32, P, P, P,
                                                P, P, P, P, P, P]
            lib.oracle_verify_chain.restype = None
            lib.oracle_verify_greedy.argtypes = [P, i32, i64, i64, P, i32, i32, i32,
                                                 P, P, P, P, P, P]
            lib.oracle_verify_greedy.restype = None
            lib.oracle_tree_build.argtypes = [P, i64, i64, i32, i32, i32, i32,
                                              P, P, P, P, P, P, P, P]
            lib.oracle_tree_build.restype = None
            lib.oracle_tree_build_bruteforce.argtypes = [P, i64, i64, i32, i32, i32, i32, i64,
                                                         P, P, P, P, P, P]
            lib.oracle_tree_build_bruteforce.restype = ctypes.c_int
            lib.oracle_verify_tree.argtypes = [P, i32, i64, i64, P, P, P, i32, i32, i32, i32,
                                               P, P, P, P]
            lib.oracle_verify_tree.restype = None
            lib.oracle_verify_tree_sample.argtypes = [P, i32, i64, i64, P, P, P, P, i32, i32, i32, i32,
                                                      f32, i32, P, P, P, P, P]
            lib.oracle_verify_tree_sample.restype = None
            lib.oracle_adaptive_len.argtypes = [P, i32, i32, f32, f32, P, P, P, P, P, P, P]
            lib.oracle_kv_compact.argtypes = [P, i64, i64, i64, P, i64, i64, i64, i32, i32, i32, i64,
                                              P, i32, P, P]
            lib.oracle_kv_compact.restype = None
            lib.oracle_adaptive_len.restype = None
            lib.oracle_eagle_expand.argtypes = [P, i64, i64, i32, i32, i32, i32, i32, i32,
                                                P, P, P, P, P, P, P, P, P, P]
            lib.oracle_eagle_expand.restype = None
            lib.oracle_eagle_rerank.argtypes = [P, P, P, P, P, i32, i32, i32, P, P, P, P, P, P, P]
            lib.oracle_eagle_rerank.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits_arg(logits):
    """fp32 array, or bf16 given as uint16/int16 raw bits."""
    a = np.ascontiguousarray(logits)
    if a.dtype == np.float32:
        return a, 0
    if a.dtype in (np.uint16, np.int16):
        return a.view(np.uint16), 1
    raise TypeError(f"logits must be float32 or bf16 bits (uint16), got {a.dtype}")


def verify_chain(logits, q, draft, uniforms, temperature, top_k=0, *,
                 K=None, V=None, k_per_req=None, l_row_off=None, q_row_off=None,
                 l_strides=None, q_strides=None):
    """Chain speculative sampling, per request (page §1).

    Dense: logits [B, K+1, V], q [B, K, V].  Ragged: logits packed rows
    [sum(k_b+1), V], q packed rows [sum(k_b), V] with exclusive offsets;
    k_per_req without offsets keeps the dense rows and caps each request at
    its k_b (page §9 "cap-accept").
    ``l_strides`` / ``q_strides`` = (batch, row) element strides override the
    contiguous defaults (batch stride 0 broadcasts one set of rows).
    Returns a dict of numpy arrays: tokens [B, K+1], num_accepted, status,
    diag [B, K+1, 4] (NaN where not examined), near_tie, rows_read.
    """
    lib = _load()
    la, ldt = _logits_arg(logits)
    qa = np.ascontiguousarray(q, dtype=np.float32)
    d = np.ascontiguousarray(draft, dtype=np.int32)
    u = np.ascontiguousarray(uniforms, dtype=np.float32)
    B = d.shape[0]
    K = d.shape[1] if K is None else K
    V = la.shape[-1] if V is None else V
    if l_strides is None:
        l_strides = ((K + 1) * V, V)
    if q_strides is None:
        q_strides = (K * V, V)
    kp = lo = qo = None
    if k_per_req is not None:
        kp = np.ascontiguousarray(k_per_req, dtype=np.int32)
        if l_row_off is not None:        # packed rows ("compact")
            lo = np.ascontiguousarray(l_row_off, dtype=np.int32)
            qo = np.ascontiguousarray(q_row_off, dtype=np.int32)
            l_strides = (0, V) if l_strides is None else (0, l_strides[1])
            q_strides = (0, V) if q_strides is None else (0, q_strides[1])
    tok = np.empty((B, K + 1), np.int32)
    n = np.empty(B, np.int32)
    st = np.empty(B, np.int32)
    diag = np.full((B, K + 1, 4), np.nan, np.float64)
    nt = np.empty(B, np.int32)
    rr = np.empty(B, np.int32)
    lib.oracle_verify_chain(_ptr(la), ldt, l_strides[0], l_strides[1],
                            _ptr(qa), q_strides[0], q_strides[1],
                            _ptr(d), _ptr(u), B, K, V, float(temperature), int(top_k),
                            _ptr(kp), _ptr(lo), _ptr(qo),
                            _ptr(tok), _ptr(n), _ptr(st), _ptr(diag), _ptr(nt), _ptr(rr))
    return dict(tokens=tok, num_accepted=n, status=st, diag=diag,
                near_tie=nt.view(np.uint32), rows_read=rr)


def verify_greedy(logits, draft, *, K=None, V=None, k_per_req=None, l_row_off=None,
                  l_strides=None):
    """Greedy argmax-match verification (page §1, greedy consistency)."""
    lib = _load()
    la, ldt = _logits_arg(logits)
    d = np.ascontiguousarray(draft, dtype=np.int32)
    B = d.shape[0]
    K = d.shape[1] if K is None else K
    V = la.shape[-1] if V is None else V
    if l_strides is None:
        l_strides = ((K + 1) * V, V)
    kp = lo = None
    if k_per_req is not None:
        kp = np.ascontiguousarray(k_per_req, dtype=np.int32)
        if l_row_off is not None:
            lo = np.ascontiguousarray(l_row_off, dtype=np.int32)
            l_strides = (0, l_strides[1])
    tok = np.empty((B, K + 1), np.int32)
    n = np.empty(B, np.int32)
    st = np.empty(B, np.int32)
    rr = np.empty(B, np.int32)
    lib.oracle_verify_greedy(_ptr(la), ldt, l_strides[0], l_strides[1], _ptr(d), B, K, V,
                             _ptr(kp), _ptr(lo), _ptr(tok), _ptr(n), _ptr(st), _ptr(rr))
    return dict(tokens=tok, num_accepted=n, status=st, rows_read=rr)


def _tree_out(B, N):
    W = (N + 63) // 64
    return dict(token=np.empty((B, N), np.int32), parent=np.empty((B, N), np.int32),
                depth=np.empty((B, N), np.int32), score=np.empty((B, N), np.float64),
                anc_mask=np.empty((B, N, W), np.uint64), num_nodes=np.empty(B, np.int32))


def tree_build(q, budget, *, q_strides=None):
    """DDTree best-first tree over per-depth marginals q [B, L, V] (page §5)."""
    lib = _load()
    qa = np.ascontiguousarray(q, dtype=np.float32)
    B, L, V = qa.shape
    if not 1 <= budget <= MAX_BUDGET:
        raise ValueError("budget must be in [1, 256]")
    if q_strides is None:
        q_strides = (L * V, V)
    o = _tree_out(B, budget)
    o["status"] = np.empty(B, np.int32)
    o["rows_needed"] = np.empty(B, np.int32)
    lib.oracle_tree_build(_ptr(qa), q_strides[0], q_strides[1], B, L, V, budget,
                          _ptr(o["token"]), _ptr(o["parent"]), _ptr(o["depth"]),
                          _ptr(o["score"]), _ptr(o["anc_mask"]), _ptr(o["num_nodes"]),
                          _ptr(o["status"]), _ptr(o["rows_needed"]))
    return o


def tree_build_bruteforce(q, budget, max_prefixes=1 << 20):
    """Every prefix enumerated, sorted, first ``budget`` kept (tiny V, L)."""
    lib = _load()
    qa = np.ascontiguousarray(q, dtype=np.float32)
    B, L, V = qa.shape
    o = _tree_out(B, budget)
    rc = lib.oracle_tree_build_bruteforce(_ptr(qa), L * V, V, B, L, V, budget, int(max_prefixes),
                                          _ptr(o["token"]), _ptr(o["parent"]), _ptr(o["depth"]),
                                          _ptr(o["score"]), _ptr(o["anc_mask"]),
                                          _ptr(o["num_nodes"]))
    if rc != 0:
        raise RuntimeError(f"brute force failed (rc={rc})")
    return o


def verify_tree(logits, token, parent, num_nodes, max_depth, *, l_strides=None):
    """Greedy tree walk over target logits [B, N, V] (page §5, DDTree)."""
    lib = _load()
    la, ldt = _logits_arg(logits)
    tk = np.ascontiguousarray(token, dtype=np.int32)
    pr = np.ascontiguousarray(parent, dtype=np.int32)
    nn = np.ascontiguousarray(num_nodes, dtype=np.int32)
    B, N = tk.shape
    V = la.shape[-1]
    if l_strides is None:
        l_strides = (N * V, V)
    pn = np.empty((B, max_depth + 1), np.int32)
    ot = np.empty((B, max_depth + 1), np.int32)
    na = np.empty(B, np.int32)
    st = np.empty(B, np.int32)
    lib.oracle_verify_tree(_ptr(la), ldt, l_strides[0], l_strides[1], _ptr(tk), _ptr(pr),
                           _ptr(nn), B, N, V, max_depth, _ptr(pn), _ptr(ot), _ptr(na), _ptr(st))
    return dict(path_nodes=pn, tokens=ot, num_accepted=na, status=st)


def verify_tree_sample(logits, token, parent, num_nodes, uniforms, max_depth, temperature, top_k=0, *,
                       l_strides=None):
    """Stochastic tree walk over target logits [B, N, V]: at depth d the
    current node's token is drawn from its p with uniforms[b, d] (page §1,
    §5 DDTree)."""
    lib = _load()
    la, ldt = _logits_arg(logits)
    tk = np.ascontiguousarray(token, dtype=np.int32)
    pr = np.ascontiguousarray(parent, dtype=np.int32)
    nn = np.ascontiguousarray(num_nodes, dtype=np.int32)
    u = np.ascontiguousarray(uniforms, dtype=np.float32)
    B, N = tk.shape
    V = la.shape[-1]
    if l_strides is None:
        l_strides = (N * V, V)
    assert u.shape == (B, max_depth + 1)
    pn = np.empty((B, max_depth + 1), np.int32)
    ot = np.empty((B, max_depth + 1), np.int32)
    na = np.empty(B, np.int32)
    st = np.empty(B, np.int32)
    nt = np.empty(B, np.int32)
    lib.oracle_verify_tree_sample(_ptr(la), ldt, l_strides[0], l_strides[1], _ptr(tk), _ptr(pr), _ptr(nn), _ptr(u),
                                  B, N, V, max_depth, float(temperature), int(top_k),
                                  _ptr(pn), _ptr(ot), _ptr(na), _ptr(st), _ptr(nt))
    return dict(path_nodes=pn, tokens=ot, num_accepted=na, status=st, near_tie=nt.view(np.uint32))


def kv_compact(src, dst, path_nodes, num_accepted, dst_pos=None):
    """Accepted-path KV compaction (page §5, DDTree): src [P, B, N, R] and
    dst [P, B, M, R] arrays of any dtype (rows of R elements); returns a copy
    of dst where row dst_pos[b] + j of every plane holds src row
    path_nodes[b, j], j = 0..num_accepted[b]."""
    lib = _load()
    s = np.ascontiguousarray(src)
    d = np.array(dst, copy=True, order="C")
    assert s.dtype == d.dtype and s.ndim == 4 and d.ndim == 4
    P, B, N, R = s.shape
    es = s.itemsize
    pn = np.ascontiguousarray(path_nodes, dtype=np.int32)
    na = np.ascontiguousarray(num_accepted, dtype=np.int32)
    dp = None if dst_pos is None else np.ascontiguousarray(dst_pos, dtype=np.int32)
    lib.oracle_kv_compact(s.ctypes.data_as(ctypes.c_void_p), s.strides[0], s.strides[1], s.strides[2],
                          d.ctypes.data_as(ctypes.c_void_p), d.strides[0], d.strides[1], d.strides[2],
                          P, B, N, R * es, _ptr(pn), pn.shape[1], _ptr(na), _ptr(dp))
    return d


def eagle_init(B, G):
    """EAGLE-2 node arrays of capacity G holding only the root (page §4)."""
    st = dict(token=np.full((B, G), -1, np.int32), parent=np.full((B, G), -1, np.int32),
              depth=np.full((B, G), -1, np.int32), score=np.zeros((B, G), np.float64),
              num_gen=np.ones(B, np.int32))
    st["depth"][:, 0] = 0
    st["score"][:, 0] = 1.0
    return st


def eagle_expand(q, state, front, num_front, K2, Fn):
    """One EAGLE-2 expansion step (page §4): q [B, F, V] holds the draft's
    conditional rows of the frontier nodes front [B, F] (num_front valid).
    Updates `state` in place; returns (front_out [B, Fn], num_front_out [B],
    status [B])."""
    lib = _load()
    qa = np.ascontiguousarray(q, dtype=np.float32)
    B, F, V = qa.shape
    G = state["token"].shape[1]
    fi = np.ascontiguousarray(front, dtype=np.int32)
    nfi = np.ascontiguousarray(num_front, dtype=np.int32)
    assert fi.shape == (B, F)
    fo = np.empty((B, Fn), np.int32)
    nfo = np.empty(B, np.int32)
    st = np.empty(B, np.int32)
    for key in ("token", "parent", "depth", "num_gen"):
        assert state[key].dtype == np.int32 and state[key].flags.c_contiguous
    lib.oracle_eagle_expand(_ptr(qa), F * V, V, B, F, V, K2, Fn, G,
                            _ptr(state["token"]), _ptr(state["parent"]), _ptr(state["depth"]),
                            _ptr(state["score"]), _ptr(state["num_gen"]), _ptr(fi), _ptr(nfi),
                            _ptr(fo), _ptr(nfo), _ptr(st))
    return fo, nfo, st


def eagle_rerank(state, budget):
    """EAGLE-2 rerank (page §4): the root and the budget-1 best generated
    nodes as a verification tree (outputs as tree_build)."""
    lib = _load()
    B, G = state["token"].shape
    o = _tree_out(B, budget)
    o["status"] = np.empty(B, np.int32)
    lib.oracle_eagle_rerank(_ptr(state["token"]), _ptr(state["parent"]), _ptr(state["depth"]),
                            _ptr(state["score"]), _ptr(state["num_gen"]), B, G, budget,
                            _ptr(o["token"]), _ptr(o["parent"]), _ptr(o["depth"]), _ptr(o["score"]),
                            _ptr(o["anc_mask"]), _ptr(o["num_nodes"]), _ptr(o["status"]))
    return o


def adaptive_len(conf, a, b, cost=None):
    """DSpark survival, expected advance and verify length (page §5); the
    cost of k positions is a + b*k, or cost[k] with a table (page §9)."""
    lib = _load()
    c = np.ascontiguousarray(conf, dtype=np.float32)
    B, Kmax = c.shape
    ct = None
    if cost is not None:
        ct = np.ascontiguousarray(cost, dtype=np.float64)
        assert ct.shape == (Kmax + 1,)
    k = np.empty(B, np.int32)
    surv = np.empty((B, Kmax), np.float64)
    adv = np.empty(B, np.float64)
    lo = np.empty(B + 1, np.int32)
    qo = np.empty(B + 1, np.int32)
    nt = np.empty(B, np.int32)
    lib.oracle_adaptive_len(_ptr(c), B, Kmax, float(a), float(b), _ptr(ct), _ptr(k), _ptr(surv),
                            _ptr(adv), _ptr(lo), _ptr(qo), _ptr(nt))
    return dict(k=k, surv=surv, exp_adv=adv, l_row_off=lo, q_row_off=qo, near_tie=nt)
