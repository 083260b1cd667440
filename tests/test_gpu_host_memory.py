"""GPU parity with the inputs (and outputs) in pinned host memory.

The C ABI takes device pointers or pinned host pointers; the kernels read
pinned host arrays in place through their device mapping (plain loads
instead of bulk copies).  Every case here runs the same call on host-resident
and on device-resident tensors, compares the two outputs bit for bit and
compares the host run with the float64 oracle (decisions exact outside
flagged near-ties).  Pageable host memory must be refused before anything is
enqueued.

Source page: "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
(chzhyang.github.io), §1 (chain verification), §5 (DDTree, DSpark).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_sampling_gb300 as sv
import workloads
from gpu_util import assert_chain_parity, compare_exact, host, oracle_chain

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(autouse=True, scope="module")
def _built():
    sv.build()
    sv.set_tuning(0, 0)
    yield


def pin(t):
    return t.cpu().pin_memory()


def _same(a, b, keys):
    """bit-for-bit equal (NaN padding at the same places)"""
    for k in keys:
        x, y = getattr(a, k).cpu(), getattr(b, k).cpu()
        if x.is_floating_point():
            assert torch.equal(x.isnan(), y.isnan()), k
            x, y = x[~x.isnan()], y[~y.isnan()]
        assert torch.equal(x, y), k


@pytest.mark.parametrize("name,over", [("dflash", dict(B=16, V=40000)),      # fp32, top-k 50, 16-byte rows: TK rows
                                       ("eagle3", dict(B=12, V=12345)),      # bf16, untruncated, odd rows: SE/RESID/RESCAN
                                       ("chain_small", {})])
def test_chain_host_inputs(name, over):
    w = workloads.make_chain(name, device=DEV, **over)
    dev = sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k, diag=True)
    hl, hq, hd, hu = pin(w.logits), pin(w.q), pin(w.draft), pin(w.uniforms)
    r = sv.verify_chain(hl, hq, hd, hu, w.temperature, w.top_k, diag=True)
    torch.cuda.synchronize()
    assert sv.workspace_error(r.ws) == 0
    _same(r, dev, ("tokens", "num_accepted", "status", "diag"))
    assert_chain_parity(r, oracle_chain(w), w.K, draft=w.draft)


def test_chain_host_outputs():
    """Outputs written in place into pinned host tensors."""
    w = workloads.make_chain("dflash", device=DEV, B=8, V=20011)
    dev = sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k)
    B, K = w.B, w.K
    out = sv.ChainResult(torch.full((B, K + 1), -7, dtype=torch.int32).pin_memory(),
                         torch.full((B,), -7, dtype=torch.int32).pin_memory(),
                         torch.full((B,), -7, dtype=torch.int32).pin_memory(), None, None)
    r = sv.verify_chain(pin(w.logits), pin(w.q), pin(w.draft), pin(w.uniforms), w.temperature, w.top_k, out=out)
    torch.cuda.synchronize()
    assert r.tokens.device.type == "cpu"
    _same(r, dev, ("tokens", "num_accepted", "status"))


def test_greedy_host_inputs():
    w = workloads.make_chain("eagle3", device=DEV, B=16, V=20011)
    am = torch.argmax(w.logits[:, :w.K].float(), dim=-1).to(torch.int32)
    mix = torch.where(torch.rand(am.shape, device=DEV) < 0.7, am, w.draft_greedy).contiguous()
    dev = sv.verify_greedy(w.logits, mix)
    r = sv.verify_greedy(pin(w.logits), pin(mix))
    torch.cuda.synchronize()
    _same(r, dev, ("tokens", "num_accepted", "status"))
    compare_exact(r.tokens, r.num_accepted, oracle.verify_greedy(host(w.logits), host(mix)))


def test_tree_build_and_walk_host_inputs():
    t = workloads.make_tree("ddtree", device=DEV, B=6, L=8, V=20000, N=48)
    g_dev = sv.tree_build(t.q, t.budget)
    g = sv.tree_build(pin(t.q), t.budget)
    torch.cuda.synchronize()
    for k in ("token", "parent", "depth", "score", "anc_mask", "num_nodes", "status"):
        assert torch.equal(getattr(g, k), getattr(g_dev, k)), k
    ref_t = oracle.tree_build(host(t.q), t.budget)
    assert np.array_equal(g.token.cpu().numpy(), ref_t["token"])
    tl = workloads.tree_target_logits(t, g.depth)
    w_dev = sv.verify_tree(tl, g.token, g.parent, g.num_nodes, 8)
    w = sv.verify_tree(pin(tl), g.token, g.parent, g.num_nodes, 8)
    torch.cuda.synchronize()
    _same(w, w_dev, ("path_nodes", "tokens", "num_accepted", "status"))
    ref = oracle.verify_tree(host(tl), ref_t["token"], ref_t["parent"], ref_t["num_nodes"], 8)
    assert np.array_equal(w.tokens.cpu().numpy(), ref["tokens"])


def test_ragged_host_inputs():
    w = workloads.make_chain("dspark", device=DEV, B=24, V=30011)
    a = sv.adaptive_len(pin(w.conf), 1.0, 0.15)
    a_dev = sv.adaptive_len(w.conf, 1.0, 0.15)
    assert torch.equal(a.k, a_dev.k)
    pl, pq = workloads.pack_ragged(w.logits, w.q, a.k, a.l_row_off, a.q_row_off)
    dev = sv.verify_chain(pl, pq, w.draft, w.uniforms, w.temperature, w.top_k, k_per_req=a.k,
                          l_row_off=a.l_row_off, q_row_off=a.q_row_off)
    r = sv.verify_chain(pin(pl), pin(pq), pin(w.draft), pin(w.uniforms), w.temperature, w.top_k,
                        k_per_req=pin(a.k), l_row_off=pin(a.l_row_off), q_row_off=pin(a.q_row_off))
    torch.cuda.synchronize()
    _same(r, dev, ("tokens", "num_accepted", "status"))


def test_pageable_host_memory_is_refused():
    """The C ABI refuses a pointer into pageable host memory (numpy arrays)
    with SPEC_INVALID_ARG and enqueues nothing; the binding refuses
    unpinned host tensors itself."""
    w = workloads.make_chain("chain_small", device=DEV)
    lib = sv.lib()
    lg = np.ascontiguousarray(host(w.logits))
    r = sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k)   # outputs + workspace
    torch.cuda.synchronize()
    before = r.tokens.clone()
    B, K, V = w.B, w.K, w.V
    vp = ctypes.c_void_p
    rc = lib.spec_verify_chain(lg.ctypes.data_as(vp), 0, (K + 1) * V, V, vp(w.q.data_ptr()), K * V, V,
                               vp(w.draft.data_ptr()), vp(w.uniforms.data_ptr()), B, K, V, float(w.temperature),
                               int(w.top_k), None, None, None, vp(r.tokens.data_ptr()),
                               vp(r.num_accepted.data_ptr()), vp(r.status.data_ptr()), None,
                               vp(r.ws.data_ptr()), r.ws.numel(), vp(torch.cuda.current_stream().cuda_stream))
    assert rc == 1
    assert b"pageable" in lib.spec_last_error()
    torch.cuda.synchronize()
    assert torch.equal(r.tokens, before)
    with pytest.raises(sv.SpecError):
        sv.verify_chain(w.logits.cpu(), w.q, w.draft, w.uniforms, w.temperature, w.top_k)
