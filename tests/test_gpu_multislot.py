"""GPU parity with several request slots per CTA.

The default launch plan gives every CTA one request slot, so the engine's
paths for a CTA that leads several slots -- the combiner polling several
arrival barriers, several slots' jobs interleaved in one CTA's ring, and the
DDTree enumeration state saved to and restored from the workspace between
rows -- run only under the tuning set here.  Batches are large enough that
a cluster holds more slots than it has CTAs; rows are short so the oracle
finishes in seconds.

Source page: "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
(chzhyang.github.io), §1 (chain verify), §4 (EAGLE-2), §5 (DDTree).
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_sampling_gb300 as sv
import workloads
from gpu_util import assert_chain_parity, compare_exact, host, oracle_chain_all, run_chunks

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
TREE_KEYS = ("token", "parent", "depth", "score", "anc_mask", "num_nodes", "status")
# (CTAs per cluster, slots per CTA)
TUNINGS = [(2, 2), (2, 4), (4, 2)]


@pytest.fixture(autouse=True)
def _tuning_reset():
    sv.build()
    sv.set_tuning(0, 0)
    yield
    sv.set_tuning(0, 0)


@pytest.mark.parametrize("C,spc", TUNINGS)
@pytest.mark.parametrize("name,over", [("dflash", dict(B=320, V=20011)),
                                       ("eagle3", dict(B=320, V=12347)),
                                       ("dspark", dict(B=320, V=9001))])
def test_chain_parity_several_slots(name, over, C, spc):
    sv.set_tuning(C, spc)
    w = workloads.make_chain(name, device=DEV, seed=workloads.seed_of(name) + 101, **over)
    r = sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k)
    torch.cuda.synchronize()
    ref = oracle_chain_all(w)
    assert_chain_parity(r, ref, w.K, check_diag=False, draft=w.draft)
    assert sv.workspace_error(r.ws) == 0


@pytest.mark.parametrize("C,spc", TUNINGS)
def test_greedy_parity_several_slots(C, spc):
    sv.set_tuning(C, spc)
    w = workloads.make_chain("eagle3", device=DEV, B=320, V=12347, seed=workloads.seed_of("eagle3") + 7)
    am = torch.argmax(w.logits[:, :w.K].float(), dim=-1).to(torch.int32)
    mix = torch.where(torch.rand(w.draft.shape, device=DEV) < 0.7, am, w.draft_greedy).contiguous()
    r = sv.verify_greedy(w.logits, mix)
    lg, mh = host(w.logits), host(mix)
    ref = run_chunks(lambda a, b: oracle.verify_greedy(lg[a:b], mh[a:b]), w.B)
    compare_exact(r.tokens, r.num_accepted, ref)
    assert np.array_equal(r.status.cpu().numpy(), ref["status"])
    assert sv.workspace_error(r.ws) == 0


@pytest.mark.parametrize("C,spc", [(2, 2), (4, 2)])
def test_tree_build_and_walk_several_slots(C, spc):
    sv.set_tuning(C, spc)
    B, L, V, N = 200, 8, 3001, 24
    t = workloads.make_tree("ddtree", device=DEV, B=B, L=L, V=V, N=N, seed=4242)
    g = sv.tree_build(t.q, t.budget)
    qh = host(t.q)
    ref = run_chunks(lambda a, b: oracle.tree_build(qh[a:b], t.budget), B)
    for k in TREE_KEYS:
        a = getattr(g, k).cpu().numpy()
        if k == "anc_mask":
            a = a.view(np.uint64)
        assert np.array_equal(a, ref[k]), k
    assert sv.workspace_error(g.ws) == 0
    tl = workloads.tree_target_logits(t, g.depth)
    w = sv.verify_tree(tl, g.token, g.parent, g.num_nodes, L)
    tlh = host(tl)
    rw = run_chunks(lambda a, b: oracle.verify_tree(tlh[a:b], ref["token"][a:b], ref["parent"][a:b],
                                                    ref["num_nodes"][a:b], L), B)
    for k in ("path_nodes", "tokens", "num_accepted", "status"):
        assert np.array_equal(getattr(w, k).cpu().numpy(), rw[k]), k
    assert sv.workspace_error(w.ws) == 0
