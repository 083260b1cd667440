"""GPU parity: the EAGLE-2 dynamic draft tree (expansion steps and rerank)
against the float64 oracle through the C ABI.

Source page: "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
(chzhyang.github.io), §4 "EAGLE-2".  Every step's node arrays, frontier and
status, and the final tree, are compared bit for bit: scores are the same
fp64 products of the same fp32 probabilities, and both orders (frontier:
score, then append order; rerank: score, depth, index) are total.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_sampling_gb300 as sv
import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
TREE_KEYS = ("token", "parent", "depth", "score", "anc_mask", "num_nodes", "status")


@pytest.fixture(autouse=True, scope="module")
def _built():
    sv.build()
    sv.set_tuning(0, 0)
    yield


def _paths(st, b):
    out = {0: ()}
    for i in range(1, int(st["num_gen"][b])):
        out[i] = out[int(st["parent"][b, i])] + (int(st["token"][b, i]),)
    return out


def _state_equal(o, g):
    for k in ("token", "parent", "depth", "score", "num_gen"):
        np.testing.assert_array_equal(getattr(g, k).cpu().numpy(), o[k], err_msg=k)


def _tree_equal(g, o):
    for k in TREE_KEYS:
        a = getattr(g, k).cpu().numpy()
        if k == "anc_mask":
            a = a.view(np.uint64)
        np.testing.assert_array_equal(a, o[k], err_msg=k)


def _run(B, V, K2, Fn, steps, G, budget, seed, rows=None):
    """Drive both sides through the same steps; rows(paths) -> q [B, F, V]."""
    if rows is None:
        rows = lambda paths: workloads.eagle2_rows(paths, V, seed, device=DEV)
    st_o = oracle.eagle_init(B, G)
    st_g = sv.eagle_state(B, G, DEV)
    fo = np.zeros((B, 1), np.int32)
    nfo = np.ones(B, np.int32)
    fg = torch.zeros((B, 1), dtype=torch.int32, device=DEV)
    nfg = torch.ones(B, dtype=torch.int32, device=DEV)
    ws = None
    for _ in range(steps):
        paths = []
        for b in range(B):
            pb = _paths(st_o, b)
            paths.append([pb[int(fo[b, f])] if f < nfo[b] else None for f in range(fo.shape[1])])
        q = rows(paths)
        fo, nfo, so = oracle.eagle_expand(q.cpu().numpy(), st_o, fo, nfo, K2, Fn)
        fg, nfg, sg = sv.eagle_expand(q, st_g, fg, nfg, K2, Fn, ws=ws)
        np.testing.assert_array_equal(fg.cpu().numpy(), fo)
        np.testing.assert_array_equal(nfg.cpu().numpy(), nfo)
        np.testing.assert_array_equal(sg.cpu().numpy(), so)
        _state_equal(st_o, st_g)
        if fo.shape[1] == 0:
            break
    t_o = oracle.eagle_rerank(st_o, budget)
    t_g = sv.eagle_rerank(st_g, budget)
    _tree_equal(t_g, t_o)
    return st_o, t_o


@pytest.mark.parametrize("B,V,K2,Fn,steps,G,budget", [
    (4, 3000, 4, 3, 4, 256, 20),
    (3, 5, 8, 6, 3, 64, 30),            # K2 > V: every token a child
    (2, 1000, 10, 10, 3, 40, 64),       # capacity reached; budget above the generated count
    (5, 20011, 7, 1, 5, 128, 9),        # a one-wide frontier (a greedy chain of best nodes)
    (2, 700, 3, 0, 2, 16, 4),           # Fn = 0: the first step's children only
])
def test_eagle_parity(B, V, K2, Fn, steps, G, budget):
    st, t = _run(B, V, K2, Fn, steps, G, budget, seed=B * 100 + V)
    if G == 40:
        assert (st["num_gen"] == 40).all()


def test_eagle_full_size():
    """The EAGLE-2 workload: B=32, V=151936, 10 children per node, frontier
    10, 6 steps, budget 60 -- every request compared."""
    cfg = workloads.DEFAULTS["eagle2"]
    B, V, K2, Fn, steps, N = cfg["B"], cfg["V"], cfg["K2"], cfg["Fn"], cfg["steps"], cfg["N"]
    G = 1 + K2 + (steps - 1) * Fn * K2
    st, t = _run(B, V, K2, Fn, steps, G, N, seed=workloads.seed_of("eagle2"))
    assert (st["num_gen"] == G).all()
    assert (t["num_nodes"] == N).all() and (t["depth"].max(axis=1) >= 2).all()


def test_eagle_bad_rows_and_ids():
    B, V, G = 3, 500, 64
    st_o = oracle.eagle_init(B, G)
    st_g = sv.eagle_state(B, G, DEV)
    g = torch.Generator(device="cpu").manual_seed(5)
    q = torch.softmax(torch.randn((B, 2, V), generator=g) * 3, dim=-1).float()
    q[1, 0, 17] = float("nan")                                # request 1: its root row is bad
    front = np.array([[0, 0], [0, 0], [0, 9]], np.int32)      # request 2: id 9 not generated yet
    nf = np.array([1, 1, 2], np.int32)
    fo, nfo, so = oracle.eagle_expand(q.numpy(), st_o, front, nf, 4, 3)
    fg, nfg, sg = sv.eagle_expand(q.to(DEV), st_g, torch.from_numpy(front).to(DEV), torch.from_numpy(nf).to(DEV), 4, 3)
    assert list(so) == [0, oracle.ST_BAD_ROW, oracle.ST_BAD_NODE]
    np.testing.assert_array_equal(sg.cpu().numpy(), so)
    np.testing.assert_array_equal(fg.cpu().numpy(), fo)
    np.testing.assert_array_equal(nfg.cpu().numpy(), nfo)
    _state_equal(st_o, st_g)


def test_eagle_factorised_rows_match_gpu_tree_build():
    """Rows that ignore the path: the rerank equals the GPU DDTree build."""
    B, L, V, N = 4, 5, 20000, 24
    t = workloads.make_tree("ddtree", device=DEV, B=B, L=L, V=V, N=N, seed=4242)

    def rows(paths):
        F = max(len(p) for p in paths)
        out = torch.zeros((B, F, V), dtype=torch.float32, device=DEV)
        for b in range(B):
            for f, p in enumerate(paths[b]):
                if p is not None:
                    out[b, f] = t.q[b, len(p)]
        return out

    _, te = _run(B, V, N - 1, N - 1, L, 1 + L * (N - 1) ** 2, N, seed=0, rows=rows)
    d = sv.tree_build(t.q, N)
    for k in TREE_KEYS:
        a = getattr(d, k).cpu().numpy()
        if k == "anc_mask":
            a = a.view(np.uint64)
        np.testing.assert_array_equal(a, te[k], err_msg=k)


def test_eagle_rerank_ties_and_inconsistent_parents():
    """Rerank alone on hand-made node arrays: equal scores at several depths,
    and a node whose parent index lies beyond the generated count."""
    B, G, N = 2, 12, 8
    st = oracle.eagle_init(B, G)
    # request 0: root -> 1, 2 (score .5 each); 1 -> 3 (q = 1: .5); 2 -> 4 (.25); 3 -> 5 (.5)
    st["token"][0, 1:6] = [3, 4, 5, 6, 7]
    st["parent"][0, 1:6] = [0, 0, 1, 2, 3]
    st["depth"][0, 1:6] = [1, 1, 2, 2, 3]
    st["score"][0, 1:6] = [.5, .5, .5, .25, .5]
    st["num_gen"][0] = 6
    # request 1: node 2's parent (11) was never generated
    st["token"][1, 1:4] = [1, 2, 3]
    st["parent"][1, 1:4] = [0, 11, 1]
    st["depth"][1, 1:4] = [1, 1, 2]
    st["score"][1, 1:4] = [.3, .9, .2]
    st["num_gen"][1] = 4
    ref = oracle.eagle_rerank(st, N)
    assert ref["status"][1] == oracle.ST_BAD_NODE and ref["num_nodes"][1] == 3
    assert list(ref["token"][0, :6]) == [-1, 3, 4, 5, 7, 6]
    g = sv.EagleState(*(torch.from_numpy(st[k]).to(DEV) for k in ("token", "parent", "depth", "score", "num_gen")))
    _tree_equal(sv.eagle_rerank(g, N), ref)


@pytest.mark.parametrize("g", [1025, 1026, 3000])
def test_eagle_rerank_large_node_counts(g):
    """Rerank of random consistent trees of a thousand nodes and more (a
    sorting network of 1024 to 4096 entries), with tied scores among
    siblings; three node counts per case."""
    B, G, N = 3, 4096, 200
    rng = np.random.default_rng(g)
    st = oracle.eagle_init(B, G)
    for b in range(B):
        par = np.zeros(g, np.int32)
        dep = np.zeros(g, np.int32)
        sc = np.ones(g, np.float64)
        for i in range(1, g):
            p = int(rng.integers(0, i))
            par[i], dep[i] = p, dep[p] + 1
            sc[i] = sc[p] * (0.5 if rng.random() < 0.2 else float(rng.uniform(0.05, 1.0)))
        st["token"][b, 1:g] = rng.integers(0, 50000, g - 1)
        st["parent"][b, 1:g] = par[1:]
        st["depth"][b, 1:g] = dep[1:]
        st["score"][b, 1:g] = sc[1:]
        st["num_gen"][b] = g - b          # three sizes per case
    ref = oracle.eagle_rerank(st, N)
    gs = sv.EagleState(*(torch.from_numpy(st[k]).to(DEV) for k in ("token", "parent", "depth", "score", "num_gen")))
    _tree_equal(sv.eagle_rerank(gs, N), ref)
