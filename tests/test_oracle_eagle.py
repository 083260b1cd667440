"""Pins for the oracle's EAGLE-2 dynamic draft tree (expand and rerank).

Source page: "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
(chzhyang.github.io), §4 "EAGLE-2": the branches of highest cumulative path
confidence are expanded, every candidate is then reranked and the best form
the tree to verify; depth and width follow the context.  §5 "DDTree" gives
the factorised special case: with per-depth marginals that do not depend on
the path, the best nodes by cumulative score are the DDTree best-first tree.

What the pins catch: a child scored by its own probability instead of the
product along its path, a parent or depth off by one, children that are not
the row's most probable tokens, a frontier chosen by local instead of
cumulative confidence, a rerank that drops the depth tie rule or emits a
child before its parent, and the capacity / bad-row status bits.
"""
import itertools

import numpy as np
import pytest

import oracle


def _paths(state, b):
    """token path of every generated node of request b"""
    out = {0: ()}
    for i in range(1, state["num_gen"][b]):
        out[i] = out[state["parent"][b, i]] + (int(state["token"][b, i]),)
    return out


def _drive(cond, B, V, L, K2, Fn, G):
    """Run L expansion steps; cond(b, path) -> the draft's row after path."""
    st = oracle.eagle_init(B, G)
    front = np.zeros((B, 1), np.int32)
    nf = np.ones(B, np.int32)
    statuses = []
    for _ in range(L):
        F = front.shape[1]
        q = np.zeros((B, F, V), np.float32)
        for b in range(B):
            paths = _paths(st, b)
            for f in range(nf[b]):
                q[b, f] = cond(b, paths[int(front[b, f])])
        front, nf, s = oracle.eagle_expand(q, st, front, nf, K2, Fn)
        statuses.append(s)
    return st, statuses


def _tables(rng, B, V, L):
    """a random conditional row for every path of length < L"""
    tab = {}
    for b in range(B):
        for d in range(L):
            for path in itertools.product(range(V), repeat=d):
                tab[(b, path)] = rng.dirichlet(np.ones(V) * 0.7).astype(np.float32)
    return tab


@pytest.mark.parametrize("V,L,budget", [(3, 3, 8), (3, 3, 40), (4, 2, 11), (2, 4, 9)])
def test_full_expansion_equals_bruteforce_topn(V, L, budget):
    """With every child kept and every node expanded the generated set is all
    paths of length <= L; the rerank must equal the brute force over them:
    score = product of the conditional probabilities along the path, sorted
    by score, then depth."""
    rng = np.random.default_rng(500 + V * 10 + L)
    B = 3
    tab = _tables(rng, B, V, L)
    st, _ = _drive(lambda b, p: tab[(b, p)], B, V, L, K2=V, Fn=V ** L, G=2048)
    t = oracle.eagle_rerank(st, budget)
    for b in range(B):
        cand = []
        for d in range(1, L + 1):
            for path in itertools.product(range(V), repeat=d):
                s = 1.0
                for i in range(d):
                    s *= float(tab[(b, path[:i])][path[i]])
                cand.append((-s, d, path))
        cand.sort()
        want = [()] + [c[2] for c in cand[: budget - 1]]
        got = []
        for n in range(t["num_nodes"][b]):
            path = ()
            m = n
            while m > 0:
                path = (int(t["token"][b, m]),) + path
                m = t["parent"][b, m]
            got.append(path)
        assert got == want
        np.testing.assert_allclose(t["score"][b, 1:t["num_nodes"][b]], [-c[0] for c in cand[: budget - 1]],
                                   rtol=1e-12)
        assert t["num_nodes"][b] == min(budget, 1 + len(cand))


def test_factorised_rows_reproduce_the_ddtree_tree():
    """Marginals that ignore the path: with K2 = Fn = budget - 1 (wide enough
    to hold every node of the best budget - 1) the rerank is the DDTree
    best-first tree of the same marginals, node for node."""
    rng = np.random.default_rng(77)
    B, L, V, N = 4, 5, 300, 24
    q = rng.random((B, L, V)) ** 6
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    st, _ = _drive(lambda b, p: q[b, len(p)], B, V, L, K2=N - 1, Fn=N - 1, G=1 + L * (N - 1) ** 2)
    e = oracle.eagle_rerank(st, N)
    d = oracle.tree_build(q, N)
    for key in ("token", "parent", "depth", "score", "anc_mask", "num_nodes"):
        np.testing.assert_array_equal(e[key], d[key], err_msg=key)


def test_hand_example_frontier_follows_cumulative_confidence():
    """V = 4, K2 = 2.  Root row [.5 .3 .2 0] -> children A=0 (.5), B=1 (.3);
    Fn = 2 keeps both.  Row after A: [.3 .3 .4 0] -> A2 (.2), A0 (.15; the
    tie .3/.3 goes to the lower id).  Row after B: [.6 .4 0 0] -> B0 (.18),
    B1 (.12).  With Fn = 1 the next frontier is A2 (.2), although B's row
    holds the larger local probability (.6).  Rerank with budget 4: root, A,
    B, A2."""
    rows = {(): [.5, .3, .2, 0.], (0,): [.3, .3, .4, 0.], (1,): [.6, .4, 0., 0.]}
    st = oracle.eagle_init(1, 16)
    q1 = np.array([[rows[()]]], np.float32)
    f1, n1, s1 = oracle.eagle_expand(q1, st, np.zeros((1, 1), np.int32), np.ones(1, np.int32), 2, 2)
    assert n1[0] == 2 and list(f1[0]) == [1, 2] and s1[0] == 0
    assert list(st["token"][0, 1:3]) == [0, 1]
    q2 = np.array([[rows[(0,)], rows[(1,)]]], np.float32)
    f2, n2, s2 = oracle.eagle_expand(q2, st, f1, n1, 2, 1)
    assert st["num_gen"][0] == 7
    assert list(st["token"][0, 3:7]) == [2, 0, 0, 1]
    assert list(st["parent"][0, 3:7]) == [1, 1, 2, 2]
    assert list(st["depth"][0, :7]) == [0, 1, 1, 2, 2, 2, 2]
    f32 = np.float32
    np.testing.assert_array_equal(st["score"][0, 3:7], [float(f32(.5)) * float(f32(.4)), float(f32(.5)) * float(f32(.3)),
                                                        float(f32(.3)) * float(f32(.6)), float(f32(.3)) * float(f32(.4))])
    assert n2[0] == 1 and f2[0, 0] == 3
    t = oracle.eagle_rerank(st, 4)
    assert t["num_nodes"][0] == 4
    assert list(t["token"][0]) == [-1, 0, 1, 2]
    assert list(t["parent"][0]) == [-1, 0, 0, 1]
    assert list(t["depth"][0]) == [0, 1, 1, 2]


def test_rerank_prefers_the_shallower_node_on_equal_scores():
    """q = 1 on a child gives it its parent's score: the parent (shallower)
    comes first, so a child never precedes its parent."""
    st = oracle.eagle_init(1, 16)
    f1, n1, _ = oracle.eagle_expand(np.array([[[0.5, 0.5, 0, 0]]], np.float32), st,
                                    np.zeros((1, 1), np.int32), np.ones(1, np.int32), 2, 2)
    oracle.eagle_expand(np.array([[[0, 0, 1.0, 0], [0, 0, 0, 1.0]]], np.float32), st, f1, n1, 1, 2)
    t = oracle.eagle_rerank(st, 5)
    # scores .5, .5, .5, .5: depth 1 first (generated order), then depth 2
    assert list(t["token"][0]) == [-1, 0, 1, 2, 3]
    assert list(t["parent"][0]) == [-1, 0, 0, 1, 2]
    assert list(t["depth"][0]) == [0, 1, 1, 2, 2]


def test_invariants_restricted_expansion():
    rng = np.random.default_rng(9)
    B, V, L, K2, Fn, N = 6, 50, 6, 4, 5, 30
    cache = {}

    def cond(b, path):
        if (b, path) not in cache:
            cache[(b, path)] = (rng.random(V) ** 4 / 1.0).astype(np.float32)
            cache[(b, path)] /= cache[(b, path)].sum()
        return cache[(b, path)]

    # step 1: the root's K2 children; step 2: min(K2, Fn) of them expanded;
    # later steps: Fn nodes, K2 children each
    want = 1 + K2 + min(K2, Fn) * K2 + (L - 2) * Fn * K2
    st, statuses = _drive(cond, B, V, L, K2, Fn, G=want)
    assert all((s == 0).all() for s in statuses)
    assert (st["num_gen"] == want).all()
    for b in range(B):
        paths = _paths(st, b)
        for i in range(1, st["num_gen"][b]):
            p = st["parent"][b, i]
            assert st["depth"][b, i] == st["depth"][b, p] + 1
            row = cond(b, paths[p])
            # a child is one of its parent row's K2 most probable tokens
            order = sorted(range(V), key=lambda x: (-float(row[x]), x))[:K2]
            assert st["token"][b, i] in order
            assert st["score"][b, i] == st["score"][b, p] * float(row[st["token"][b, i]])
    t = oracle.eagle_rerank(st, N)
    W = (N + 63) // 64
    for b in range(B):
        nn = t["num_nodes"][b]
        assert nn == N
        for n in range(1, nn):
            par = t["parent"][b, n]
            assert 0 <= par < n                                   # parents first
            assert t["score"][b, n] <= t["score"][b, par]
            assert t["depth"][b, n] == t["depth"][b, par] + 1
            m = 0
            a = n
            while a >= 0:
                m |= 1 << a
                a = t["parent"][b, a]
            got = sum(int(t["anc_mask"][b, n, w]) << (64 * w) for w in range(W))
            assert got == m
            assert bin(got).count("1") - 1 == t["depth"][b, n]
        # no node left out scores above one kept (score, then depth)
        kept = set()
        for n in range(1, nn):
            kept.add((float(t["score"][b, n]), int(t["depth"][b, n])))
        worst = min(kept, key=lambda x: (x[0], -x[1]))
        for i in range(1, st["num_gen"][b]):
            key = (float(st["score"][b, i]), int(st["depth"][b, i]))
            if key not in kept:
                assert (key[0], -key[1]) <= (worst[0], -worst[1])


def test_capacity_and_bad_rows_are_flagged():
    st = oracle.eagle_init(2, 4)
    q = np.array([[[0.4, 0.3, 0.2, 0.1, 0.0]], [[np.nan, 0.5, 0.5, 0.0, 0.0]]], np.float32)
    f, n, s = oracle.eagle_expand(q, st, np.zeros((2, 1), np.int32), np.ones(2, np.int32), 4, 2)
    assert s[0] == oracle.ST_TREE_FULL and st["num_gen"][0] == 4    # three of four children fit
    assert list(st["token"][0, 1:4]) == [0, 1, 2]
    assert s[1] == oracle.ST_BAD_ROW and st["num_gen"][1] == 1 and n[1] == 0
    assert list(f[1]) == [-1, -1]
    # a frontier id outside the generated nodes
    st2 = oracle.eagle_init(1, 8)
    _, n2, s2 = oracle.eagle_expand(np.ones((1, 1, 3), np.float32) / 3, st2, np.full((1, 1), 5, np.int32),
                                    np.ones(1, np.int32), 2, 2)
    assert s2[0] == oracle.ST_BAD_NODE and n2[0] == 0
