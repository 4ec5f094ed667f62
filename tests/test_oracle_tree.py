"""Pins of the oracle's token-tree verification.

The tree walk applies the pages' accept rule at every node; these check its
outputs against what fixes them independently of its code: a tree of one
child per node is the chain the pages define (the chain oracle, itself pinned
in test_oracle_pins.py); the first token out of a tree of independent
proposals from q is distributed as p (the losslessness the pages state), and
the first proposal is kept at the pages' printed rate 0.78 on their V=5 pair;
at T = 0 the walk follows the target argmax; malformed trees give -1.
"""
import numpy as np
from scipy import stats

import oracle
import workloads as W


def _chain_as_tree(inp):
    """The chain workload in the tree layout: node n is chain position n
    (its children are tested against target / draft row n), node n + 1 holds
    the proposal x_n and its uniform; slot 0 is the final draw."""
    B, Kmax, V = inp["B"], inp["Kmax"], inp["V"]
    N = Kmax + 1
    dt = inp["target"].dtype
    tgt = inp["target"].copy()
    drf = np.zeros((B, N, V), dt)
    drf[:, :Kmax] = inp["draft"]
    tok = np.zeros((B, N), np.int32)
    tok[:, 1:] = inp["tokens"]
    uni = np.zeros((B, N), np.float32)
    K = inp["K"]
    for b in range(B):
        uni[b, 1:K[b] + 1] = inp["uniforms"][b, :K[b]]
        uni[b, 0] = inp["uniforms"][b, K[b]]
    parent = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    return dict(target=tgt, draft=drf, dtype=inp["dtype"], tokens=tok, parent=parent, uniforms=uni,
                temperature=inp["temperature"], n_nodes=(K + 1).astype(np.int32))


def _tree(d):
    return oracle.tree_verify(d["target"], d["draft"], d["dtype"], d["tokens"], d["parent"],
                              d["uniforms"], d["temperature"], d["n_nodes"])


def test_chain_trees_are_the_chain():
    for seed, (B, V, dtype) in enumerate([(40, 300, "f32"), (30, 1000, "bf16"), (20, 5, "f32")]):
        K = W.configs.ragged_k(6, B) if hasattr(W.configs, "ragged_k") else np.full(B, 4)
        temps = np.where(np.arange(B) % 3 == 0, 0.0, np.where(np.arange(B) % 3 == 1, 1.0, 0.7))
        inp = W.make_host(B, K, V, dtype, 2.0, 1.0, temps.astype(np.float32), seed=300 + seed)
        ref = oracle.verify_inputs(inp)
        got = _tree(_chain_as_tree(inp))
        assert np.array_equal(got["out_len"], ref["num_accepted"])
        assert np.array_equal(got["out_tokens"], ref["out_tokens"])
        assert np.array_equal(got["tie"], ref["tie"])
        for b in range(B):
            n = got["out_len"][b]
            assert np.array_equal(got["out_path"][b, :n], np.arange(1, n + 1))


def test_independent_proposals_keep_the_target_distribution():
    """Three proposals drawn independently from q at the root of the pages'
    V=5 pair: the first token out (the kept proposal, else the draw from the
    last residual) is distributed as p, and the first proposal is kept at
    sum_x min(p, q) = 0.78, the rate the pages print."""
    B = 200_000
    d = W.make_tree_pair(W.TOY_P, W.TOY_Q, B, 3, seed=2024)
    got = _tree(d)
    assert np.all(got["out_len"] >= 0)
    first = got["out_tokens"][:, 0]
    counts = np.bincount(first, minlength=5)
    assert stats.chisquare(counts, W.TOY_P * B).pvalue > 1e-3
    kept_first = np.mean(got["out_path"][:, 0] == 1)
    assert abs(kept_first - 0.78) < 4 * np.sqrt(0.78 * 0.22 / B)


def test_greedy_follows_the_target_argmax():
    """T = 0: the child equal to the target argmax is kept whatever its place
    among its siblings; with none equal, the token is the argmax."""
    V = 6
    parent = np.array([[-1, 0, 0, 0, 2, 2]], np.int32)
    tgt = np.zeros((1, 6, V), np.float32)
    tgt[0, 0, 4] = 3.0   # root argmax 4: the second child (node 2) holds it
    tgt[0, 2, 1] = 2.0   # node 2 argmax 1: neither child (5, 3) holds it
    tgt[0, 2, 3] = 1.0
    tok = np.array([[0, 5, 4, 4, 5, 3]], np.int32)
    d = dict(target=tgt, draft=np.zeros_like(tgt), dtype="f32", tokens=tok, parent=parent,
             uniforms=np.zeros((1, 6), np.float32), temperature=np.zeros(1, np.float32),
             n_nodes=np.array([6], np.int32))
    got = _tree(d)
    assert got["out_len"][0] == 1
    assert got["out_path"][0, 0] == 2
    assert got["out_tokens"][0, :3].tolist() == [4, 1, -1]


def test_malformed_trees_give_minus_one():
    d = W.make_tree_host(3, W.full_tree(2, 2), 40, "f32", 2.0, 1.0, 1.0, seed=9)
    d["parent"][0, 3] = 5          # a parent after its child
    d["tokens"][1, 1] = 40          # a token outside [0, V)
    d["n_nodes"][2] = 0             # no root
    got = _tree(d)
    assert got["out_len"].tolist() == [-1, -1, -1]
    assert np.all(got["out_tokens"] == -1)


def test_leaf_root_is_a_draw_from_p():
    """A tree of the root alone is the chain with K = 0: one draw from p."""
    B, V = 50_000, 5
    logits = np.log(W.TOY_P).astype(np.float32)
    d = dict(target=np.tile(logits, (B, 1, 1)), draft=np.zeros((B, 1, V), np.float32), dtype="f32",
             tokens=np.zeros((B, 1), np.int32), parent=np.full((B, 1), -1, np.int32),
             uniforms=W.uniform_grid(77, 1, B, 1), temperature=np.ones(B, np.float32),
             n_nodes=np.ones(B, np.int32))
    got = _tree(d)
    assert np.all(got["out_len"] == 0)
    counts = np.bincount(got["out_tokens"][:, 0], minlength=V)
    assert stats.chisquare(counts, W.TOY_P * B).pvalue > 1e-3


def _f32_softmax(logits32):
    from scipy import special
    return special.softmax(np.asarray(logits32, np.float64))


def _two_children(tl, dl, x1, x2, u1, u2, u0):
    """Root with children 1 and 2 (tokens x1, x2) tested in that order;
    uniforms u1, u2 test them, u0 is the final draw."""
    V = len(tl)
    tgt = np.zeros((1, 3, V), np.float32)
    drf = np.zeros((1, 3, V), np.float32)
    tgt[0, :] = tl
    drf[0, 0] = dl
    d = dict(target=tgt, draft=drf, dtype="f32", tokens=np.array([[0, x1, x2]], np.int32),
             parent=np.array([[-1, 0, 0]], np.int32),
             uniforms=np.array([[u0, u1, u2]], np.float32), temperature=np.ones(1, np.float32),
             n_nodes=np.array([3], np.int32))
    return _tree(d)


def test_tree_tie_flag_at_each_sibling_threshold():
    """The tie flag marks a child test whose uniform lies within 1e-6 of its
    threshold R(x)/q(x): R = p for the first child, and R =
    normalize(max(0, p - q)) (the distribution tech-tldr.com, section
    受理判定の数理, draws from after a rejection) for the second; inside the
    band (5e-7 away) the flag is set, outside it (2e-6 away) clear, and the
    decision follows the side of the threshold.  Thresholds come from scipy's
    softmax of the float32 logits."""
    tl = np.log(np.array([0.30, 0.25, 0.25, 0.20])).astype(np.float32)
    dl = np.log(np.array([0.50, 0.22, 0.18, 0.10])).astype(np.float32)
    p, q = _f32_softmax(tl), _f32_softmax(dl)
    R1 = np.maximum(p - q, 0.0)
    R1 /= R1.sum()
    th1, th2 = p[0] / q[0], R1[1] / q[1]
    assert 0.5 < th1 < 0.7 and 0.6 < th2 < 0.75
    u_final = 0.05    # far from the boundaries of every distribution drawn from here
    for delta in (-5e-7, 5e-7, -2e-6, 2e-6):
        inside = abs(delta) < 1e-6
        # first child at its threshold; the second (token 3, R(3)/q(3) = 2) is
        # then kept whatever happens, with u = 0.5 far from it
        g = _two_children(tl, dl, 0, 3, np.float32(th1 + delta), 0.5, u_final)
        assert g["out_path"][0, 0] == (1 if delta < 0 else 2)
        assert bool(g["tie"][0]) == inside, delta
        # first child rejected far from its threshold (u = 0.95), the second
        # at its threshold against R1
        g = _two_children(tl, dl, 0, 1, 0.95, np.float32(th2 + delta), u_final)
        assert g["out_len"][0] == (1 if delta < 0 else 0)
        assert bool(g["tie"][0]) == inside, delta
