"""Pins of the oracle's sparse-tree rounds ("RVQ Position Aware Speculative
Decoding for On Device TTS", section 2.2, tree attention and sparse tree
attention, Figure 2).

Reading: the drafts of depth t come from head_{s+t} on h_s, so a tree node
is (depth, rank of its token among that depth's draft logits); every node
is verified against the committed prefix and its ancestors; acceptance walks
down from the committed code, testing the children in rank order as
point-mass drafts with residual renormalisation, and draws one code from
what is left when no child is accepted (or at a leaf).

- Greedy tree decoding equals the greedy AR loop for several trees.
- A one-rank chain tree reproduces the greedy chain rounds exactly (codes,
  rounds, passes, acceptance by offset): the rank-0 candidate is the greedy
  draft.
- With a branching tree, each first round of a frame accepts at least as
  deep as the chain (greedy).
- The law of (c_1, c_2, c_3), enumerated exactly on a tiny model, matches
  the tree decoder's frequencies (chi-square).
- Malformed trees are rejected.
"""
import itertools
import math

import numpy as np
import pytest

from speculative_decoding_rvq_gb300 import synth as S

TREES = {
    "chain3": ([-1, 0, 1], [0, 0, 0]),
    "wide": ([-1, -1, -1, 0, 1], [0, 1, 2, 0, 0]),
    "sparse": ([-1, -1, 0, 0, 1, 2, 3], [0, 1, 0, 1, 0, 0, 0]),
}


def _small(G=8, V=8):
    return S.ModelSpec(hidden=32, n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=16, ffn=64, vocab=V,
                       num_code_groups=G, dtype=S.DTYPE_F32)


@pytest.mark.parametrize("name", sorted(TREES))
@pytest.mark.parametrize("G", [4, 8])
def test_greedy_tree_equals_greedy_ar(orc, name, G):
    spec = _small(G=G)
    m = orc.Model(spec, S.gen_weights(spec, seed=3, std=0.5))
    x, c0 = S.gen_frames(spec, 2, 4, seed=1)
    ar, _, _ = m.decode_frames(0, 50, 0.0, 1, x, c0)
    par, rk = TREES[name]
    tr, st, _ = m.decode_frames_tree(par, rk, 50, 0.0, 1, x, c0)
    assert np.array_equal(tr, ar)
    assert st["committed"] == 8 * (G - 1)


def test_chain_tree_is_the_greedy_chain(orc):
    spec = _small()
    m = orc.Model(spec, S.gen_weights(spec, seed=3, std=0.5))
    x, c0 = S.gen_frames(spec, 2, 6, seed=2)
    ch, sc, _ = m.decode_frames(4, 50, 0.0, 1, x, c0)
    tr, st, _ = m.decode_frames_tree([-1, 0, 1], [0, 0, 0], 50, 0.0, 1, x, c0)
    assert np.array_equal(tr, ch)
    assert (st["rounds"], st["passes"]) == (sc["rounds"], sc["passes"])
    assert st["accepted_by_offset"] == sc["accepted_by_offset"]
    assert sum(sc["accepted_by_offset"]) > 0  # the comparison is not vacuous


def test_branching_tree_accepts_at_least_the_chain(orc):
    spec = _small()
    m = orc.Model(spec, S.gen_weights(spec, seed=3, std=0.5))
    x, c0 = S.gen_frames(spec, 1, 8, seed=4)
    _, _, lc = m.decode_frames_tree([-1, 0, 1], [0, 0, 0], 50, 0.0, 1, x, c0, log_cap=500)
    _, _, lt = m.decode_frames_tree(*TREES["sparse"], 50, 0.0, 1, x, c0, log_cap=500)
    fc, ft = lc[lc["s"] == 1], lt[lt["s"] == 1]  # the first round of each frame starts from the same state
    assert len(fc) == len(ft) == 8
    assert np.all(ft["n_acc"] >= fc["n_acc"])
    assert np.sum(ft["n_acc"]) > np.sum(fc["n_acc"])


def test_tree_law_equals_autoregressive_law(orc):
    spec = S.ModelSpec(hidden=16, n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=8, ffn=32, vocab=4,
                       num_code_groups=4, dtype=S.DTYPE_F32)
    m = orc.Model(spec, S.gen_weights(spec, seed=21, std=0.5))
    x, c0 = S.gen_frames(spec, 1, 1, seed=22)
    k, T = 3, 0.9
    law = {}
    for tup in itertools.product(range(4), repeat=3):
        lg, _ = m.teacher_logits(x[0, 0], [int(c0[0, 0]), *tup[:2]], 4)
        pr = 1.0
        for j in range(3):
            pj, _ = orc.process(lg[j], k, T)
            pr *= float(pj[tup[j]])
        law[tup] = pr
    F = 30000
    xs = np.broadcast_to(x, (F, 1, spec.hidden)).copy()
    cs = np.broadcast_to(c0, (F, 1)).copy()
    codes, st, _ = m.decode_frames_tree([-1, -1, 0, 0, 1], [0, 1, 0, 1, 0], k, T, 77, xs, cs)
    assert st["rounds"] > 0 and sum(st["accepted_by_offset"]) > 0
    cnt = {}
    for row in codes[:, 0, 1:]:
        key = tuple(int(v) for v in row)
        cnt[key] = cnt.get(key, 0) + 1
    chi2, df = 0.0, -1
    for tup, pr in law.items():
        o = cnt.get(tup, 0)
        if pr == 0.0:
            assert o == 0, tup
            continue
        e = pr * F
        chi2 += (o - e) ** 2 / e
        df += 1
    z = ((chi2 / df) ** (1 / 3) - (1 - 2 / (9 * df))) / math.sqrt(2 / (9 * df))
    assert z < 3.7, (chi2, df)


def _max_tree():
    """A tree at both limits: 62 nodes, depth 7, parents first, siblings in
    ascending rank.  Depth 1 holds ranks 0..7; below it the rank-0 path
    keeps branching (8, 6, 4, 3, 3, 2 children), with smaller side branches."""
    par, rk = [], []

    def add(p, ranks):
        first = len(par)
        for r in ranks:
            par.append(p)
            rk.append(r)
        return list(range(first, len(par)))

    l1 = add(-1, range(8))
    l2 = add(l1[0], range(8)) + add(l1[1], range(4))
    for p in l1[2:]:
        l2 += add(p, range(2))
    l3 = add(l2[0], range(6))
    for p in l2[1:8]:
        l3 += add(p, [0])
    l4 = add(l3[0], range(4))
    for p in l3[1:6]:
        l4 += add(p, [0])
    l5 = add(l4[0], range(3))
    l6 = add(l5[0], range(3))
    add(l6[0], range(2))
    return par, rk


def test_max_tree_shape():
    par, rk = _max_tree()
    dep = []
    for p in par:
        dep.append(1 if p < 0 else dep[p] + 1)
    assert len(par) == 62 and max(dep) == 7


@pytest.mark.parametrize("G", [9, 16])
def test_max_tree_greedy_equals_greedy_ar(orc, G):
    spec = _small(G=G)
    m = orc.Model(spec, S.gen_weights(spec, seed=3, std=0.5))
    x, c0 = S.gen_frames(spec, 2, 4, seed=1)
    ar, _, _ = m.decode_frames(0, 50, 0.0, 1, x, c0)
    tr, st, _ = m.decode_frames_tree(*_max_tree(), 50, 0.0, 1, x, c0)
    assert np.array_equal(tr, ar)
    # the 8 depth-1 candidates are the whole vocabulary: every round accepts depth 1
    assert st["accepted_by_offset"][1] == st["rounds"]


@pytest.mark.parametrize("G", [9, 16])
def test_max_tree_zero_heads_walks_to_full_depth(orc, G):
    """Zero lm_heads: every logit is 0, so the greedy target is code 0 and the
    rank-r candidate of every depth is code r.  The rank-0 path (depth 7) is
    then accepted node by node as deep as the frame allows, the bonus follows
    when the path stops short of c_{G-1}, and each round verifies the root
    plus every node short of the frame end."""
    spec = _small(G=G)
    w = S.gen_weights(spec, seed=3, std=0.5)
    w = {**w, "lm_head": np.zeros_like(w["lm_head"])}
    m = orc.Model(spec, w)
    F, B = 4, 2
    x, c0 = S.gen_frames(spec, B, F, seed=1)
    par, rk = _max_tree()
    dep = []
    for p in par:
        dep.append(1 if p < 0 else dep[p] + 1)
    codes, st, log = m.decode_frames_tree(par, rk, 50, 0.0, 1, x, c0, log_cap=500)
    assert np.all(codes[:, :, 1:] == 0)
    # expected rounds of one frame: from s = 1, accept min(7, G-1-s) codes, plus a bonus below G-1
    acc = [0] * 9
    rounds = bonus = 0
    rows, s = [], 1
    while s < G - 1:
        n = min(7, G - 1 - s)
        rows.append(1 + sum(1 for t in dep if s + t <= G - 1))
        for t in range(1, n + 1):
            acc[t] += 1
        rounds += 1
        s += n
        if s < G - 1:
            s += 1
            bonus += 1
    FB = F * B
    assert st["rounds"] == FB * rounds and st["passes"] == FB * (rounds + 1)
    assert st["committed"] == FB * (G - 1) and st["bonus"] == FB * bonus and st["rejections"] == 0
    assert st["accepted_by_offset"] == [FB * a for a in acc]
    first = log[log["s"] == 1]
    assert np.all(first["n_acc"] == min(7, G - 2)) and np.all(first["m"] == rows[0])
    assert sorted(set(log["m"][log["s"] > 0].tolist())) == sorted(set(rows))


@pytest.mark.parametrize("par,rk", [([0], [0]), ([-1, -1], [1, 0]), ([-1, -1], [0, 0]), ([-1, 2, 0], [0, 0, 0]),
                                    ([-1], [-1])])
def test_malformed_trees_are_rejected(orc, par, rk):
    spec = _small()
    m = orc.Model(spec, S.gen_weights(spec, seed=3, std=0.5))
    x, c0 = S.gen_frames(spec, 1, 1, seed=4)
    with pytest.raises(ValueError):
        m.decode_frames_tree(par, rk, 50, 0.0, 1, x, c0)
