"""Host-side checks of the seeded workload generator (tree shapes, layouts)."""
import torch

from gdn_speculative_tree_gb300 import workloads as wl


def test_width_tree_sizes_match_table2():
    # TreeWY paper Table 2: (1,1,1)->3, (2,1,1)->6, (2,2,1)->10, (2,2,2)->14,
    # (3,2,2)->21, (3,3,2)->30, (3,3,3)->39
    for widths, n in [((1, 1, 1), 3), ((2, 1, 1), 6), ((2, 2, 1), 10), ((2, 2, 2), 14),
                      ((3, 2, 2), 21), ((3, 3, 2), 30), ((3, 3, 3), 39)]:
        par = wl.width_tree_parents(widths)
        assert len(par) == n
        assert all(-1 <= p < i for i, p in enumerate(par))
        assert int((par == -1).sum()) == widths[0]
        assert wl.tree_depths(par).max() == len(widths)


def test_binary_tree_dfs_preorder():
    par = wl.complete_binary_parents(4)
    assert len(par) == 15
    assert list(par[:5]) == [-1, 0, 1, 2, 2]
    d = wl.tree_depths(par)
    assert d.max() == 4 and (d == 4).sum() == 8
    # DFS pre-order: each subtree occupies a contiguous index range
    for i in range(15):
        desc = [j for j in range(15) if i in _ancestors(par, j)]
        if desc:
            assert desc == list(range(i + 1, i + 1 + len(desc)))


def _ancestors(par, j):
    out = []
    p = par[j]
    while p >= 0:
        out.append(p)
        p = par[p]
    return out


def test_random_trees_respect_depth_and_size():
    trees, acc = wl.make_trees(wl.CONFIGS["wide"])
    assert len(trees) == 256
    for t, a in zip(trees, acc):
        assert 16 <= len(t) <= 64
        assert t[0] == -1 and all(0 <= p < i for i, p in enumerate(t) if i > 0)
        assert wl.tree_depths(t).max() <= 8
        assert 0 <= a < len(t)


def test_branches_and_chain_shapes():
    par = wl.branches_parents(8, 8)
    assert len(par) == 64 and (par == -1).sum() == 8 and wl.tree_depths(par).max() == 8
    trees, acc = wl.make_trees(wl.CONFIGS["chain"])
    assert all(list(t) == [-1, 0, 1, 2] for t in trees)
    assert acc.min() >= -1 and acc.max() <= 3 and (acc == -1).any()
    trees, acc = wl.make_trees(wl.CONFIGS["tiny"])
    assert list(trees[0]) == [-1, 0, 1, 2] and list(acc) == [1]


def test_generated_layout_and_seeding():
    cfg = wl.CONFIGS["binary"]
    a = wl.generate(cfg, R=5)
    b = wl.generate(cfg, R=5)
    assert a.T == 75 and a.node_offset.tolist() == [0, 15, 30, 45, 60, 75]
    assert a.q.dtype == torch.bfloat16 and a.q.shape == (75, 32, 128)
    assert a.state.shape == (5, 32, 128, 128) and a.state.dtype == torch.float32
    assert sorted(a.state_slot.tolist()) == list(range(5))
    assert torch.equal(a.q, b.q) and torch.equal(a.state, b.state)
    n = a.k.float().norm(dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-2)
    assert float(a.alpha.min()) >= 0.9 and float(a.alpha.max()) <= 0.999
    assert 0 < float(a.beta.min()) and float(a.beta.max()) < 1
    c = wl.generate(cfg, R=5, layer=1)
    assert not torch.equal(a.q, c.q)


def test_tiny_is_fp32():
    w = wl.generate(wl.CONFIGS["tiny"])
    assert w.q.dtype == torch.float32 and w.dk == 16 and w.T == 4
