"""Pins for the CPU oracle: checks against things other than the oracle itself.

* hand-derived values of a 3-node tree (tests/golden/hand_tree3_dk2.txt);
* the pages' closed form (dense system of the TreeWY paper §3 Eq. (2) solved
  by LU, read out with the review's Eq. (5)/(6)) on every tree topology with
  N <= 5 and on random larger trees, with dk != dv so a transposed operand
  cannot hide;
* a chain equals the sequential token loop (review §3.2: the chain is
  DeltaNet's WY case);
* every node's result equals the chain loop over its own root-to-node path,
  and is bit-identical when any non-ancestor's inputs change (review §3.2,
  "not siblings, not descendants");
* beta = 0 reduces to pure decay; beta = alpha = 1 with unit keys writes
  exactly (S_n k_n = v_n, the delta rule of review §2.4);
* planted mistakes in a copy of the oracle are caught by these pins.
"""
import inspect
import itertools
import os
import textwrap

import numpy as np
import pytest

from oracle import gdn_tree_oracle as orc
from tests.closed_form import ancestor_sets, closed_form_head, sequential_gdn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_tree3_dk2.txt")


def load_golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *nums = line.split()
            vals[key] = np.array([float(x) for x in nums])
    return vals


def one_head(parent, q, k, v, alpha, beta, S0, fn=None):
    fn = fn or orc.verify_request
    res = fn(S0[None], parent, q[:, None], k[:, None], v[:, None], alpha[:, None], beta[:, None])
    return (res.o[:, 0], res.U[:, 0], res.gamma[:, 0], res.states[:, 0])


def random_head(rng, N, dk, dv, unit_keys=True):
    k = rng.standard_normal((N, dk))
    q = rng.standard_normal((N, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=1, keepdims=True)
        q /= np.linalg.norm(q, axis=1, keepdims=True)
    v = rng.standard_normal((N, dv))
    alpha = rng.uniform(0.8, 0.999, N)
    beta = rng.uniform(0.05, 0.95, N)
    S0 = rng.standard_normal((dv, dk)) * 0.3
    return q, k, v, alpha, beta, S0


def rel_err(a, b):
    scale = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / scale) if a.size else 0.0


def all_topologies(N):
    """Every parent array with parent[n] in [-1, n) (N! trees)."""
    return itertools.product(*[range(-1, n) for n in range(N)])


# ---------------------------------------------------------------- golden

def test_golden_hand_tree():
    g = load_golden()
    parent = g["parent"].astype(int)
    S0 = g["S0"].reshape(2, 2)
    k = g["k"].reshape(3, 2)
    v = g["v"].reshape(3, 2)
    q = g["q"].reshape(3, 2)
    o, U, gamma, states = one_head(parent, q, k, v, g["alpha"], g["beta"], S0)
    np.testing.assert_allclose(o, g["o"].reshape(3, 2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(U, g["U"].reshape(3, 2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(gamma, g["gamma"], rtol=0, atol=1e-15)
    for n in range(3):
        np.testing.assert_allclose(states[n], g[f"state{n}"].reshape(2, 2), rtol=0, atol=1e-12)
    res = orc.verify_request(S0[None], parent, q[:, None], k[:, None], v[:, None],
                             g["alpha"][:, None], g["beta"][:, None])
    np.testing.assert_allclose(orc.commit_request(S0[None], res, 2)[0],
                               g["state2"].reshape(2, 2), rtol=0, atol=1e-12)
    assert np.array_equal(orc.commit_request(S0[None], res, -1)[0], S0)


# ---------------------------------------------------------------- closed form

@pytest.mark.parametrize("N", [1, 2, 3, 4, 5])
def test_closed_form_every_topology(N):
    rng = np.random.default_rng(100 + N)
    dk, dv = 3, 4
    worst = 0.0
    for parent in all_topologies(N):
        parent = np.array(parent)
        q, k, v, alpha, beta, S0 = random_head(rng, N, dk, dv)
        o, U, gamma, states = one_head(parent, q, k, v, alpha, beta, S0)
        o2, Vt, g, S2 = closed_form_head(S0, parent, q, k, v, alpha, beta)
        worst = max(worst, rel_err(o, o2), rel_err(U, Vt), rel_err(gamma, g), rel_err(states, S2))
    # the pages report ~1e-15 agreement in fp64
    assert worst < 1e-12, worst


def test_closed_form_random_trees():
    rng = np.random.default_rng(7)
    for trial in range(40):
        N = int(rng.integers(6, 20))
        parent = np.array([-1] + [int(rng.integers(-1, n)) for n in range(1, N)])
        q, k, v, alpha, beta, S0 = random_head(rng, N, 5, 7)
        o, U, gamma, states = one_head(parent, q, k, v, alpha, beta, S0)
        o2, Vt, g, S2 = closed_form_head(S0, parent, q, k, v, alpha, beta)
        assert rel_err(o, o2) < 1e-12
        assert rel_err(U, Vt) < 1e-12
        assert rel_err(states, S2) < 1e-12


def test_closed_form_fp32_agreement_matches_pages():
    """The pages report ~1e-7 agreement in fp32; the oracle route run in fp32
    against the fp64 closed form lands in that range."""
    rng = np.random.default_rng(11)
    N, dk, dv = 12, 16, 16
    parent = np.array([-1] + [int(rng.integers(-1, n)) for n in range(1, N)])
    q, k, v, alpha, beta, S0 = random_head(rng, N, dk, dv)
    o2, _, _, _ = closed_form_head(S0, parent, q, k, v, alpha, beta)
    S = {}
    o32 = np.empty((N, dv), np.float32)
    for n in range(N):
        Sp = S0.astype(np.float32) if parent[n] < 0 else S[parent[n]]
        kn = k[n].astype(np.float32)
        a, b = np.float32(alpha[n]), np.float32(beta[n])
        Sn = a * (Sp - b * np.outer(Sp @ kn, kn)) + b * np.outer(v[n].astype(np.float32), kn)
        S[n] = Sn.astype(np.float32)
        o32[n] = S[n] @ q[n].astype(np.float32)
    err = rel_err(o32.astype(np.float64), o2)
    assert 1e-9 < err < 1e-5, err


# ---------------------------------------------------------------- chain / paths

def test_chain_equals_sequential_loop():
    rng = np.random.default_rng(3)
    N, dk, dv = 9, 6, 5
    parent = np.arange(-1, N - 1)
    q, k, v, alpha, beta, S0 = random_head(rng, N, dk, dv)
    o, U, gamma, states = one_head(parent, q, k, v, alpha, beta, S0)
    o2, S2 = sequential_gdn(S0, q, k, v, alpha, beta)
    assert rel_err(o, o2) < 1e-13
    assert rel_err(states, S2) < 1e-13
    np.testing.assert_allclose(gamma, np.cumprod(alpha), rtol=1e-15)


def test_every_path_equals_its_chain():
    rng = np.random.default_rng(5)
    for trial in range(10):
        N = int(rng.integers(5, 30))
        parent = np.array([-1] + [int(rng.integers(-1, n)) for n in range(1, N)])
        q, k, v, alpha, beta, S0 = random_head(rng, N, 4, 6)
        o, U, gamma, states = one_head(parent, q, k, v, alpha, beta, S0)
        anc = ancestor_sets(parent)
        for n in range(N):
            path = list(reversed(anc[n])) + [n]
            o2, S2 = sequential_gdn(S0, q[path], k[path], v[path], alpha[path], beta[path])
            assert rel_err(o[n], o2[-1]) < 1e-13
            assert rel_err(states[n], S2[-1]) < 1e-13
            np.testing.assert_allclose(gamma[n], np.prod(alpha[path]), rtol=1e-14)


def test_non_ancestors_do_not_matter():
    rng = np.random.default_rng(9)
    N = 24
    parent = np.array([-1] + [int(rng.integers(-1, n)) for n in range(1, N)])
    q, k, v, alpha, beta, S0 = random_head(rng, N, 5, 5)
    base = one_head(parent, q, k, v, alpha, beta, S0)
    anc = ancestor_sets(parent)
    for n in range(N):
        keep = set(anc[n]) | {n}
        other = [i for i in range(N) if i not in keep]
        if not other:
            continue
        q2, k2, v2, a2, b2 = q.copy(), k.copy(), v.copy(), alpha.copy(), beta.copy()
        q2[other] = rng.standard_normal((len(other), 5))
        k2[other] = rng.standard_normal((len(other), 5))
        v2[other] = rng.standard_normal((len(other), 5))
        a2[other] = rng.uniform(0.1, 0.9, len(other))
        b2[other] = rng.uniform(0.1, 0.9, len(other))
        pert = one_head(parent, q2, k2, v2, a2, b2, S0)
        for x, y in zip(base, pert):
            assert np.array_equal(x[n], y[n])


# ---------------------------------------------------------------- special cases

def test_beta_zero_is_pure_decay():
    rng = np.random.default_rng(13)
    N = 16
    parent = np.array([-1] + [int(rng.integers(-1, n)) for n in range(1, N)])
    q, k, v, alpha, beta, S0 = random_head(rng, N, 6, 4)
    beta[:] = 0.0
    o, U, gamma, states = one_head(parent, q, k, v, alpha, beta, S0)
    assert np.all(U == 0.0)
    for n in range(N):
        np.testing.assert_allclose(states[n], gamma[n] * S0, rtol=1e-14, atol=0)
        np.testing.assert_allclose(o[n], gamma[n] * (S0 @ q[n]), rtol=1e-13, atol=1e-15)


def test_full_write_stores_value_exactly():
    """alpha = beta = 1 and unit k: the delta rule stores v under k, S_n k_n = v_n."""
    rng = np.random.default_rng(17)
    N = 20
    parent = np.array([-1] + [int(rng.integers(-1, n)) for n in range(1, N)])
    q, k, v, alpha, beta, S0 = random_head(rng, N, 7, 5)
    alpha[:] = 1.0
    beta[:] = 1.0
    o, U, gamma, states = one_head(parent, q, k, v, alpha, beta, S0)
    for n in range(N):
        np.testing.assert_allclose(states[n] @ k[n], v[n], rtol=0, atol=1e-12)
    # reading with q = k returns the stored value
    o2, _, _, _ = one_head(parent, k, k, v, alpha, beta, S0)
    np.testing.assert_allclose(o2, v, rtol=0, atol=1e-12)


def test_commit_semantics():
    rng = np.random.default_rng(19)
    N = 10
    parent = np.array([-1, 0, 1, 0, 3, -1, 5, 6, 6, 2])
    q, k, v, alpha, beta, S0 = random_head(rng, N, 4, 4)
    res = orc.verify_request(S0[None], parent, q[:, None], k[:, None], v[:, None],
                             alpha[:, None], beta[:, None])
    assert np.array_equal(orc.commit_request(S0[None], res, -1)[0], S0)
    anc = ancestor_sets(parent)
    for a in range(N):
        path = list(reversed(anc[a])) + [a]
        _, S2 = sequential_gdn(S0, q[path], k[path], v[path], alpha[path], beta[path])
        assert rel_err(orc.commit_request(S0[None], res, a)[0], S2[-1]) < 1e-13
    with pytest.raises(ValueError):
        orc.commit_request(S0[None], res, N)


def test_bad_trees_are_rejected():
    for parent in ([0], [-1, 1], [-1, 0, 5], [-2]):
        with pytest.raises(ValueError):
            orc.check_tree(parent)


def test_batch_layout_matches_per_request():
    rng = np.random.default_rng(23)
    H, dk, dv = 3, 4, 5
    trees = [np.array([-1, 0, 0]), np.array([], dtype=int), np.array([-1, -1, 1, 2])]
    sizes = [len(t) for t in trees]
    off = np.concatenate([[0], np.cumsum(sizes)])
    T = off[-1]
    parent = np.concatenate(trees)
    q, k = rng.standard_normal((T, H, dk)), rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    alpha, beta = rng.uniform(0.5, 1, (T, H)), rng.uniform(0, 1, (T, H))
    state = rng.standard_normal((5, H, dv, dk))
    slot = np.array([4, 0, 2])
    out = orc.verify_batch(off, parent, q, k, v, alpha, beta, state, slot)
    for r in range(3):
        lo, hi = off[r], off[r + 1]
        for h in range(H):
            ref = one_head(trees[r], q[lo:hi, h], k[lo:hi, h], v[lo:hi, h], alpha[lo:hi, h],
                           beta[lo:hi, h], state[slot[r], h])
            assert np.array_equal(out[r].o[:, h], ref[0])
            assert np.array_equal(out[r].states[:, h], ref[3])


# ---------------------------------------------------------------- planted mistakes

MUTATIONS = {
    "wrong erase sign": ("S_par - b * pred", "S_par + b * pred"),
    "transposed state in prediction": ('pred = np.einsum("hij,hj->hi", S_par, kn)',
                                       'pred = np.einsum("hji,hj->hi", S_par, kn)'),
    "write term without beta": ("+ b * v[n][:, :, None]", "+ v[n][:, :, None]"),
    "read-out before update": ('o[n] = np.einsum("hij,hj->hi", S_n, q[n])',
                               'o[n] = np.einsum("hij,hj->hi", S_par, q[n])'),
    "gamma excludes own alpha": ("gamma[n] = alpha[n] * (1.0 if p < 0 else gamma[p])",
                                 "gamma[n] = (1.0 if p < 0 else alpha[p] * gamma[p])"),
    "previous node as parent": ("S_par = S0 if p < 0 else states[p]",
                                "S_par = S0 if n == 0 else states[n - 1]"),
    "pseudo-value without decay": ("(v[n] - alpha[n][:, None] * pred)", "(v[n] - pred)"),
}


def mutant(name):
    src = textwrap.dedent(inspect.getsource(orc.verify_request))
    old, new = MUTATIONS[name]
    assert old in src, name
    ns = dict(orc.__dict__)
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    return ns["verify_request"]


def pins_pass(fn):
    """Run the golden and closed-form pins against a candidate oracle function."""
    g = load_golden()
    parent = g["parent"].astype(int)
    o, U, gamma, states = one_head(parent, g["q"].reshape(3, 2), g["k"].reshape(3, 2),
                                   g["v"].reshape(3, 2), g["alpha"], g["beta"],
                                   g["S0"].reshape(2, 2), fn=fn)
    if not (np.allclose(o, g["o"].reshape(3, 2), atol=1e-12, rtol=0)
            and np.allclose(U, g["U"].reshape(3, 2), atol=1e-12, rtol=0)
            and np.allclose(gamma, g["gamma"], atol=1e-15, rtol=0)):
        return False
    rng = np.random.default_rng(29)
    for parent in all_topologies(4):
        parent = np.array(parent)
        q, k, v, alpha, beta, S0 = random_head(rng, 4, 3, 4)
        o, U, gamma, states = one_head(parent, q, k, v, alpha, beta, S0, fn=fn)
        o2, Vt, gg, S2 = closed_form_head(S0, parent, q, k, v, alpha, beta)
        if max(rel_err(o, o2), rel_err(U, Vt), rel_err(gamma, gg), rel_err(states, S2)) > 1e-12:
            return False
    return True


def test_pins_accept_the_oracle():
    assert pins_pass(orc.verify_request)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name):
    assert not pins_pass(mutant(name))


# ------------------------------------------------------------ bf16 state rounding

def test_round_to_bf16_hand_cases():
    """Nearest bfloat16 (8 significant bits), ties to even, from fp64 in one step."""
    cases = [
        (1.0 + 2.0 ** -8, 1.0),                    # tie: stays on the even neighbour 1
        (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),    # tie: goes up to the even neighbour
        (-(1.0 + 2.0 ** -8), -1.0),                # sign symmetric
        (1.0 + 2.0 ** -8 + 2.0 ** -30, 1.0 + 2.0 ** -7),  # just above a tie: up (no fp32 step)
        (255.5, 256.0),                            # tie at the top of a binade carries
        (1.0 - 2.0 ** -9, 1.0),                    # tie below 1 (spacing 2^-8 there)
        (0.0, 0.0),
        (3.0, 3.0),
        (0.1, 0.10009765625),                      # 0x3DCD
    ]
    x = np.array([c[0] for c in cases])
    want = np.array([c[1] for c in cases])
    assert np.array_equal(orc.round_to_bf16(x), want)


def test_round_to_bf16_matches_torch_on_fp32_inputs():
    """On fp32 inputs the one-step rounding equals torch's float32 -> bfloat16
    conversion (round to nearest even), a library routine."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(17)
    x = np.concatenate([rng.standard_normal(200000) * 0.05, rng.standard_normal(2000) * 1e3,
                        rng.uniform(-1, 1, 2000) * 1e-20]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(orc.round_to_bf16(x.astype(np.float64)), ref)


def test_commit_bf16_state_rounds_the_accepted_state():
    rng = np.random.default_rng(23)
    parent = np.array([-1, 0, 1, 0])
    q, k, v, alpha, beta, S0 = random_head(rng, 4, 3, 5)
    S0 = orc.round_to_bf16(S0)
    res = orc.verify_request(S0[None], parent, q[:, None], k[:, None], v[:, None], alpha[:, None],
                             beta[:, None])
    S_f = orc.commit_request(S0[None], res, 2)
    S_b = orc.commit_request(S0[None], res, 2, state_dtype="bf16")
    assert np.array_equal(S_b, orc.round_to_bf16(S_f))
    assert np.all(np.abs(S_b - S_f) <= 2.0 ** -8 * np.abs(S_f))
    assert np.array_equal(orc.commit_request(S0[None], res, -1, state_dtype="bf16"), S0[None])
