"""Byte-budgeted per-expert format assignment (Strata 4090 post, section 5,
first paragraph): the oracle pinned against brute force on tiny instances,
then the library's host entry point against the oracle, bit for bit.  No GPU."""
import itertools

import numpy as np
import pytest

import synth
from oracle import assign as OA

TQ1, Q2_0, Q3_K = 1, 2, 3
# bytes of one DeepSeek-V4.1-Flash expert in each format (3 x 5120 x 2304 weights)
NB = [7741440, 9953280, 15206400]


def _cost(err, energy, weight):
    L, E, _ = err.shape
    return [[[float(weight[l]) * float(err[l, e, f]) / float(energy[l]) for f in range(3)] for e in range(E)]
            for l in range(L)]


def _feasible(L, E, locked, cap):
    """Every assignment (format indices 0..2) that keeps locked experts at Q2_0
    and at most cap[l] ternary experts per layer (brute force)."""
    choices = []
    for l in range(L):
        for e in range(E):
            choices.append((1,) if locked[l][e] else (0, 1, 2))
    for combo in itertools.product(*choices):
        rows = [list(combo[l * E:(l + 1) * E]) for l in range(L)]
        if all(sum(1 for f in rows[l] if f == 0) <= cap[l] for l in range(L)):
            yield rows


def _instance(seed, L, E, lock_some=True):
    rng = np.random.default_rng(seed)
    err, energy, tokens = synth.format_error_proxy(rng, L, E)
    if not lock_some:
        tokens = None
    else:
        tokens = tokens.copy()
        tokens[0, 0] = 3  # at least one locked expert
    return err, energy, tokens


def _to_lists(err, energy, tokens):
    return (err.tolist(), energy.tolist(), None if tokens is None else tokens.tolist())


# ---------------------------------------------------------------------------
# oracle pins
# ---------------------------------------------------------------------------
def test_layer_weights_double_the_outer_layers():
    w = OA.layer_weights(43)
    assert w[:2] == [2.0, 2.0] and w[-3:] == [2.0, 2.0, 2.0]
    assert all(v == 1.0 for v in w[2:-3]) and len(w) == 43


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_relaxed_problem_is_solved_exactly(seed):
    """At any multiplier, the relaxed assignment minimises cost + lam * bytes
    over every assignment the guard rails allow (brute force, 2 layers x 4)."""
    L, E = 2, 4
    err, energy, tokens = _instance(seed, L, E)
    weight = OA.layer_weights(L)
    cost = _cost(err, energy, weight)
    locked = [[tokens[l, e] < 8 for e in range(E)] for l in range(L)]
    cap = [E // 2] * L
    spread = max(max(c) - min(c) for row in cost for c in row)
    for lam in [0.0, spread / 1e7, spread / 3e6, spread / 1e6, spread / 1e5, 10 * spread]:
        pick = OA.relaxed(cost, locked, cap, lam, NB)
        val = sum(cost[l][e][pick[l][e]] + lam * NB[pick[l][e]] for l in range(L) for e in range(E))
        best = min(sum(cost[l][e][r[l][e]] + lam * NB[r[l][e]] for l in range(L) for e in range(E))
                   for r in _feasible(L, E, locked, cap))
        assert locked[0][0] and pick[0][0] == 1
        assert all(sum(1 for f in pick[l] if f == 0) <= cap[l] for l in range(L))
        assert val <= best * (1 + 1e-12) + 1e-300


@pytest.mark.parametrize("seed", [4, 5, 6, 7])
@pytest.mark.parametrize("frac", [1.0, 0.96, 1.1])
def test_assignment_against_brute_force(seed, frac):
    """The Lagrangian assignment (before the greedy pass) is the cheapest of
    all allowed assignments of no more bytes; the final one fits the budget,
    keeps the guard rails, costs no more, and leaves no single upgrade that
    would still fit."""
    L, E = 2, 4
    err, energy, tokens = _instance(seed, L, E)
    weight = OA.layer_weights(L)
    budget = int(frac * L * E * NB[1])
    res = OA.assign(*_to_lists(err, energy, tokens)[:2], weight, tokens.tolist(), 8, 0.5, NB, budget)
    assert res is not None
    fmts, lam, nbytes, total = res
    cost = _cost(err, energy, weight)
    locked = [[tokens[l, e] < 8 for e in range(E)] for l in range(L)]
    cap = [E // 2] * L
    relaxed = OA.relaxed(cost, locked, cap, lam, NB)
    rb = sum(NB[f] for row in relaxed for f in row)
    rc = sum(cost[l][e][relaxed[l][e]] for l in range(L) for e in range(E))
    assert rb <= budget
    for r in _feasible(L, E, locked, cap):
        if sum(NB[f] for row in r for f in row) <= rb:
            assert sum(cost[l][e][r[l][e]] for l in range(L) for e in range(E)) >= rc * (1 - 1e-12)
    pick = [[{TQ1: 0, Q2_0: 1, Q3_K: 2}[f] for f in row] for row in fmts]
    assert nbytes == sum(NB[f] for row in pick for f in row) <= budget
    assert all(pick[l][e] == 1 for l in range(L) for e in range(E) if locked[l][e])
    assert all(sum(1 for f in pick[l] if f == 0) <= cap[l] for l in range(L))
    assert total <= rc * (1 + 1e-12)
    left = budget - nbytes
    for l in range(L):
        for e in range(E):
            if locked[l][e]:
                continue
            for g in range(pick[l][e] + 1, 3):
                if NB[g] - NB[pick[l][e]] <= left:
                    assert cost[l][e][g] >= cost[l][e][pick[l][e]]


def test_special_cases():
    L, E = 3, 6
    err, energy, tokens = _instance(9, L, E)
    weight = OA.layer_weights(L)
    e_, en_, tok_ = _to_lists(err, energy, tokens)
    locked = tokens < 8
    # a budget that holds everything: every unlocked expert at its least error
    fmts, lam, nbytes, _ = OA.assign(e_, en_, weight, tok_, 8, 0.5, NB, 10 ** 12)
    assert lam == 0.0
    for l in range(L):
        for e in range(E):
            want = Q2_0 if locked[l, e] else (1 + int(np.argmin(err[l, e])))
            assert fmts[l][e] == want
    # the least the guard rails allow: half the layer ternary, the rest Q2_0
    n_lock = int(locked.sum())
    tq_each = [min(E // 2, E - int(locked[l].sum())) for l in range(L)]
    least = sum(tq_each) * NB[0] + (L * E - sum(tq_each)) * NB[1]
    fmts, lam, nbytes, _ = OA.assign(e_, en_, weight, tok_, 8, 0.5, NB, least)
    assert nbytes == least and lam > 0.0 and n_lock >= 1
    assert [sum(1 for f in row if f == TQ1) for row in fmts] == tq_each
    assert OA.assign(e_, en_, weight, tok_, 8, 0.5, NB, least - 1) is None
    # the same error in every format: nothing is worth a byte more
    flat = np.repeat(err[:, :, :1], 3, axis=2)
    fmts, lam, nbytes, _ = OA.assign(flat.tolist(), en_, weight, None, 8, 0.5, NB, L * E * NB[1])
    assert lam == 0.0 and all(sum(1 for f in row if f == TQ1) == E // 2 for row in fmts)
    assert all(f in (TQ1, Q2_0) for row in fmts for f in row)


def test_pages_mix_is_budget_neutral():
    """The post's mix (42.8 / 39.2 / 18.0 % of the weights ternary / Q2_0 /
    Q3_K) averages to the 2.25 bits of all-Q2_0 (within 0.01 %)."""
    bpw = 0.428 * 1.75 + 0.392 * 2.25 + 0.180 * 3.4375
    assert abs(bpw - 2.25) / 2.25 < 1e-3
    assert [b * 8 / (3 * 5120 * 2304) for b in NB] == [1.75, 2.25, 3.4375]


# ---------------------------------------------------------------------------
# the library's host entry point against the oracle (bit for bit)
# ---------------------------------------------------------------------------
def _both(err, energy, tokens, min_tokens, frac, budget, weight=None):
    from bit_quantised_expert_gb300 import _abi as A
    L = err.shape[0]
    weight = OA.layer_weights(L) if weight is None else weight
    ref = OA.assign(err.tolist(), energy.tolist(), list(weight), None if tokens is None else tokens.tolist(),
                    min_tokens, frac, NB, budget)
    try:
        got = A.bqe_assign_formats(err, energy, np.asarray(weight, np.float64), tokens, min_tokens, frac,
                                   np.asarray(NB, np.uint64), budget)
    except A.BqeError as ex:
        assert ref is None, ex
        assert ex.status == A.BQE_EINVAL
        return None
    assert ref is not None
    fmts, lam, nbytes, total = ref
    assert np.array_equal(got[0], np.asarray(fmts, np.int32))
    assert got[1] == lam and got[2] == nbytes and got[3] == total
    return got


@pytest.mark.parametrize("seed,L,E", [(11, 4, 16), (12, 6, 32), (13, 10, 64), (14, 1, 7)])
@pytest.mark.parametrize("frac", [1.0, 0.9, 1.2])
def test_library_matches_oracle(seed, L, E, frac):
    err, energy, tokens = _instance(seed, L, E)
    _both(err, energy, tokens, 8, 0.5, int(frac * L * E * NB[1]))


def test_library_matches_oracle_on_ties_and_edges():
    rng = np.random.default_rng(21)
    L, E = 5, 12
    err = np.ones((L, E, 3))  # every cost equal: ties everywhere
    energy = np.ones(L)
    _both(err, energy, None, 8, 0.5, L * E * NB[1])
    err2 = np.repeat(rng.lognormal(0, 1, size=(L, E, 1)), 3, axis=2) * np.array([4.0, 2.0, 1.0])
    _both(err2, energy, None, 8, 0.25, L * E * NB[1])
    _both(err2, energy, None, 8, 0.0, L * E * NB[0])           # below the least allowed: refused
    _both(err2, energy, None, 8, 0.0, L * E * NB[1])           # no ternary allowed: the budget is exact
    tok = np.zeros((L, E), np.int32)
    _both(err2, energy, tok, 8, 0.5, L * E * NB[1])            # everything locked at Q2_0
    _both(err2, energy, None, 8, 0.5, 10 ** 12)                # nothing binds


def test_library_matches_oracle_full_size():
    """40 layers x 384 experts at the all-Q2_0 budget (the post's setting)."""
    err, energy, tokens = _instance(31, 40, 384)
    got = _both(err, energy, tokens, 8, 0.5, 40 * 384 * NB[1])
    fm = got[0]
    share = [(fm == f).mean() for f in (TQ1, Q2_0, Q3_K)]
    assert max((fm == TQ1).mean(axis=1)) <= 0.5
    assert share[0] > 0.2 and share[2] > 0.05  # a real mix, not one format


def test_library_rejects_bad_arguments():
    from bit_quantised_expert_gb300 import _abi as A
    err, energy, tokens = _instance(41, 2, 4)
    w = np.ones(2)
    fb = np.asarray(NB, np.uint64)
    with pytest.raises(A.BqeError):
        A.bqe_assign_formats(err, -energy, w, tokens, 8, 0.5, fb, 10 ** 9)
    with pytest.raises(A.BqeError):
        A.bqe_assign_formats(err, energy, w, tokens, 8, 1.5, fb, 10 ** 9)
    with pytest.raises(A.BqeError):
        A.bqe_assign_formats(err, energy, w, tokens, 8, 0.5, fb[::-1].copy(), 10 ** 9)
    bad = err.copy()
    bad[0, 0, 0] = np.nan
    with pytest.raises(A.BqeError):
        A.bqe_assign_formats(bad, energy, w, tokens, 8, 0.5, fb, 10 ** 9)
