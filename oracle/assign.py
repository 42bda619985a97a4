"""Oracle for the byte-budgeted per-expert format assignment.  TEST
INFRASTRUCTURE ONLY.

What it computes follows the Strata 4090 post, section 5, first paragraph
(quantisation):

  * every routed expert gets one of three formats, ternary PTQ1_0 (1.75 bpw),
    Q2_0 (2.25) or Q3_K (3.44);
  * the byte budget is exactly what the same experts take as all-Q2_0 (the
    mix is budget-neutral);
  * the assignment comes from a Lagrangian relaxation with a bisection on the
    multiplier, then a greedy pass that spends the bytes left over;
  * the cost of a format for an expert is its held-out error divided by the
    routed output energy of its layer (every layer weighs the same), with the
    first two and the last three layers counted twice;
  * guard rails: at most half of a layer's experts ternary, and an expert
    seen by fewer than 8 held-out tokens stays Q2_0.

Readings where the post is silent (each one also in the design notes):
  * the half is floor(0.5 * experts of the layer), counted over all of them;
  * for a multiplier lam every unlocked expert takes the format of least
    cost + lam * bytes (ties: fewer bytes); if more than the cap take
    ternary, those with the largest loss from giving it up keep it (ties:
    lower expert index) and the rest take their best other format, which is
    the exact minimum of that layer's relaxed problem under the cap;
  * the bisection runs 100 halvings of [0, lam_max] and keeps the upper end
    (the least multiplier found whose assignment fits the budget); if lam = 0
    already fits, that one is taken;
  * the greedy pass repeatedly takes the single upgrade (an expert moved to
    a format of more bytes and strictly lower cost) of the largest cost
    decrease per byte that still fits the bytes left (ties: lower layer,
    then expert, then format), until none fits;
  * a budget below the least the guard rails allow is refused.

Formats are numbered as the library numbers them: 1 ternary, 2 Q2_0, 3 Q3_K.
"""
from __future__ import annotations

TQ1, Q2_0, Q3_K = 1, 2, 3
FORMATS = (TQ1, Q2_0, Q3_K)


def layer_weights(n_layers: int) -> list[float]:
    """2 for the first two and the last three layers, 1 for the others."""
    return [2.0 if (l < 2 or l >= n_layers - 3) else 1.0 for l in range(n_layers)]


def costs(err, energy, weight):
    """cost[l][e][f] = weight[l] * err[l][e][f] / energy[l]."""
    return [[[weight[l] * err[l][e][f] / energy[l] for f in range(3)] for e in range(len(err[l]))]
            for l in range(len(err))]


def relaxed_layer(cost_l, locked_l, cap: int, lam: float, nbytes):
    """The relaxed problem of one layer at multiplier lam (see the module
    docstring); returns format indices 0..2 (ternary, Q2_0, Q3_K)."""
    n = len(cost_l)
    pick = [1] * n
    alt = [1] * n
    keen = []  # (loss from giving ternary up, expert) of the experts whose best is ternary
    for e in range(n):
        if locked_l[e]:
            continue
        score = [cost_l[e][f] + lam * nbytes[f] for f in range(3)]
        best = 0
        for f in (1, 2):
            if score[f] < score[best]:
                best = f
        other = 1 if score[1] <= score[2] else 2
        pick[e] = best
        alt[e] = other
        if best == 0:
            keen.append((score[other] - score[0], e))
    if len(keen) > cap:
        keen.sort(key=lambda t: (-t[0], t[1]))
        for _, e in keen[cap:]:
            pick[e] = alt[e]
    return pick


def relaxed(cost, locked, caps, lam, nbytes):
    return [relaxed_layer(cost[l], locked[l], caps[l], lam, nbytes) for l in range(len(cost))]


def total_bytes(pick, nbytes) -> int:
    return sum(nbytes[f] for row in pick for f in row)


def total_cost(pick, cost) -> float:
    t = 0.0
    for l, row in enumerate(pick):
        for e, f in enumerate(row):
            t += cost[l][e][f]
    return t


def assign(err, energy, weight, tokens, min_tokens: int, cap_frac: float, nbytes, budget: int):
    """Returns (formats [l][e] as 1..3, lam, bytes, cost), or None when the
    budget is below the least the guard rails allow."""
    L = len(err)
    cost = costs(err, energy, weight)
    locked = [[tokens is not None and tokens[l][e] < min_tokens for e in range(len(err[l]))] for l in range(L)]
    caps = [int(cap_frac * len(err[l])) for l in range(L)]
    # the upper end of the bisection: large enough that every expert takes
    # its format of fewest bytes the cap allows
    spread = 0.0
    for l in range(L):
        for e in range(len(err[l])):
            c = cost[l][e]
            spread = max(spread, max(c) - min(c))
    gap = min(nbytes[1] - nbytes[0], nbytes[2] - nbytes[1])
    lam_max = 2.0 * spread / gap + 1.0
    if total_bytes(relaxed(cost, locked, caps, lam_max, nbytes), nbytes) > budget:
        return None
    pick0 = relaxed(cost, locked, caps, 0.0, nbytes)
    if total_bytes(pick0, nbytes) <= budget:
        lam, pick = 0.0, pick0
    else:
        lo, hi = 0.0, lam_max
        for _ in range(100):
            mid = 0.5 * (lo + hi)
            if total_bytes(relaxed(cost, locked, caps, mid, nbytes), nbytes) <= budget:
                hi = mid
            else:
                lo = mid
        lam = hi
        pick = relaxed(cost, locked, caps, hi, nbytes)
    # greedy: spend the bytes left on the best upgrades per byte
    left = budget - total_bytes(pick, nbytes)
    while True:
        best = None
        for l in range(L):
            for e in range(len(err[l])):
                if locked[l][e]:
                    continue
                f = pick[l][e]
                for g in range(f + 1, 3):
                    db = nbytes[g] - nbytes[f]
                    dc = cost[l][e][g] - cost[l][e][f]
                    if dc < 0.0 and db <= left:
                        r = dc / db
                        if best is None or r < best[0]:
                            best = (r, l, e, g)
        if best is None:
            break
        _, l, e, g = best
        left -= nbytes[g] - nbytes[pick[l][e]]
        pick[l][e] = g
    fmts = [[FORMATS[f] for f in row] for row in pick]
    return fmts, lam, total_bytes(pick, nbytes), total_cost(pick, cost)
