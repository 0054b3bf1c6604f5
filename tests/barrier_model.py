"""Play the roles of a warp-specialized kernel against their mbarriers on the host.

A role is a list of operations: ("a", bar) arrives once on barrier `bar`;
("w", bar, k) waits until the barrier has completed its phase number k (0, 1,
...).  A barrier completes a phase when it has collected `counts[bar]` arrivals.

The hardware waits on a phase's parity, not its number: a wait for phase k
passes once the barrier has completed k and the parity has flipped, and would
wrongly block if the barrier had already completed k + 1 as well (two phases
ahead).  So besides running every role to completion, `play` reports a wait
that finds its barrier two or more phases past the one it waits for.

One run follows one schedule: the roles in a given order, each run as far as it
can before the next.  `play` tries the given order, its reverse and every
rotation, so that each role in turn runs ahead of the others as far as the
protocol lets it.
"""


def _run(roles, counts, order):
    pos = [0] * len(roles)
    arrived = {k: 0 for k in counts}
    phases = {k: 0 for k in counts}
    progress = True
    while progress:
        progress = False
        for ri in order:
            role = roles[ri]
            while pos[ri] < len(role):
                op = role[pos[ri]]
                if op[0] == "w":
                    if phases[op[1]] >= op[2] + 2:
                        return "overrun", (ri, pos[ri], op)
                    if phases[op[1]] <= op[2]:
                        break
                else:
                    arrived[op[1]] += 1
                    if arrived[op[1]] == counts[op[1]]:
                        arrived[op[1]] = 0
                        phases[op[1]] += 1
                pos[ri] += 1
                progress = True
    if all(pos[ri] == len(role) for ri, role in enumerate(roles)):
        return "done", None
    return "stalled", [(ri, pos[ri], roles[ri][pos[ri]]) for ri in range(len(roles)) if pos[ri] < len(roles[ri])]


def play(roles, counts):
    """'done' if every schedule tried runs every role to the end, else the first
    failure: 'stalled' (a wait that never passes) or 'overrun'."""
    n = len(roles)
    base = list(range(n))
    orders = [base[i:] + base[:i] for i in range(n)]
    orders += [list(reversed(o)) for o in orders]
    for order in orders:
        res, _ = _run(roles, counts, order)
        if res != "done":
            return res
    return "done"
