"""Tuning-plan oracle (test infrastructure only).

Restates the burn "autotune" page, section "one op, thirty-odd candidates":
every candidate belongs to a group; a group's priority and a candidate's
priority inside its group are functions of the key, and a negative value
skips it for that key.  Groups are tried from the highest priority down, and
once any candidate of a group gives a valid result no later group is tried.
Inside a group only the highest priority tier forms the round; lower tiers
are backups used only if the whole round fails.  Candidates the device (here:
the problem's alignment) cannot run are demoted to the minimum priority (0)
instead of being dropped, so the plan is never empty.

Ties between groups of equal priority keep registration order (the order in
which the first candidate of each group was registered); candidates inside a
tier keep registration order.
"""
from __future__ import annotations


def make_plan(cands):
    """cands: list of dicts {index, group, group_prio, prio, supported}.

    Returns [(group, [[indices of tier 0], [tier 1], ...]), ...] in try order.
    """
    order = []
    gprio = {}
    members = {}
    for c in cands:
        g = c["group"]
        if g not in members:
            order.append(g)
            members[g] = []
            gprio[g] = c["group_prio"]
        p = c["prio"]
        if p >= 0 and not c["supported"]:
            p = 0
        if p < 0:
            continue
        members[g].append((c["index"], p))
    groups = [g for g in order if gprio[g] >= 0 and members[g]]
    groups.sort(key=lambda g: -gprio[g])  # stable: registration order on ties
    plan = []
    for g in groups:
        tiers = sorted({p for _, p in members[g]}, reverse=True)
        plan.append((g, [[i for i, p in members[g] if p == t] for t in tiers]))
    return plan
