"""Draft-cap selection from a measured verify-cost curve (test infrastructure only).

Source: "Draft caps and calibration" (mlx-dspark docs), the cost model given
"in formula form, for a cap C" and the section "How mlx-dspark picks it":

    speedup(C) ~ accepted(C) / (drafter + verify(C + 1))
    accepted(C) = 1 + p + p^2 + ... + p^C     tokens committed per round
    verify(w)   = cost of one pass over w rows, in single-token steps

and the best fixed cap is the C that maximises speedup(C), derived from the
measured curves.

Readings taken where the page leaves a step open:

* Costs may be given in any unit (microseconds, say); they are expressed in
  single-token steps by dividing by verify(1), the cost of a plain decode step.
* C = 0 is plain decoding: nothing is drafted, one row is verified, one token
  is committed, so speedup(0) = 1 exactly (no drafter term).
* The drafter's cost is either one number for every C >= 1 (the formula's
  single term) or one number per cap, drafter[C].
* Ties go to the smaller cap (less work that may be thrown away).
* accepted(C) is summed term by term in float64, the same precision the
  library decides the argmax in.

parity pinned: tests/test_draft_cap.py checks accepted(C) against the
geometric-series closed form, the chosen cap against a worked example done by
hand, and the page's qualitative statements (a flat verify curve means
"draft a lot"; a costlier drafter never raises the cap).
"""

from __future__ import annotations


def accepted(p: float, C: int) -> float:
    """Expected tokens committed per round with cap C: 1 + p + ... + p^C."""
    total, term = 0.0, 1.0
    for _ in range(C + 1):
        total += term
        term *= p
    return total


def speedups(p: float, verify, drafter, max_cap: int):
    """speedup(C) for C = 0 .. the largest cap the inputs allow (see module doc)."""
    verify = [float(x) for x in verify]
    drafter = [float(x) for x in drafter]
    limit = min(int(max_cap), len(verify) - 1)
    if len(drafter) > 1:
        limit = min(limit, len(drafter) - 1)
    step = verify[0]
    out = [1.0]
    for C in range(1, limit + 1):
        d = drafter[0] if len(drafter) == 1 else drafter[C]
        out.append(accepted(p, C) * step / (d + verify[C]))
    return out


def select_draft_cap(p: float, verify, drafter, max_cap: int):
    """(best cap, speedups): the C of largest speedup, the smaller on a tie."""
    s = speedups(p, verify, drafter, max_cap)
    best = 0
    for C in range(1, len(s)):
        if s[C] > s[best]:
            best = C
    return best, s
