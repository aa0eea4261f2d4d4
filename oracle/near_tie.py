"""Near-tie bookkeeping for decisions taken on derived floating-point values.

TEST INFRASTRUCTURE ONLY -- see the package docstring.

The library computes node values and probabilities from fp32 inputs with its
own rounding order; the oracle computes them in fp64.  A decision whose two
operands lie within ``REL_TOL`` (relative) of each other can legitimately
come out differently on the two sides, so every such decision is recorded
here with its margin and reported by the parity tests instead of being
silently passed.  Decisions on raw input values (comparisons of two fp32
logits) are exact on both sides and are recorded with ``exact=True``.
"""

REL_TOL = 1e-6


def rel_margin(a, b):
    """|a - b| / max(|a|, |b|), 0 when both are zero."""
    a = float(a)
    b = float(b)
    scale = max(abs(a), abs(b))
    if scale == 0.0:
        return 0.0
    return abs(a - b) / scale


class NearTieLog:
    """Collects (kind, where, a, b, margin) for decisions within REL_TOL."""

    def __init__(self):
        self.flags = []
        self.n_checked = 0

    def check(self, kind, where, a, b, exact=False):
        self.n_checked += 1
        m = rel_margin(a, b)
        if m <= REL_TOL:
            self.flags.append(dict(kind=kind, where=where, a=float(a), b=float(b),
                                   margin=m, exact=bool(exact)))
        return m

    @property
    def inexact_flags(self):
        return [f for f in self.flags if not f["exact"]]

    def __bool__(self):
        return bool(self.inexact_flags)

    def summary(self):
        return "; ".join(f"{f['kind']}@{f['where']} margin={f['margin']:.3g}"
                         for f in self.inexact_flags)
