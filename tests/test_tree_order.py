"""The pairwise (tree) summation order as the fold kernel builds it.

The oracle adds neighbours level by level and carries an odd last value up;
the brute-force formulation splits recursively at the largest power of two
below the count; the kernel cannot hold a whole level, so it runs a binary
counter: contribution q merges the partials of the set bits below the lowest
clear bit of q, and at the end the partials left (one per set bit of W) are
added from the lowest level up, the earlier ranks on the left.  Stage fills of
a power-of-two number of ranks, starting at multiples of it, are complete
subtrees of that counter.  This checks symbolically that all of these build
the same expression for every world size the library accepts."""


def _levelwise(xs):
    xs = list(xs)
    while len(xs) > 1:
        nxt = [f"({xs[2 * i]}+{xs[2 * i + 1]})" for i in range(len(xs) // 2)]
        if len(xs) % 2:
            nxt.append(xs[-1])
        xs = nxt
    return xs[0]


def _split(xs):
    if len(xs) == 1:
        return xs[0]
    h = 1
    while 2 * h < len(xs):
        h *= 2
    return f"({_split(xs[:h])}+{_split(xs[h:])})"


def _counter(xs):
    slot = {}
    for q, x in enumerate(xs):
        carry, lvl = x, 0
        while (q >> lvl) & 1:
            carry = f"({slot.pop(lvl)}+{carry})"
            lvl += 1
        slot[lvl] = carry
    out = None
    for lvl in range(len(xs).bit_length()):
        if (len(xs) >> lvl) & 1:
            out = slot[lvl] if out is None else f"({slot[lvl]}+{out})"
    return out


def _counter_by_fills(xs, rg):
    """The kernel's two-level form: a counter over each fill of rg ranks
    (rg a power of two), then a counter over the complete fills' partials;
    a last, partial fill is folded by itself and then joins the fill
    partials from the lowest level up."""
    W = len(xs)
    nfull, rem = divmod(W, rg)
    fills = [_counter(xs[g * rg:(g + 1) * rg]) for g in range(nfull)]
    out = _counter(xs[nfull * rg:]) if rem else None
    slot = {}
    for g, f in enumerate(fills):
        carry, lvl = f, 0
        while (g >> lvl) & 1:
            carry = f"({slot.pop(lvl)}+{carry})"
            lvl += 1
        slot[lvl] = carry
    for lvl in range(nfull.bit_length()):
        if (nfull >> lvl) & 1:
            out = slot[lvl] if out is None else f"({slot[lvl]}+{out})"
    return out


def test_tree_constructions_agree():
    for W in range(1, 1025):
        xs = [f"x{i}" for i in range(W)]
        want = _levelwise(xs)
        assert _split(xs) == want, W
        assert _counter(xs) == want, W
        for rg in (1, 2, 4, 8):
            if rg <= W:
                assert _counter_by_fills(xs, rg) == want, (W, rg)
