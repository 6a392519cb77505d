"""Host-side checks of the stream-K work split (no GPU needed).

The kernels split the stream of work units (prepared tiles, row tile after
row tile) over the CTAs in chunks of one or two units, as evenly as the
chunks allow, the first CTAs taking one chunk more.  A CTA writes a row tile's
outputs itself when its run covers the whole row tile, else it stores its
partial sums in one of its two slots: side 0 for the first row tile of its
run (the one that began at or before its first unit), side 1 for the last.
The host plan tells every contributor of a shared row tile where the other
contributors' slots are and which rows it finishes: an even slice each, or,
for small tiles, all of them by the one contributor that holds the finisher
flag.  These tests replay the
kernels' owner/side rule against the plan that the library computes and
check that every output row is produced exactly once from every unit."""
import pytest

from bit_weight_only_gb300 import build, qgemv


@pytest.fixture(scope="module")
def lib():
    build.build()
    return qgemv.load()


def split(c, U, G, unit=1):
    """Start of CTA c's run: the kernels' stream_split, restated."""
    if unit == 0:
        return c * U // G
    n = -(-U // unit)
    q, r = divmod(n, G)
    return min((c * q + min(c, r)) * unit, U)


def kernel_view(U, G, upr, unit=1):
    """What each CTA's kernel does: per row tile, the CTAs that store a
    partial (with the slot side they use) and the CTA that writes y."""
    writers, partials = {}, {}
    for c in range(G):
        u0, u1 = split(c, U, G, unit), split(c + 1, U, G, unit)
        for rt in range(u0 // upr, (u1 - 1) // upr + 1):
            owner = rt * upr >= u0 and (rt + 1) * upr <= u1
            if owner:
                writers.setdefault(rt, []).append(c)
            else:
                side = 0 if rt * upr <= u0 else 1
                lo, hi = max(u0, rt * upr), min(u1, (rt + 1) * upr)
                partials.setdefault(rt, []).append((c, side, lo, hi))
    return writers, partials


CASES = [
    # (units = tiles, grid, tiles per row tile, rows)
    (32 * 8, 152, 8, 128),          # 4096 x 4096 CBK4: 32 row tiles x 8 k tiles
    (258 * 8, 152, 8, 128),         # 33024-row stack, 8 k tiles per row tile
    (86 * 22, 152, 22, 128),        # 11008-wide down projection (Q4_0 / CBK4)
    (7, 7, 1, 128),                 # one k tile per row tile, grid = tiles
    (3 * 50, 152, 50, 128),         # long row tiles: several CTAs share each
    (1000, 999, 10, 128),           # almost one tile per CTA
    (35 * 4, 140, 4, 2048),         # AQLM units of 2048 rows
    (17, 17, 17, 128),              # one row tile, one tile per CTA
    # GLU handles: the finisher's row slices count gate/up pairs (64 per tile)
    (172 * 8, 304, 8, 64),          # 7B gate|up interleaved (11008 pairs), Q4_0, two CTAs per SM
    (32, 32, 32, 64),               # one row tile split over 32 CTAs (the lost-CTA test's shape)
    (272 * 5, 304, 5, 64),          # 17408 pairs x 5120, PQ2_0
]


@pytest.mark.parametrize("unit", [0, 1, 2])
@pytest.mark.parametrize("U, G, upr, rows", CASES)
def test_plan_matches_the_kernels_split(lib, U, G, upr, rows, unit):
    G = min(G, U)
    plan = qgemv.qgemv_stream_k_plan(U, G, upr, rows, unit)
    writers, partials = kernel_view(U, G, upr, unit)
    n_rt = U // upr
    for rt in range(n_rt):
        w, parts = writers.get(rt, []), partials.get(rt, [])
        # every unit of the row tile is covered once, by one writer or by partials
        if w:
            assert len(w) == 1 and not parts
            continue
        covered = sorted((lo, hi) for _, _, lo, hi in parts)
        assert covered[0][0] == rt * upr and covered[-1][1] == (rt + 1) * upr
        assert all(a[1] == b[0] for a, b in zip(covered, covered[1:]))
        ctas = [c for c, _, _, _ in parts]
        assert ctas == list(range(ctas[0], ctas[0] + len(ctas)))
        # each contributor's plan names this row tile once, with the same
        # contributors, and the slot the first contributor really used
        rows_done = []
        for c, side, _, _ in parts:
            segs = [s for s in range(2) if plan[c]["rt"][s] == rt]
            assert len(segs) == 1, (rt, c, plan[c])
            s = segs[0]
            assert plan[c]["cf"][s] == ctas[0]
            assert plan[c]["S"][s] == len(ctas)
            first_side = [sd for cc, sd, _, _ in parts if cc == ctas[0]][0]
            assert plan[c]["side1"][s] == first_side
            # the later contributors used side 0 (the row tile began before them)
            if c != ctas[0]:
                assert side == 0
            rows_done.extend(range(plan[c]["r0"][s], plan[c]["r0"][s] + plan[c]["nr"][s]))
        assert sorted(rows_done) == list(range(rows))
        # one finisher for the whole-tile mode: a contributor whose part closes
        # its run (the last one, unless its part opens a run that goes on)
        fins = [c for c, _, _, _ in parts
                if plan[c]["fin"][[s for s in range(2) if plan[c]["rt"][s] == rt][0]]]
        assert len(fins) == 1, (rt, fins)
        fc = fins[0]
        hi_of = {c: hi for c, _, _, hi in parts}
        assert hi_of[fc] == split(fc + 1, U, G, unit)
        cl = ctas[-1]
        assert fc == (cl - 1 if split(cl + 1, U, G, unit) > (rt + 1) * upr else cl)
    # a CTA's plan names no row tile that it does not share
    for c in range(G):
        for s in range(2):
            rt = plan[c]["rt"][s]
            if rt >= 0:
                assert any(cc == c for cc, _, _, _ in partials.get(rt, []))


@pytest.mark.parametrize("unit", [1, 2])
def test_plan_is_balanced_to_one_chunk_first_ctas_first(lib, unit):
    for U, G in [(258 * 8, 152), (96 * 8, 152), (172 * 8, 152), (32 * 22, 152), (1001, 152)]:
        sizes = [split(c + 1, U, G, unit) - split(c, U, G, unit) for c in range(G)]
        assert sum(sizes) == U and split(G, U, G, unit) == U
        # one chunk apart, and the stream's last chunk may be short
        assert max(sizes) - min(sizes) <= 2 * unit - 1
        # the larger runs come first (the CTAs placed first)
        assert sizes == sorted(sizes, reverse=True) or sizes[-1] < unit
        # chunks of two start on even units
        assert all(split(c, U, G, unit) % unit == 0 or split(c, U, G, unit) == U for c in range(G))


@pytest.mark.parametrize("args", [(0, 1, 1, 128), (10, 11, 10, 128), (12, 2, 5, 128), (10, 2, 5, 0)])
def test_plan_rejects_bad_sizes(lib, args):
    with pytest.raises(qgemv.QgemvError):
        qgemv.qgemv_stream_k_plan(*args)
