"""Host-side check of the split-KV work partition the decode kernel uses.

The pages of every (sequence b, KV head h) are laid end to end (b outer, then
h, then range 0 before range 1); with TP pages in all, n = min(grid,
ceil(TP / 4)) CTAs are active and CTA i takes [floor(i*TP/n),
floor((i+1)*TP/n)).  A piece is one CTA's part of one (b, h, segment), where
FOLD's two ranges are two segments and every other mode has one; it writes
slot cta + seq with seq = (b*H + h)*2 + segment.  Checks, for many shapes,
that the pieces written are exactly the pieces the merge reads (CTAs with
empty stretches skipped), that slots are unique and fit the workspace
(grid + 2*B*H), that every CTA gets floor or ceil of TP / n pages, and that
each (b, h)'s counter total equals the pages its pieces report."""
import random

MIN_PAGES_PER_CTA = 4


def begin(i, TP, n):
    return (i * TP) // n


def cta_of(x, TP, n):
    return ((x + 1) * n - 1) // TP


def active(TP, grid):
    want = (TP + MIN_PAGES_PER_CTA - 1) // MIN_PAGES_PER_CTA
    return max(1, min(want, grid))


def line(B, H, n0, n1, fold):
    """Owner (b, h, seq) of every flat position."""
    out = []
    for b in range(B):
        for h in range(H):
            for r, n in ((0, n0[b]), (1, n1[b])):
                seg = r if fold else 0
                out += [(b, h, (b * H + h) * 2 + seg)] * n
    return out


def check(B, H, n0, n1, fold, grid):
    own = line(B, H, n0, n1, fold)
    TP = len(own)
    if TP == 0:
        return
    n = active(TP, grid)
    written = {}
    for i in range(n):
        for x in range(begin(i, TP, n), begin(i + 1, TP, n)):
            b, h, seq = own[x]
            written.setdefault((i, seq), 0)
            written[(i, seq)] += 1
    read = set()
    start = 0
    for b in range(B):
        nb = n0[b] + n1[b]
        for h in range(H):
            x0 = start + h * nb
            segs = [(x0, n0[b], 0), (x0 + n0[b], n1[b], 1)] if fold else [(x0, nb, 0)]
            for beg, ln, seg in segs:
                if ln == 0:
                    continue
                for i in range(cta_of(beg, TP, n), cta_of(beg + ln - 1, TP, n) + 1):
                    if begin(i, TP, n) < begin(i + 1, TP, n):
                        read.add((i, (b * H + h) * 2 + seg))
        start += H * nb
    assert set(written) == read
    slots = [i + seq for i, seq in written]
    assert len(slots) == len(set(slots))
    assert max(slots) < grid + 2 * B * H
    sizes = [begin(i + 1, TP, n) - begin(i, TP, n) for i in range(n)]
    assert sum(sizes) == TP and max(sizes) - min(sizes) <= 1
    # page counters: each (b, h) collects exactly its n0 + n1 pages
    per_bh = {}
    for (i, seq), pages in written.items():
        per_bh[seq >> 1] = per_bh.get(seq >> 1, 0) + pages
    for b in range(B):
        for h in range(H):
            if n0[b] + n1[b]:
                assert per_bh[b * H + h] == n0[b] + n1[b]


def test_pieces_written_equal_pieces_read():
    rng = random.Random(0)
    for _ in range(1500):
        B = rng.randint(1, 6)
        H = rng.choice([1, 2, 3, 8])
        fold = rng.random() < 0.5
        n0 = [rng.choice([0, 0, 1, 2, 5, 33]) for _ in range(B)]
        n1 = [rng.choice([0, 1, 3, 32, 64, 200]) for _ in range(B)]
        grid = rng.choice([1, 2, 3, 7, 13, 148, 600])
        check(B, H, n0, n1, fold, grid)


def test_active_ctas():
    assert active(16392 * 8, 148) == 148          # full 128K: every SM
    assert active(32 * 8, 148) == 64              # 2048-token window over 8 heads
    assert active(65 * 8, 148) == 130             # 4096 + 4 window
    assert active(1, 148) == 1
