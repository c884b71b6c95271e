"""Host-side check of the split-KV work partition the decode kernel uses.

The pages of every (sequence b, KV head h) are laid end to end (b outer, then
h, then ranges 0, 1, 2 in turn); with TP pages in all, n = min(grid,
ceil(TP / min_pages)) CTAs are active and CTA i takes [floor(i*TP/n),
floor((i+1)*TP/n)).  A piece is one CTA's part of one (b, h, segment): FOLD's
range 0 (far memory) is one segment and its ranges 1 and 2 (sinks and window)
the other; every other mode has one segment.  A piece writes slot cta + seq
with seq = (b*H + h)*2 + segment.  Checks, for many shapes, split floors and
grids, that the pieces written are exactly the pieces the merge reads (CTAs
with empty stretches skipped), that slots are unique and fit the workspace
(grid + 2*B*H), that every CTA gets floor or ceil of TP / n pages, and that
each (b, h)'s counter total equals the pages its pieces report."""
import random


def begin(i, TP, n):
    return (i * TP) // n


def cta_of(x, TP, n):
    return ((x + 1) * n - 1) // TP


def active(TP, grid, min_pages=1):
    want = (TP + min_pages - 1) // min_pages
    return max(1, min(want, grid))


def line(B, H, n, fold):
    """Owner (b, h, seq) of every flat position; n[r][b] pages of range r."""
    out = []
    for b in range(B):
        for h in range(H):
            for r in range(3):
                seg = (1 if r else 0) if fold else 0
                out += [(b, h, (b * H + h) * 2 + seg)] * n[r][b]
    return out


def check(B, H, n, fold, grid, min_pages):
    own = line(B, H, n, fold)
    TP = len(own)
    if TP == 0:
        return
    na = active(TP, grid, min_pages)
    written = {}
    for i in range(na):
        for x in range(begin(i, TP, na), begin(i + 1, TP, na)):
            b, h, seq = own[x]
            written.setdefault((i, seq), 0)
            written[(i, seq)] += 1
    # what merge_sequence reads: the far range, then the rest (FOLD); or all
    read = set()
    start = 0
    for b in range(B):
        nb = n[0][b] + n[1][b] + n[2][b]
        n0 = n[0][b] if fold else nb
        for h in range(H):
            x0 = start + h * nb
            for beg, ln, seg in ((x0, n0, 0), (x0 + n0, nb - n0, 1)):
                if ln == 0:
                    continue
                for i in range(cta_of(beg, TP, na), cta_of(beg + ln - 1, TP, na) + 1):
                    if begin(i, TP, na) < begin(i + 1, TP, na):
                        read.add((i, (b * H + h) * 2 + seg))
        start += H * nb
    assert set(written) == read
    slots = [i + seq for i, seq in written]
    assert len(slots) == len(set(slots))
    assert max(slots) < grid + 2 * B * H
    sizes = [begin(i + 1, TP, na) - begin(i, TP, na) for i in range(na)]
    assert sum(sizes) == TP and max(sizes) - min(sizes) <= 1
    # page counters: each (b, h) collects exactly its pages over all ranges
    per_bh = {}
    for (i, seq), pages in written.items():
        per_bh[seq >> 1] = per_bh.get(seq >> 1, 0) + pages
    for b in range(B):
        for h in range(H):
            tot = n[0][b] + n[1][b] + n[2][b]
            if tot:
                assert per_bh[b * H + h] == tot


def test_pieces_written_equal_pieces_read():
    rng = random.Random(0)
    for _ in range(1500):
        B = rng.randint(1, 6)
        H = rng.choice([1, 2, 3, 8])
        fold = rng.random() < 0.5
        n = [[rng.choice([0, 0, 1, 2, 5, 33]) for _ in range(B)],
             [rng.choice([0, 0, 1, 2]) for _ in range(B)],        # FOLD's sinks / window's window
             [rng.choice([0, 1, 3, 32, 64, 200]) for _ in range(B)]]
        grid = rng.choice([1, 2, 3, 7, 13, 148, 600])
        check(B, H, n, fold, grid, rng.choice([1, 1, 2, 4]))


def test_active_ctas():
    assert active(16392 * 8, 148) == 148          # full 128K: every SM
    assert active(33 * 8, 148) == 148             # 2048-token window over 8 heads
    assert active(33 * 8, 148, 4) == 66           # the same with a split floor of 4
    assert active(1, 148) == 1
