"""Host-side check of the split-KV work partition the kernels use: the pages
of every (sequence, range, KV head) are laid end to end and CTA i of n takes
[floor(i*TP/n), floor((i+1)*TP/n)); a piece (CTA, sequence) writes slot
cta + sequence.  Checks, for many shapes, that the pieces written are exactly
the pieces the combine reads (CTAs with empty ranges skipped), that slots
are unique and that they fit the workspace (n + number of sequences)."""
import random


def begin(i, TP, n):
    return (i * TP) // n


def cta_of(x, TP, n):
    return ((x + 1) * n - 1) // TP


def test_pieces_written_equal_pieces_read():
    rng = random.Random(0)
    for _ in range(2000):
        n = rng.choice([1, 2, 3, 5, 7, 13, 148, 300])
        seqs = [rng.choice([0, 0, 1, 2, 3, 5, 64, 1000]) for _ in range(rng.randint(1, 40))]
        TP = sum(seqs)
        if TP == 0:
            continue
        starts = [0]
        for s in seqs:
            starts.append(starts[-1] + s)
        owner = []
        for s, npg in enumerate(seqs):
            owner += [s] * npg
        written = set()
        for i in range(n):
            for x in range(begin(i, TP, n), begin(i + 1, TP, n)):
                written.add((i, owner[x]))
        read = set()
        for s, npg in enumerate(seqs):
            if npg == 0:
                continue
            x0 = starts[s]
            for i in range(cta_of(x0, TP, n), cta_of(x0 + npg - 1, TP, n) + 1):
                if begin(i, TP, n) < begin(i + 1, TP, n):
                    read.add((i, s))
        assert written == read
        slots = [i + s for i, s in written]
        assert len(slots) == len(set(slots))
        assert max(slots) < n + len(seqs)


def test_balance():
    """Every CTA gets floor or ceil of TP / n pages."""
    for TP in (1, 7, 16392, 131080, 355000):
        for n in (1, 148, 296):
            sizes = [begin(i + 1, TP, n) - begin(i, TP, n) for i in range(n)]
            assert sum(sizes) == TP and max(sizes) - min(sizes) <= 1
