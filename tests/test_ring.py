"""Ring-buffer draft KV for window mode, host side: the ring size and the
block-table row the C ABI builds, and the property that makes it valid -- for
every context length, the pages window attention reads (the oracle's
selection) and the page the newest token is appended to map to distinct
physical pages."""
import os

import numpy as np
import pytest

import oracle.draft_attn_oracle as orc
from draft_attention_decode_b300 import binding as B

pytestmark = pytest.mark.skipif(not os.path.exists(B.LIB_PATH), reason="library not built")


@pytest.mark.parametrize("W,ns,want", [(2048, 0, (33, 0)), (2048, 4, (34, 1)), (4096, 4, (66, 1)),
                                       (1, 0, (2, 0)), (64, 64, (3, 1)), (65, 65, (5, 2))])
def test_ring_size(W, ns, want):
    assert B.draft_attn_ring_size(W, ns) == want


def test_ring_table_layout():
    ring = [40, 7, 13, 2, 99]
    t = B.draft_attn_ring_block_table(12, ring, 1)
    assert t.tolist() == [40, 7, 13, 2, 99, 7, 13, 2, 99, 7, 13, 2]
    t = B.draft_attn_ring_block_table(5, ring, 0)
    assert t.tolist() == [40, 7, 13, 2, 99]


def test_ring_rejects_bad_arguments():
    with pytest.raises(B.DraftAttnError):
        B.draft_attn_ring_size(0, 0)
    with pytest.raises(B.DraftAttnError):
        B.draft_attn_ring_size(16, -1)
    with pytest.raises(B.DraftAttnError):
        B.draft_attn_ring_block_table(4, [1, 2], 2)        # no window slot left
    with pytest.raises(B.DraftAttnError):
        B.draft_attn_ring_block_table(0, [1, 2], 0)


@pytest.mark.parametrize("W,ns", [(2048, 0), (2048, 4), (100, 3), (64, 0), (1, 1), (4096, 4),
                                  (130, 70)])
def test_window_reads_never_alias(W, ns):
    n_ring, n_sp = B.draft_attn_ring_size(W, ns)
    ring = np.arange(1000, 1000 + n_ring)
    max_pages = (W + ns) // 64 + 60
    table = B.draft_attn_ring_block_table(max_pages, ring, n_sp)
    Ls = sorted(set(range(1, 64 * (max_pages - 1), 7)) |
                {64 * k + d for k in range(max_pages - 1) for d in (-1, 0, 1) if 64 * k + d >= 1})
    for L in Ls:
        pos = orc.select_keys("window", L, W, ns)["loc"]
        pages = np.unique(pos // 64)
        newest = (L - 1) // 64          # the page the step's token was appended to
        assert newest in pages
        phys = table[pages]
        assert len(np.unique(phys)) == len(pages), L
        # the last page written into each read page's slot (appends go in page
        # order) must be that page itself, or its contents were overwritten
        for pg in pages:
            writers = np.nonzero(table[: newest + 1] == table[pg])[0]
            assert writers.max() == pg, (L, pg)
