"""A model of how the fused attention-norm and RoPE-table launch deals out its blocks, written out in
Python: groups of K norm blocks and one table block, then the norm blocks left over (K = norm blocks
// table blocks, 0 putting the table blocks first); a table block covers 8 passes of 256 / (hd/2)
positions.  Every norm block index and every table block appears exactly once, and every position of
the call gets its (cos, sin) row.  This checks the scheme; the GPU parity tests check the kernel."""
import pytest

PASSES = 8


def block_roles(norm_blocks, tab_blocks):
    K = norm_blocks // tab_blocks
    lead = tab_blocks * (K + 1)
    norms, tabs = [], []
    for b in range(norm_blocks + tab_blocks):
        if b < lead:
            grp, pos = divmod(b, K + 1)
            (tabs.append(grp) if pos == K else norms.append(grp * K + pos))
        else:
            norms.append(tab_blocks * K + (b - lead))
    return norms, tabs


@pytest.mark.parametrize("rows,S,hd", [(8192, 8192, 128), (512, 256, 64), (600, 300, 64), (8, 4, 2),
                                       (16384, 2048, 128), (4096, 4096, 96), (9, 9, 256)])
def test_every_norm_block_and_position_once(rows, S, hd):
    half = hd // 2
    per = 256 // half
    norm_blocks = (rows + 7) // 8
    tab_blocks = (S + per * PASSES - 1) // (per * PASSES)
    norms, tabs = block_roles(norm_blocks, tab_blocks)
    assert sorted(norms) == list(range(norm_blocks))
    assert sorted(tabs) == list(range(tab_blocks))
    covered = [(t * PASSES + p) * per + j for t in tabs for p in range(PASSES) for j in range(per)]
    assert sorted(s for s in covered if s < S) == list(range(S))
