"""Host check of the batch-1 streaming contract between the loader, the consumer warps and the
bind-time capacity rule (no GPU).

At batch 1 a matvec tile streams through the page ring: every page holds whole rows (a gate/up
page: the gate rows of its pairs, then their up rows), and each consumer warp waits for one page
at a time and gives it back when done.  Warp w computes segment w mod G of every row it touches (G, the segments per row,
depends on the row length only) and units (row, segment) j = w, w + 16, ... of each page.  This
test restates that mapping for every batch-1 matvec tile of every workload (rows per tile from the
scheduler's restatement) and checks that the pages cover the rows exactly once in order, that
every (row, segment) unit is computed by exactly one warp that always holds the same segment, that
a page's units fit the shared partial area the bind sizes (every unit leaves a partial), and
that the bind's page rule (one page, or an attention tile) fits the 6-page ring of the default
32 KB pages.
"""
import pytest

from oracle import schedule_ref as sr
from workload import WORKLOADS, get_workload

PB = 32768          # default page bytes
N_PAGES = 6         # pages the 1B / 8B configurations get from the 227 KB of shared memory
WARPS = 16          # consumer warps
CPL = 4             # 16-byte chunks a lane holds of its segment, at most
MAX_SEG = 16


def segments(K):
    """Segments per row: the smallest power of two keeping a segment within 32 * CPL chunks."""
    chunks, G = K // 8, 1
    while -(-chunks // G) > 32 * CPL and G < MAX_SEG:
        G *= 2
    return G


def tile_pages(op, rows, K):
    """Yields, per page, the (side, tile row) pairs it holds in page order: side 0 a row (or a gate
    row), side 1 an up row."""
    rpp = PB // (2 * K)
    pair = op == sr.UPGATE
    if pair:
        rpp //= 2
    assert rpp >= 1
    for r0 in range(0, rows, rpp):
        n = min(rpp, rows - r0)
        yield [(0, r) for r in range(r0, r0 + n)] + ([(1, r) for r in range(r0, r0 + n)] if pair else [])


def bind_rule_pages(cfg, chunk):
    """The bind's page rule at batch 1 (restated): one page, or an attention tile's K and V rows."""
    return max(1, -(-(2 * chunk * cfg.head_dim * 2) // PB))


@pytest.mark.parametrize("name", [w for w in WORKLOADS if get_workload(w).cfg.batch == 1])
@pytest.mark.parametrize("S", [1, 37, 152])
def test_batch1_groups_cover_every_unit_once(name, S):
    cfg = get_workload(name).cfg
    o = sr.SchedOpts()
    tiles, _, _ = sr.enumerate_tiles(cfg, o, S)
    K = {sr.QKV: cfg.hidden, sr.OPROJ: cfg.q_dim, sr.UPGATE: cfg.hidden, sr.DOWN: cfg.ffn,
         sr.LMHEAD: cfg.hidden}
    comb_stride = max((PB // (2 * k)) * segments(k) for k in K.values())
    seen = 0
    for t in tiles:
        if t.op not in K:
            continue
        k_len = K[t.op]
        G = segments(k_len)
        lg = G.bit_length() - 1
        chunks = k_len // 8
        segch = -(-chunks // G)
        assert segch <= 32 * CPL and WARPS % G == 0
        done = {}
        pages_seen = 0
        for prow in tile_pages(t.op, t.a1, k_len):
            pages_seen += 1
            units = len(prow) << lg
            assert units <= comb_stride   # the page slot's partial area holds every unit
            assert len(prow) * 2 * k_len <= PB
            for w in range(WARPS):
                for j in range(w, units, WARPS):
                    assert j % G == w % G            # a warp keeps its own segment
                    side, row = prow[j >> lg]
                    key = (side, row, j % G)
                    done[key] = done.get(key, 0) + 1
        # every (row, segment) -- for gate/up, of the gate and the up row -- exactly once
        sides = 2 if t.op == sr.UPGATE else 1
        assert sorted(done) == sorted((side, r, s) for side in range(sides) for r in range(t.a1)
                                      for s in range(G))
        assert set(done.values()) == {1}
        assert pages_seen == sr.tile_pages(t, cfg, o)
        seen += 1
    assert seen > 0
    assert bind_rule_pages(cfg, sr.attn_chunk(cfg, o, S)) <= N_PAGES


def test_segments_depend_on_the_row_length_only():
    assert [segments(k) for k in (256, 688, 1024, 2048, 4096, 8192, 14336, 16384)] == [1, 1, 1, 2, 4, 8, 16, 16]
