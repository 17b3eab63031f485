"""Host check of the batch-1 streaming contract between the loader, the consumer warps and the
bind-time capacity rule (no GPU).

At batch 1 a matvec tile streams through the page ring: every page holds whole rows (gate/up:
the gate rows and the up rows of one row group in two consecutive pages), and the consumer warps
walk the pages in groups of two, each warp waiting for the group's pages and giving them back
when done.  Warp w computes segment w mod G of every row it touches (G, the segments per row,
depends on the row length only) and units (row, segment) j = w, w + 8, ... of each page.  This
test restates that mapping for every batch-1 matvec tile of every workload (rows per tile from the
scheduler's restatement) and checks that the pages cover the rows exactly once in order, that
every (row, segment) unit is computed by exactly one warp that always holds the same segment, that
a page's units fit the shared partial area the bind sizes (every unit leaves a partial), and that the bind's page rule (two
pages per step, plus an attention tile) fits the 6-page ring of the default 32 KB pages.
"""
import pytest

from oracle import schedule_ref as sr
from workload import WORKLOADS, get_workload

PB = 32768          # default page bytes
N_PAGES = 6         # pages the 1B / 8B configurations get from the 227 KB of shared memory
WARPS = 8           # consumer warps
MAX_SEG = 8


def cpl_of(cfg):
    """16-byte chunks a lane holds of its segment: 4 when the longest row fits 8 segments of 128
    chunks, else 8."""
    kmax = max(cfg.hidden, cfg.q_dim, cfg.ffn)
    return 4 if -(-(kmax // 8) // MAX_SEG) <= 128 else 8


def segments(K, cpl):
    """Segments per row: the smallest power of two keeping a segment within 32 * cpl chunks."""
    chunks, G = K // 8, 1
    while -(-chunks // G) > 32 * cpl and G < MAX_SEG:
        G *= 2
    return G


def tile_groups(op, rows, K):
    """Yields, per two-page group, the tile rows in each page (a list of two lists)."""
    rpp = PB // (2 * K)
    assert rpp >= 1
    pair = op == sr.UPGATE
    n_pages = -(-rows // rpp) * (2 if pair else 1)
    for k in range(0, n_pages, 2):
        pages = []
        for pg in (k, k + 1):
            if pg >= n_pages:
                pages.append([])
                continue
            grp = pg // 2 if pair else pg
            pages.append(list(range(grp * rpp, min(rows, (grp + 1) * rpp))))
        yield pages
    return n_pages


def bind_rule_pages(cfg, chunk):
    """The bind's page rule at batch 1 (restated): a group of two pages, or an attention tile."""
    return max(2, -(-(2 * chunk * cfg.head_dim * 2) // PB))


@pytest.mark.parametrize("name", [w for w in WORKLOADS if get_workload(w).cfg.batch == 1])
@pytest.mark.parametrize("S", [1, 37, 152])
def test_batch1_groups_cover_every_unit_once(name, S):
    cfg = get_workload(name).cfg
    o = sr.SchedOpts()
    tiles, _, _ = sr.enumerate_tiles(cfg, o, S)
    K = {sr.QKV: cfg.hidden, sr.OPROJ: cfg.q_dim, sr.UPGATE: cfg.hidden, sr.DOWN: cfg.ffn,
         sr.LMHEAD: cfg.hidden}
    cpl = cpl_of(cfg)
    comb_stride = max((PB // (2 * k)) * segments(k, cpl) for k in K.values())
    seen = 0
    for t in tiles:
        if t.op not in K:
            continue
        k_len = K[t.op]
        G = segments(k_len, cpl)
        lg = G.bit_length() - 1
        chunks = k_len // 8
        segch = -(-chunks // G)
        assert segch <= 32 * cpl and WARPS % G == 0
        done = {}
        pages_seen = 0
        for pages in tile_groups(t.op, t.a1, k_len):
            pages_seen += sum(1 for p in pages if p)
            for pi, prow in enumerate(pages):
                units = len(prow) << lg
                assert units <= comb_stride   # the page slot's partial area holds every unit
                for w in range(WARPS):
                    for j in range(w, units, WARPS):
                        assert j % G == w % G            # a warp keeps its own segment
                        key = (pi if t.op == sr.UPGATE else 0, prow[j >> lg], j % G)
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


def test_segments_depend_on_the_row_length_and_configuration_only():
    Ks = (256, 688, 1024, 2048, 4096, 8192, 14336, 16384)
    assert [segments(k, 4) for k in Ks[:6]] == [1, 1, 1, 2, 4, 8]
    assert [segments(k, 8) for k in Ks] == [1, 1, 1, 1, 2, 4, 8, 8]
    assert {w: cpl_of(get_workload(w).cfg) for w in WORKLOADS} == {
        "tiny": 4, "llama1b_ctx512": 4, "llama1b_ctx8192": 4, "llama1b_batch8": 4, "llama8b_ctx2048": 8}
