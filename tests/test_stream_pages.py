"""Host check of the batch-1 streaming contract between the loader, the consumer warps and the
bind-time capacity rule (no GPU).

At batch 1 a matvec tile streams through the page ring: a consumer warp waits for the pages of
its next step and gives back every page no later step reads, so the slowest warp can always
progress as long as the pages one step touches fit the ring.  The bind accepts a schedule only
when its rule for those pages fits; this test walks every batch-1 matvec tile of every workload
(rows per tile from the scheduler's restatement) through the unit -> byte -> page mapping the
consumer warps use -- 16 row segments or 8 gate/up pairs per step, gate/up rows interleaved by
page -- and checks that every step's page span stays within the rule, that the steps cover the
tile's pages in order, and that the rule fits the 6-page ring of the default 32 KB pages.
"""
import pytest

from oracle import schedule_ref as sr
from workload import WORKLOADS, get_workload

PB = 32768          # default page bytes
N_PAGES = 6         # pages the 1B / 8B configurations get from the 227 KB of shared memory


def nseg_of(K):
    n = 1
    while K > 2048 * n:
        n *= 2
    return n


def bind_rule_pages(cfg, chunk):
    """The bind's upper bound of the pages one batch-1 step can touch (restated)."""
    def span(nbytes):
        n = -(-nbytes // PB)
        return n if (nbytes % PB == 0 or PB % nbytes == 0) else n + 1
    need = 2
    for K in (cfg.hidden, cfg.q_dim, cfg.ffn):
        need = max(need, span(16 * (2 * K // nseg_of(K))))
    rpp = PB // (2 * cfg.hidden)
    groups = max(1, 8 // rpp) if (rpp % 8 == 0 or 8 % rpp == 0) else -(-8 // rpp) + 1
    need = max(need, 2 * groups)
    need = max(need, -(-(2 * chunk * cfg.head_dim * 2) // PB))
    return need


def step_spans(op, rows, K):
    """(first page, last page) of every step of a batch-1 tile of `rows` rows (pairs for gate/up)
    of length K, and the tile's page count, as the loader lays the stream out."""
    pair = op == sr.UPGATE
    nseg = nseg_of(K)
    split = nseg > 1
    lognseg = nseg.bit_length() - 1
    rowbytes = 2 * K
    segbytes = rowbytes // nseg
    rpp = PB // rowbytes
    U = rows * nseg if split else rows
    per_step = 8 if pair else 16

    def unit_off(u, s):
        row = (u >> lognseg) if split else u
        if pair:
            return (row // rpp) * 2 * PB + (row % rpp) * rowbytes + s * segbytes
        return row * rowbytes + s * segbytes

    spans = []
    for k in range(-(-U // per_step)):
        u0 = k * per_step
        first = unit_off(u0, (u0 & (nseg - 1)) if split else 0) // PB
        u1 = min(U, (k + 1) * per_step) - 1
        if pair:
            last = unit_off(u1, (u1 & (nseg - 1)) if split else 0) // PB + 1
        else:
            last = (unit_off(u1, (u1 & (nseg - 1)) if split else nseg - 1) + segbytes - 1) // PB
        spans.append((first, last))
    n_pages = 2 * -(-rows // rpp) if pair else -(-(rows * rowbytes) // PB)
    return spans, n_pages


@pytest.mark.parametrize("name", [w for w in WORKLOADS if get_workload(w).cfg.batch == 1])
@pytest.mark.parametrize("S", [1, 37, 152])
def test_batch1_steps_fit_the_bind_rule(name, S):
    cfg = get_workload(name).cfg
    o = sr.SchedOpts()
    tiles, _, _ = sr.enumerate_tiles(cfg, o, S)
    need = bind_rule_pages(cfg, sr.attn_chunk(cfg, o, S))
    K = {sr.QKV: cfg.hidden, sr.OPROJ: cfg.q_dim, sr.UPGATE: cfg.hidden, sr.DOWN: cfg.ffn,
         sr.LMHEAD: cfg.hidden}
    seen = 0
    for t in tiles:
        if t.op not in K:
            continue
        if 2 * K[t.op] > PB and t.op == sr.UPGATE:
            continue   # (rejected at schedule time: a page must hold a gate/up row)
        spans, n_pages = step_spans(t.op, t.a1, K[t.op])
        prev_first = 0
        for first, last in spans:
            assert first >= prev_first and first <= last < n_pages, (t, first, last, n_pages)
            assert last - first + 1 <= need, (name, t.op, t.a1, first, last, need)
            prev_first = first
        assert spans[0][0] == 0 and spans[-1][1] == n_pages - 1
        seen += 1
    assert seen > 0
    if name != "tiny":
        assert need <= N_PAGES
