"""The host scheduler (C++, in libmk.so) against its independent restatement on the oracle side,
the schedule validator and the host simulator of the queue interpreter (no GPU).

Bit-exact: the C++ queues [S, Q, 32] and per-step counter totals equal the restatement's, for
every workload, several SM counts and the shuffled placement."""
import numpy as np
import pytest

from oracle import schedule_ref as sr
from workload import WORKLOADS, get_workload, small_config

mk = pytest.importorskip("persistent_megakernel_decode_sm_gb300")

SMS = [1, 2, 7, 37, 132, 148, 152]


@pytest.mark.parametrize("name", WORKLOADS)
@pytest.mark.parametrize("S", [1, 7, 37, 152])
def test_cpp_schedule_bit_exact_vs_restatement(name, S):
    cfg = get_workload(name).cfg
    s = mk.Schedule(cfg, S)
    q, t, _ = sr.build_schedule(cfg, S)
    assert np.array_equal(s.queues(), q)
    assert np.array_equal(s.totals(), t)


def test_default_attention_chunk_depends_on_the_configuration_only():
    """128 positions, doubled up to 512 while a layer has more than 152 chunks -- whatever the SM
    count, so outputs stay bit-identical across SM counts."""
    expect = {"tiny": 128, "llama1b_ctx512": 128, "llama1b_reduced": 128, "llama8b_ctx2048": 128,
              "llama1b_ctx8192": 512, "llama1b_batch8": 512}
    for name, C in expect.items():
        cfg = get_workload(name).cfg
        for S in (1, 37, 152, 1000):
            assert mk.Schedule(cfg, S).attn_chunk == C, (name, S)
            assert sr.attn_chunk(cfg, sr.SchedOpts(), S) == C, (name, S)
        assert mk.Schedule(cfg, 152, attn_chunk=32).attn_chunk == 32


@pytest.mark.parametrize("seed", [1, 12345, 2 ** 63 + 17])
def test_cpp_shuffled_placement_bit_exact(seed):
    cfg = get_workload("llama1b_ctx512").cfg
    s = mk.Schedule(cfg, 148, shuffle_seed=seed)
    q, t, _ = sr.build_schedule(cfg, 148, sr.SchedOpts(shuffle_seed=seed))
    assert np.array_equal(s.queues(), q) and np.array_equal(s.totals(), t)


@pytest.mark.parametrize("kw", [dict(kv_limit=[100, 300, 1, 233]), dict(kv_limit=[65, 0, 7], shuffle_seed=5),
                                dict(page_bytes=16384, tile_bytes=32768, attn_chunk=32),
                                dict(rows_qkv=4, rows_o=3, pairs_up=5, rows_down=7, rows_lm=9),
                                dict(attn_chunk=100)])
def test_cpp_knobs_bit_exact(kw):
    cfg = small_config(n_layers=3, max_seq=300)
    s = mk.Schedule(cfg, 11, **kw)
    q, t, _ = sr.build_schedule(cfg, 11, sr.SchedOpts(**kw))
    assert np.array_equal(s.queues(), q) and np.array_equal(s.totals(), t)


@pytest.mark.parametrize("name", ["tiny", "llama1b_ctx512", "llama1b_batch8"])
@pytest.mark.parametrize("S,seed", [(152, 0), (37, 0), (5, 99)])
def test_schedule_valid_and_deadlock_free(name, S, seed):
    cfg = get_workload(name).cfg
    q, t, _ = sr.build_schedule(cfg, S, sr.SchedOpts(shuffle_seed=seed))
    assert sr.validate(q, t, cfg, sr.SchedOpts(shuffle_seed=seed)) == []
    assert sr.simulate(q, t, cfg, n_epochs=2, seed=seed) == []


@pytest.mark.parametrize("name,S", [("tiny", 152), ("tiny", 7), ("llama1b_ctx512", 152), ("llama1b_batch8", 152)])
def test_schedule_tiles_cover_every_row_once(name, S):
    cfg = get_workload(name).cfg
    tiles, cnt, R = sr.enumerate_tiles(cfg, sr.SchedOpts(), S)
    for op, total in ((sr.QKV, cfg.qkv_rows), (sr.OPROJ, cfg.hidden), (sr.UPGATE, cfg.ffn),
                      (sr.DOWN, cfg.hidden), (sr.LMHEAD, cfg.vocab)):
        # (batch > 1 down projection of rows longer than a staging range: once per range)
        nrg = sr.down_ranges(cfg) if op == sr.DOWN else 1
        for l in (range(cfg.n_layers) if op != sr.LMHEAD else [cfg.n_layers]):
            rows = np.zeros((nrg, total), int)
            for t in tiles:
                if t.op == op and t.layer == l:
                    rows[t.a2 if op == sr.DOWN else 0, t.a0:t.a0 + t.a1] += 1
            assert np.all(rows == 1)


def test_batch1_wave_spread_one_matvec_tile_per_sm():
    # at batch 1 every matvec operator has at most S tiles and no SM holds two tiles of a wave
    cfg = get_workload("llama1b_ctx512").cfg
    S = 152
    q, t, _ = sr.build_schedule(cfg, S)
    for s in range(S):
        waves = [int(w[22]) for w in q[s] if w[0] != sr.END]
        assert len(waves) == len(set(waves)), f"sm {s} holds two tiles of one wave"
    n_up = sum(1 for s in range(S) for w in q[s] if w[0] == sr.UPGATE and w[1] == 0)
    assert n_up == -(-cfg.ffn // 56) <= S   # 54 pairs per SM, rounded up to whole groups of 8


def _mutate(q, fn):
    q = q.copy()
    fn(q)
    return q


def test_validator_and_simulator_catch_planted_errors():
    cfg = get_workload("tiny").cfg
    q, t, _ = sr.build_schedule(cfg, 5)
    # a dropped tile
    s0 = next(i for i in range(q.shape[1]) if q[0, i, 0] != 0)
    bad = _mutate(q, lambda a: a.__setitem__((0, s0), 0))
    assert sr.validate(bad, t, cfg)
    # a wait that asks for one more completion than the producers publish -> deadlock
    qi = [(s, i) for s in range(q.shape[0]) for i in range(q.shape[1]) if q[s, i, 6] > 0][0]
    bad = q.copy()
    bad[qi][8] += 1
    assert sr.validate(bad, t, cfg)
    assert any("deadlock" in e for e in sr.simulate(bad, t, cfg, n_epochs=1))
    # a wait removed: the simulator sees a read before its producer ran
    bad = q.copy()
    for s in range(q.shape[0]):
        for i in range(q.shape[1]):
            if q[s, i, 0] == sr.UPGATE:
                bad[s, i, 6] = 0
    # (some random interleaving runs an up/gate tile before its O rows are written)
    assert any(any("before" in e for e in sr.simulate(bad, t, cfg, n_epochs=1, seed=sd)) for sd in range(16))
    # per-SM wave order broken
    S_, Q_ = q.shape[0], q.shape[1]
    s = max(range(S_), key=lambda k: int((q[k, :, 0] != 0).sum()))
    n = int((q[s, :, 0] != 0).sum())
    bad = q.copy()
    bad[s, [0, n - 1]] = bad[s, [n - 1, 0]]
    assert sr.validate(bad, t, cfg)
    # batch > 1, down rows over two staging ranges: a range-0 tile relabelled as range 1 leaves
    # the last range's tile of those rows waiting for a partial nobody writes
    cfg = small_config(batch=2, ffn=4096, max_seq=64)
    q, t, _ = sr.build_schedule(cfg, 5)
    assert sr.down_ranges(cfg) == 2 and sr.simulate(q, t, cfg, n_epochs=1) == []
    at = next((s, i) for s in range(q.shape[0]) for i in range(q.shape[1]) if q[s, i, 0] == sr.DOWN and q[s, i, 5] == 0)
    bad = q.copy()
    bad[at][5] = 1
    assert sr.validate(bad, t, cfg)
    assert any("deadlock" in e for e in sr.simulate(bad, t, cfg, n_epochs=1))


def test_counter_totals_match_waits():
    cfg = get_workload("llama1b_ctx512").cfg
    q, t, info = sr.build_schedule(cfg, 152)
    cnt = info["counters"]
    L, B, nkv = cfg.n_layers, cfg.batch, cfg.n_kv_heads
    assert t[cnt.comb(3)] == B * nkv   # one completion per (sequence, KV group)
    assert len(t) == L * nkv + 4 * L + 2
    assert t[cnt.lm()] == -(-cfg.vocab // info["rows"]["lm"])
    assert t[cnt.final()] == B


def test_random_small_configs_bit_exact_valid_and_deadlock_free():
    """Seeded random small shapes and SM counts: the C++ schedule equals the restatement, passes
    the validator, and the host simulator runs it without a deadlock or an early read."""
    rng = np.random.default_rng(2024)
    checked = 0
    for _ in range(60):
        nkv = int(rng.choice([1, 2, 4]))
        hpg = int(rng.choice([1, 2, 4]))
        d = int(rng.choice([64, 128]))
        cfg = small_config(n_layers=int(rng.integers(1, 4)), hidden=int(rng.choice([128, 256, 512])),
                           n_q_heads=nkv * hpg, n_kv_heads=nkv, head_dim=d,
                           ffn=8 * int(rng.integers(16, 120) if rng.random() < 0.7 else rng.integers(257, 800)),
                           vocab=8 * int(rng.integers(64, 600)),
                           batch=int(rng.choice([1, 1, 2, 3])), max_seq=int(rng.integers(8, 400)))
        S = int(rng.choice([1, 3, 7, 16, 37]))
        try:
            s = mk.Schedule(cfg, S)
        except mk.MkError:
            continue
        q, t, _ = sr.build_schedule(cfg, S)
        assert np.array_equal(s.queues(), q), cfg
        assert np.array_equal(s.totals(), t), cfg
        assert sr.validate(q, t, cfg) == [], cfg
        assert sr.simulate(q, t, cfg, n_epochs=1, seed=checked) == [], cfg
        checked += 1
    assert checked >= 40


def test_queues_run_each_wave_in_tile_id_order_also_when_shuffled():
    cfg = get_workload("llama1b_ctx512").cfg
    for seed in (0, 7):
        q, t, _ = sr.build_schedule(cfg, 5, sr.SchedOpts(shuffle_seed=seed))
        for s in range(q.shape[0]):
            live = [w for w in q[s] if w[0] != sr.END]
            keys = [(int(w[22]), int(w[21])) for w in live]
            assert keys == sorted(keys)


@pytest.mark.parametrize("pos", [0, 63, 64, 300, 639])
def test_combining_tile_waits_inside_its_wave_without_deadlock(pos):
    """Five queues hold many attention chunk tiles each; the tile of the chunk holding pos waits
    for the lower chunks of its group inside the wave -- at every position and under shuffled
    placement the simulator completes two steps."""
    cfg = get_workload("llama1b_ctx512").cfg
    for seed in (0, 3):
        q, t, _ = sr.build_schedule(cfg, 5, sr.SchedOpts(shuffle_seed=seed))
        assert sr.simulate(q, t, cfg, n_epochs=2, seed=seed, pos=[pos]) == []


def test_combining_tile_ahead_of_a_lower_chunk_deadlocks_and_is_rejected():
    """Planted: on one queue a group's chunk-9 tile moved ahead of its chunk-3 tile (same wave).
    The validator flags the order and the simulator, decoding position 639 (chunk 9 combines),
    reports the deadlock."""
    cfg = get_workload("llama1b_ctx512").cfg
    o = sr.SchedOpts(attn_chunk=64)   # ten chunks of 64 positions per group
    q, t, _ = sr.build_schedule(cfg, 1, o)
    live = [i for i in range(q.shape[1]) if q[0, i, 0] == sr.ATTN and q[0, i, 1] == 0 and q[0, i, 3] == 0]
    i3 = next(i for i in live if q[0, i, 4] == 3)
    i9 = next(i for i in live if q[0, i, 4] == 9)
    bad = q.copy()
    bad[0, [i3, i9]] = bad[0, [i9, i3]]
    assert any("same wave" in e for e in sr.validate(bad, t, cfg, o))
    assert any("deadlock" in e for e in sr.simulate(bad, t, cfg, n_epochs=1, pos=[639]))
    assert sr.simulate(q, t, cfg, n_epochs=1, pos=[639]) == []


@pytest.mark.parametrize("seed", [0, 9])
def test_kv_windows_drop_the_chunks_past_each_sequence(seed):
    """Variable-length re-planning: a batch-8 schedule with per-sequence windows keeps exactly the
    attention chunks inside each window (C++ bit-exact with the restatement), stays valid, and the
    host simulator completes steps at the windows' last positions and at smaller ones."""
    cfg = get_workload("llama1b_batch8").cfg
    lens = get_workload("llama1b_batch8").kv_len
    lim = [n + 4 for n in lens]
    o = sr.SchedOpts(kv_limit=tuple(lim), shuffle_seed=seed)
    q, t, info = sr.build_schedule(cfg, 37, o)
    s = mk.Schedule(cfg, 37, kv_limit=lim, shuffle_seed=seed)
    assert np.array_equal(s.queues(), q) and np.array_equal(s.totals(), t)
    assert sr.validate(q, t, cfg, o) == []
    C = s.attn_chunk
    for b in range(cfg.batch):
        chunks = sorted({int(w[4]) for w in q.reshape(-1, q.shape[-1]) if w[0] == sr.ATTN and w[2] == b and w[1] == 0 and w[3] == 0})
        assert chunks == list(range(-(-lim[b] // C)))
    assert sr.simulate(q, t, cfg, n_epochs=2, seed=seed) == []
    assert sr.simulate(q, t, cfg, n_epochs=1, seed=seed, pos=[n // 2 for n in lens]) == []
    full, _, _ = sr.build_schedule(cfg, 37, sr.SchedOpts(shuffle_seed=seed))
    assert (q[..., 0] == sr.ATTN).sum() < (full[..., 0] == sr.ATTN).sum()


def test_kv_limit_out_of_range_is_rejected():
    cfg = get_workload("tiny").cfg
    with pytest.raises(mk.MkError) as e:
        mk.Schedule(cfg, 4, kv_limit=[cfg.max_seq + 1])
    assert e.value.status == mk.MK_ERR_ARG
