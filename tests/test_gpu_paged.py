"""Paged KV cache (mk_bind_paged): the cache is a pool of blocks per (layer, KV head) reached
through a block table, one block per split-K attention chunk.

- Decoding with the blocks scattered over the pool (a seeded permutation, plus unused blocks)
  gives logits and tokens bit-identical to the contiguous cache, and the rows each step appends
  land in the right blocks (the pool gathered back equals the contiguous cache).
- A table entry outside the pool stops the step with MK_ERR_BOUNDS before anything is accessed
  there.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import persistent_megakernel_decode_sm_gb300 as mk  # noqa: E402
from gpu_helpers import make_setup  # noqa: E402
from workload import KVCache  # noqa: E402

def to_paged(kv: KVCache, block: int, spare: int, seed: int):
    """The contiguous cache [B, L, nkv, max_seq, d] scattered into a pool of blocks of block
    positions (the schedule's attention chunk)."""
    B, L, nkv, max_seq, d = kv.k.shape
    mb = -(-max_seq // block)
    n_blocks = B * mb + spare
    order = np.random.default_rng(seed).permutation(n_blocks)[:B * mb].reshape(B, mb)
    pool = [torch.zeros((L, nkv, n_blocks * block, d), dtype=kv.k.dtype, device=kv.k.device) for _ in range(2)]
    for b in range(B):
        for j in range(mb):
            lo, hi = j * block, min(max_seq, (j + 1) * block)
            blk = int(order[b, j])
            for src, dst in ((kv.k, pool[0]), (kv.v, pool[1])):
                dst[:, :, blk * block:blk * block + hi - lo] = src[b, :, :, lo:hi]
    table = torch.from_numpy(order.astype(np.int32)).to(kv.k.device)
    return KVCache(pool[0], pool[1]), table, n_blocks


def from_paged(pool: KVCache, table: torch.Tensor, shape, block: int):
    B, L, nkv, max_seq, d = shape
    out = [torch.zeros(shape, dtype=pool.k.dtype, device=pool.k.device) for _ in range(2)]
    tab = table.cpu().numpy()
    for b in range(B):
        for j in range(tab.shape[1]):
            lo, hi = j * block, min(max_seq, (j + 1) * block)
            blk = int(tab[b, j])
            for src, dst in ((pool.k, out[0]), (pool.v, out[1])):
                dst[b, :, :, lo:hi] = src[:, :, blk * block:blk * block + hi - lo]
    return KVCache(out[0], out[1])


@pytest.mark.parametrize("name,steps", [("tiny", 6), ("llama1b_batch8", 2)])
def test_paged_cache_matches_contiguous(name, steps):
    s = make_setup(name)
    S = mk.device_sm_count()
    blk = mk.Schedule(s.cfg, S).attn_chunk
    pool, table, n_blocks = to_paged(s.kv, blk, spare=5, seed=7)
    a = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, s.kv)
    b = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, pool, pages=(table, blk, n_blocks))
    tokens, pos = list(s.tokens), list(s.pos)
    for _ in range(steps):
        ta = a.step(tokens, pos)
        tb = b.step(tokens, pos)
        assert ta == tb
        assert torch.equal(a.logits, b.logits)
        tokens, pos = ta, [p + 1 for p in pos]
    back = from_paged(pool, table, tuple(s.kv.k.shape), blk)
    assert torch.equal(back.k, s.kv.k) and torch.equal(back.v, s.kv.v)
    a.close()
    b.close()


def test_paged_entry_outside_the_pool_is_reported():
    s = make_setup("tiny")
    sched = mk.Schedule(s.cfg, mk.device_sm_count())
    pool, table, n_blocks = to_paged(s.kv, sched.attn_chunk, spare=0, seed=3)
    table[0, 0] = n_blocks   # the first chunk's block lies past the pool
    dec = mk.Decoder(sched, s.weights, pool, pages=(table, sched.attn_chunk, n_blocks))
    with pytest.raises(mk.MkError) as e:
        dec.step(s.tokens, s.pos)
    assert e.value.status == mk.MK_ERR_BOUNDS
    with pytest.raises(mk.MkError) as e:
        dec.step(s.tokens, s.pos)
    assert e.value.status == mk.MK_ERR_POISONED
    dec.close()


def test_paged_bind_rejects_a_block_size_other_than_the_chunk():
    s = make_setup("tiny")
    sched = mk.Schedule(s.cfg, mk.device_sm_count())
    pool, table, n_blocks = to_paged(s.kv, sched.attn_chunk, spare=0, seed=1)
    with pytest.raises(mk.MkError) as e:
        mk.Decoder(sched, s.weights, pool, pages=(table, sched.attn_chunk // 2, n_blocks))
    assert e.value.status == mk.MK_ERR_ARG


def test_paged_chained_counters_mode_matches_contiguous_tags_mode():
    """The paged cache, chained steps and the counters synchronisation together give the same
    tokens and logits as the contiguous cache stepped one call at a time in the default mode."""
    s = make_setup("tiny")
    S = mk.device_sm_count()
    blk = mk.Schedule(s.cfg, S).attn_chunk
    pool, table, n_blocks = to_paged(s.kv, blk, spare=3, seed=11)
    a = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, s.kv)
    b = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, pool, pages=(table, blk, n_blocks))
    b.set_sync("counters")
    n = 5
    toks_b = b.steps(s.tokens, s.pos, n)
    t, toks_a = list(s.tokens), []
    for i in range(n):
        t = a.step(t, [p + i for p in s.pos])
        toks_a.append(t)
    assert toks_a == toks_b
    assert torch.equal(a.logits, b.logits)
    back = from_paged(pool, table, tuple(s.kv.k.shape), blk)
    assert torch.equal(back.k, s.kv.k) and torch.equal(back.v, s.kv.v)
    a.close()
    b.close()
