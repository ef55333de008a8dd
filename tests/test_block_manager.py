"""The host block manager (pa_bm_* calls) without a GPU.

Pins the nano-vLLM learning note's BlockManager behaviour (Block, compute_hash,
can_allocate, allocate, deallocate, can_append, may_append and hash_blocks
listings): oldest-first reuse of free blocks, prefix sharing of full blocks
with reference counts, the last prompt block never taken from the cache,
released blocks that keep their hash until handed out again, and growth by
one block when a sequence's length becomes 1 mod block_size.  A randomized
run checks the invariants after every operation.
"""
import numpy as np
import pytest

import paged_kv_gqa_08_gb300 as pa
from paged_kv_gqa_08_gb300 import build
from paged_kv_gqa_08_gb300.block_manager import BlockManager

P = 4


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return pa.load_library()


def toks(*blocks, tail=()):
    """Token ids: each block given by one int (P copies of it) plus a partial tail."""
    out = []
    for b in blocks:
        out += [b * 100 + i for i in range(P)]
    return out + list(tail)


def table(bm, sid, maxp=16):
    bt, lens = bm.block_tables([sid], maxp, pad_page=-7)
    n = bm.seq_info(sid)[2]
    assert (bt[0, n:] == -7).all()
    return list(bt[0, :n]), int(lens[0])


def test_fresh_allocation_takes_oldest_blocks_and_free_returns_them_last_block_first():
    bm = BlockManager(10, P)
    assert bm.allocate(1, toks(1, 2, tail=[5])) == 0
    t1, n1 = table(bm, 1)
    assert t1 == [0, 1, 2] and n1 == 2 * P + 1
    assert bm.num_free_blocks() == 7
    assert all(bm.ref_count(b) == 1 for b in t1)
    bm.free(1)
    assert bm.num_free_blocks() == 10
    assert all(bm.ref_count(b) == 0 for b in t1)
    # the never-used blocks 3..9 are older in the free list than the released ones
    bm.allocate(2, toks(7, 8, 9))
    assert table(bm, 2)[0] == [3, 4, 5]


def test_prefix_sharing_counts_references_and_reports_cached_tokens():
    bm = BlockManager(16, P)
    a = toks(1, 2, 3, tail=[9, 9])
    bm.allocate(1, a)
    bm.hash_blocks(1, len(a))            # three full blocks computed and registered
    assert bm.counts()[2] == 3
    b = toks(1, 2, 4, tail=[8])
    assert bm.can_allocate(b) == 2
    assert bm.allocate(2, b) == 2 * P
    ta, tb = table(bm, 1)[0], table(bm, 2)[0]
    assert tb[:2] == ta[:2] and tb[2] not in ta
    assert [bm.ref_count(x) for x in ta] == [2, 2, 1, 1]
    assert bm.seq_info(2) == (len(b), 2 * P, 4)
    bm.free(1)
    assert [bm.ref_count(x) for x in ta[:2]] == [1, 1] and bm.ref_count(ta[2]) == 0


def test_the_last_prompt_block_is_never_taken_from_the_cache():
    bm = BlockManager(16, P)
    a = toks(1, 2, 3)
    bm.allocate(1, a)
    bm.hash_blocks(1, len(a))
    assert bm.allocate(2, toks(1, 2, 3)) == 2 * P    # block 3 is full and cached, but it is the last one
    assert bm.allocate(3, toks(1, 2, 3, tail=[1])) == 3 * P


def test_equal_tokens_after_a_different_prefix_are_not_shared():
    bm = BlockManager(16, P)
    a = toks(1, 2, tail=[0])
    bm.allocate(1, a)
    bm.hash_blocks(1, len(a))
    assert bm.allocate(2, toks(5, 2, tail=[0])) == 0   # block "2" follows another prefix: a different chain hash


def test_released_blocks_keep_their_hash_until_reused():
    bm = BlockManager(8, P)
    a = toks(1, 2, 3, tail=[0])
    bm.allocate(1, a)
    bm.hash_blocks(1, len(a))
    ta = table(bm, 1)[0]
    bm.free(1)
    assert bm.num_free_blocks() == 8
    # a later prompt with the same prefix gets the released blocks back from the free list
    assert bm.allocate(2, toks(1, 2, 3, tail=[4])) == 3 * P
    assert table(bm, 2)[0][:3] == ta[:3]
    assert bm.num_free_blocks() == 8 - 4
    bm.free(2)
    # exhaust the free list: the released blocks are handed out fresh and lose their hash
    bm.allocate(3, toks(*range(10, 18)))
    bm.free(3)
    assert bm.can_allocate(toks(1, 2, 3, tail=[4])) == 0


def test_capacity_errors_change_nothing():
    bm = BlockManager(4, P)
    bm.allocate(1, toks(1, 2, 3))
    assert bm.can_allocate(toks(5, 6)) == -1
    with pytest.raises(pa.PagedAttnError) as e:
        bm.allocate(2, toks(5, 6))
    assert e.value.status == pa.PA_ERR_CAPACITY
    assert bm.counts()[:2] == (1, 1)
    bm.append_token(1, 42)                 # length 13 = 1 mod 4: takes the last free block
    assert bm.num_free_blocks() == 0 and bm.seq_info(1)[2] == 4
    for t in range(3):
        bm.append_token(1, t)              # fills the block: no new block needed
    with pytest.raises(pa.PagedAttnError) as e:
        bm.append_token(1, 7)              # length 17 would need a fifth block
    assert e.value.status == pa.PA_ERR_CAPACITY
    assert bm.seq_info(1) == (16, 0, 4)


def test_argument_errors():
    bm = BlockManager(4, P)
    bm.allocate(1, [1, 2])
    with pytest.raises(pa.PagedAttnError):
        bm.allocate(1, [3])                # id already registered
    with pytest.raises(pa.PagedAttnError):
        bm.free(99)
    with pytest.raises(pa.PagedAttnError):
        bm.allocate(2, [])
    with pytest.raises(pa.PagedAttnError):
        bm.block_tables([1], 0)
    with pytest.raises(pa.PagedAttnError):
        bm.hash_blocks(1, 3)               # more than the sequence holds


def test_slot_mapping_follows_the_block_tables():
    bm = BlockManager(32, P)
    bm.allocate(1, list(range(9)))
    bm.allocate(2, list(range(50, 53)))
    for t in range(4):
        bm.append_token(2, 90 + t)
    bt, lens = bm.block_tables([1, 2], 8)
    slots = bm.slot_mapping([1, 2], [3, 5])
    want = []
    for i, n_new in enumerate([3, 5]):
        for pos in range(lens[i] - n_new, lens[i]):
            want.append(bt[i, pos // P] * P + pos % P)
    assert slots.tolist() == want


def _check_invariants(bm, live, nblocks):
    """live: seq id -> token list."""
    refs = np.zeros(nblocks, dtype=np.int64)
    tables = {}
    for sid, tk in live.items():
        t, n = table(bm, sid, maxp=64)
        assert n == len(tk) and len(t) == -(-len(tk) // P)
        assert len(set(t)) == len(t)
        tables[sid] = t
        for b in t:
            refs[b] += 1
    assert [bm.ref_count(b) for b in range(nblocks)] == refs.tolist()
    assert bm.num_free_blocks() == int((refs == 0).sum())
    # a block held by two sequences sits at the same index of both tables, and
    # both sequences hold identical tokens up to the end of that block
    owner = {}
    for sid, t in tables.items():
        for i, b in enumerate(t):
            if b in owner:
                s2, i2 = owner[b]
                assert i == i2
                assert live[sid][:(i + 1) * P] == live[s2][:(i + 1) * P]
            else:
                owner[b] = (sid, i)


def test_randomized_operations_keep_the_invariants():
    rng = np.random.default_rng(0)
    nblocks = 20                # small enough that allocations and appends also run out of blocks
    bm = BlockManager(nblocks, P)
    live = {}
    prefixes = [list(rng.integers(0, 5, size=3 * P)) for _ in range(3)]
    next_id = 0
    stats = {"hits": 0, "capacity": 0}
    for step in range(600):
        op = rng.integers(0, 6)         # allocate, append and free at 2 : 3 : 1
        if op < 2 or not live:
            pre = prefixes[rng.integers(0, 3)][: int(rng.integers(0, 3 * P + 1))]
            tk = [int(x) for x in pre] + [int(x) for x in rng.integers(0, 5, size=int(rng.integers(1, 2 * P)))]
            fits = bm.can_allocate(tk) >= 0
            try:
                cached = bm.allocate(next_id, tk)
                assert fits and cached % P == 0 and cached < len(tk)
                stats["hits"] += cached > 0
                live[next_id] = tk
                bm.hash_blocks(next_id, len(tk))
            except pa.PagedAttnError as e:
                assert not fits and e.status == pa.PA_ERR_CAPACITY
                stats["capacity"] += 1
            next_id += 1
        elif op < 5:
            sid = list(live)[rng.integers(0, len(live))]
            tok = int(rng.integers(0, 5))
            try:
                bm.append_token(sid, tok)
                live[sid].append(tok)
                bm.hash_blocks(sid, len(live[sid]))
            except pa.PagedAttnError as e:
                assert e.status == pa.PA_ERR_CAPACITY and len(live[sid]) % P == 0
                stats["capacity"] += 1
        else:
            sid = list(live)[rng.integers(0, len(live))]
            bm.free(sid)
            del live[sid]
        _check_invariants(bm, live, nblocks)
    assert next_id > 100 and stats["hits"] > 20 and stats["capacity"] > 5
