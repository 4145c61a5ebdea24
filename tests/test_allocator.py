"""The host block allocator (pkv_allocator_*), on the CPU: the pages' walk,
the accounting invariants after every operation, and operation-by-operation
agreement with the plain-Python model in oracle/block_allocator.py."""
import random

import pytest

from conftest import load_golden
from oracle.block_allocator import AllocatorError, ModelAllocator, OutOfBlocks


def test_walk_decode_slots_match_the_trace(pkv):
    """A (6 tokens in [7, 2]) and B (3 tokens in [5]) on a pool of 8 blocks of 4:
    the two decode steps append at the slots of the golden trace, B's second
    step taking the lowest free block (0)."""
    g = load_golden("walk_trace.json")["derived_by_the_page_rules"]["steps"]
    a = pkv.pkv_allocator_create(8, 4)
    pkv.pkv_allocator_add_sequence(a, 0, 6, [7, 2])
    pkv.pkv_allocator_add_sequence(a, 1, 3, [5])
    for step in g[1:]:
        got = pkv.pkv_allocator_append(a, 0) + pkv.pkv_allocator_append(a, 1)
        assert got == step["slots"]
        assert pkv.pkv_allocator_check(a) == 0
    assert pkv.pkv_allocator_block_table(a, 1, 3) == ([5, 0, -1], 5, 2)
    assert pkv.pkv_allocator_stats(a) == {"free": 4, "allocated": 4, "referenced": 4, "sequences": 2}


def test_new_block_exactly_when_len_mod_bs_is_one(pkv):
    bs = 16
    a = pkv.pkv_allocator_create(64, bs)
    pkv.pkv_allocator_add_sequence(a, 7, 0)
    for n in range(1, 100):
        before = pkv.pkv_allocator_stats(a)["allocated"]
        slot = pkv.pkv_allocator_append(a, 7)[0]
        after = pkv.pkv_allocator_stats(a)["allocated"]
        assert (after - before == 1) == (n % bs == 1)
        row, length, used = pkv.pkv_allocator_block_table(a, 7, 8)
        assert length == n and used == -(-n // bs)
        assert slot == row[(n - 1) // bs] * bs + (n - 1) % bs


def test_sharing_lifecycle(pkv):
    """A forked prefix counts once; it goes back to the pool only when the last
    sequence that references it is released."""
    a = pkv.pkv_allocator_create(10, 4)
    pkv.pkv_allocator_add_sequence(a, 0, 10)  # blocks 0, 1, 2
    pkv.pkv_allocator_fork(a, 0, 1, 8)        # shares 0, 1
    assert pkv.pkv_allocator_stats(a) == {"free": 7, "allocated": 3, "referenced": 3, "sequences": 2}
    assert pkv.pkv_allocator_append(a, 1, 2) == [12, 13]  # the child's own block 3
    pkv.pkv_allocator_release(a, 0)
    assert pkv.pkv_allocator_stats(a)["free"] == 10 - 3  # 0, 1 (child) and 3 stay; 2 is back
    assert pkv.pkv_allocator_check(a) == 0
    pkv.pkv_allocator_release(a, 1)
    assert pkv.pkv_allocator_stats(a) == {"free": 10, "allocated": 0, "referenced": 0, "sequences": 0}


def test_errors_change_nothing(pkv):
    a = pkv.pkv_allocator_create(4, 4)
    pkv.pkv_allocator_add_sequence(a, 0, 9)  # 3 blocks
    snapshot = (pkv.pkv_allocator_stats(a), pkv.pkv_allocator_block_table(a, 0, 4))
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_allocator_append(a, 0, 8)    # needs 2 more blocks, 1 free
    assert e.value.status == pkv.PKV_ERR_OUT_OF_RANGE
    for bad in (lambda: pkv.pkv_allocator_fork(a, 0, 1, 6),         # not whole blocks
                lambda: pkv.pkv_allocator_fork(a, 5, 1, 4),         # no such parent
                lambda: pkv.pkv_allocator_add_sequence(a, 0, 1),    # duplicate id
                lambda: pkv.pkv_allocator_add_sequence(a, 2, 4, [1]),  # block 1 is taken
                lambda: pkv.pkv_allocator_release(a, 9)):
        with pytest.raises(pkv.PkvError) as e:
            bad()
        assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    assert (pkv.pkv_allocator_stats(a), pkv.pkv_allocator_block_table(a, 0, 4)) == snapshot
    with pytest.raises(pkv.PkvError):
        pkv.pkv_allocator_block_table(a, 0, 2)  # row too short
    assert pkv.pkv_allocator_check(a) == 0


@pytest.mark.parametrize("seed", range(6))
def test_random_lifecycle_matches_the_model(pkv, seed):
    """Admit, grow, fork, release at random; after every operation the library
    and the model agree on the outcome, every block table, the slots and the
    counts, and both report the invariants intact."""
    rng = random.Random(seed)
    nb, bs = rng.choice([(40, 4), (64, 16), (300, 16)])
    a, m = pkv.pkv_allocator_create(nb, bs), ModelAllocator(nb, bs)
    live, next_id = [], 0
    for _ in range(400):
        op = rng.random()
        try:
            if op < 0.25 or not live:
                n = rng.randint(0, 5 * bs)
                exp = ("ok", m.add_sequence(next_id, n))
                got = ("ok", pkv.pkv_allocator_add_sequence(a, next_id, n))
                live.append(next_id)
                next_id += 1
            elif op < 0.7:
                s, k = rng.choice(live), rng.randint(1, 3)
                exp = ("ok", m.append(s, k))
                got = ("ok", pkv.pkv_allocator_append(a, s, k))
            elif op < 0.82:
                s = rng.choice(live)
                k = bs * rng.randint(0, m.seqs[s]["len"] // bs)
                exp = ("ok", m.fork(s, next_id, k))
                got = ("ok", pkv.pkv_allocator_fork(a, s, next_id, k))
                live.append(next_id)
                next_id += 1
            else:
                s = live.pop(rng.randrange(len(live)))
                exp = ("ok", m.release(s))
                got = ("ok", pkv.pkv_allocator_release(a, s))
        except OutOfBlocks:
            exp = ("full", None)
            with pytest.raises(pkv.PkvError) as e:
                if op < 0.25 or len(live) == 0:
                    pkv.pkv_allocator_add_sequence(a, next_id, n)
                else:
                    pkv.pkv_allocator_append(a, s, k)
            assert e.value.status == pkv.PKV_ERR_OUT_OF_RANGE
            got = ("full", None)
        assert got == exp
        assert pkv.pkv_allocator_stats(a) == m.stats()
        assert pkv.pkv_allocator_check(a) == 0 == m.check()
        for s in live:
            assert pkv.pkv_allocator_block_table(a, s, 16) == m.block_table(s, 16)


def test_model_check_catches_a_planted_leak(orc):
    """The invariants are not vacuous: a model that forgets to drop a
    reference on release breaks rule 2 (and leaks a block)."""
    m = ModelAllocator(8, 4)
    m.add_sequence(0, 5)
    m.fork(0, 1, 4)
    m.seqs.pop(1)  # released without dropping its reference
    assert m.check() == 2
    m2 = ModelAllocator(8, 4)
    m2.add_sequence(0, 5)
    m2.ref[7] = 1  # a block marked used that no table references
    assert m2.check() == 2
    with pytest.raises(AllocatorError):
        m2.fork(0, 1, 3)
