"""Prefix-caching block manager (host code in libwllm.so), on CPU.

The key check is content, independent of how blocks are chosen: a simulated
pool records which token every slot holds; prompts write their non-cached
tokens, appends write theirs, copy-on-write copies slots; after every
operation each live sequence must read back exactly its own tokens through its
block table.  Reference counts, the free count and the cache count are checked
against the tables, and a few scenarios pin sharing, copy-on-write, eviction
order and failure atomicity."""
import random

import numpy as np
import pytest
import torch

from paged_kv_cache_185_gb300 import binding


@pytest.fixture(scope="module")
def lib():
    try:
        return binding.load_library()
    except RuntimeError as e:
        pytest.skip(str(e))


class Sim:
    """Slot contents and the expected tokens of every live sequence."""

    def __init__(self, bm, num_blocks, bs, max_blocks):
        self.bm, self.bs, self.max_blocks = bm, bs, max_blocks
        self.pool = np.full(num_blocks * bs, -1, np.int64)
        self.seqs = {}

    def add(self, sid, toks):
        slots, cached = self.bm.add_sequence(sid, toks)
        slots = slots.numpy()
        assert cached % self.bs == 0 and 0 <= cached <= len(toks)
        # the cached part must already hold these very tokens
        assert (self.pool[slots[:cached]] == np.asarray(toks[:cached])).all()
        self.pool[slots[cached:]] = toks[cached:]
        self.seqs[sid] = list(toks)
        return slots, cached

    def append(self, sid, tok):
        slot, copy = self.bm.append_token(sid, tok)
        n = len(self.seqs[sid])
        if copy is not None:
            src, dst = copy
            k = n % self.bs
            assert k > 0, "a copy is only needed for a partly filled block"
            self.pool[dst * self.bs:dst * self.bs + k] = self.pool[src * self.bs:src * self.bs + k]
        self.pool[slot] = tok
        self.seqs[sid].append(tok)
        return slot, copy

    def fork(self, parent, child):
        self.bm.fork(parent, child)
        self.seqs[child] = list(self.seqs[parent])

    def free(self, sid):
        self.bm.free_sequence(sid)
        del self.seqs[sid]

    def check(self):
        refs = np.zeros(self.bm.num_blocks, np.int64)
        for sid, toks in self.seqs.items():
            row, n = self.bm.block_table(sid, self.max_blocks)
            row = row.numpy()
            nb = (n + self.bs - 1) // self.bs
            assert n == len(toks)
            assert (row[:nb] >= 0).all() and (row[nb:] == -1).all()
            for b in row[:nb]:
                refs[b] += 1
            t = np.arange(n)
            got = self.pool[row[t // self.bs].astype(np.int64) * self.bs + t % self.bs]
            assert (got == np.asarray(toks)).all(), f"sequence {sid} reads other tokens"
        for b in range(self.bm.num_blocks):
            assert self.bm.block_ref(b) == refs[b], f"block {b}: ref {self.bm.block_ref(b)} vs {refs[b]}"
        assert self.bm.num_free_blocks() == int((refs == 0).sum())
        assert 0 <= self.bm.num_cached_blocks() <= self.bm.num_blocks


def test_shared_prefix_blocks_are_reused(lib):
    bm = binding.BlockManager(64, 16)
    sim = Sim(bm, 64, 16, 16)
    prefix = list(range(1000, 1040))  # 2.5 blocks
    s0, c0 = sim.add(0, prefix + [1, 2, 3])
    s1, c1 = sim.add(1, prefix + [7, 8])
    assert c0 == 0 and c1 == 32  # two full shared blocks
    assert (s1[:32] == s0[:32]).all() and s1[32] // 16 != s0[32] // 16
    sim.check()
    assert bm.block_ref(int(s0[0]) // 16) == 2


def test_fork_then_append_copies_on_write(lib):
    bm = binding.BlockManager(32, 16)
    sim = Sim(bm, 32, 16, 8)
    sim.add(0, list(range(20)))  # one full block + 4 tokens
    sim.fork(0, 1)
    _, copy = sim.append(1, 99)
    assert copy is not None and copy[0] != copy[1]
    _, copy0 = sim.append(0, 98)  # the parent now owns its block alone
    assert copy0 is None
    sim.check()


def test_filled_block_is_cached_for_later_prompts(lib):
    bm = binding.BlockManager(32, 8)
    sim = Sim(bm, 32, 8, 8)
    sim.add(0, [5, 6, 7])
    for t in [8, 9, 10, 11, 12]:
        sim.append(0, t)  # fills block 0 with 5..12
    _, cached = sim.add(1, [5, 6, 7, 8, 9, 10, 11, 12, 40])
    assert cached == 8
    sim.check()


def test_freed_blocks_stay_cached_and_evict_oldest_first(lib):
    bm = binding.BlockManager(4, 4)
    sim = Sim(bm, 4, 4, 4)
    sim.add(0, list(range(8)))      # 2 full cached blocks
    sim.free(0)
    assert bm.num_free_blocks() == 4 and bm.num_cached_blocks() == 2
    _, cached = sim.add(1, list(range(8)) + [50])  # both blocks hit again
    assert cached == 8
    sim.free(1)
    sim.add(2, [60, 61, 62, 63, 64, 65, 66, 67, 68, 69, 70, 71, 72])  # needs all 4 blocks: evicts both
    assert bm.num_cached_blocks() == 3  # its own three full blocks
    sim.check()


def test_out_of_blocks_leaves_state_unchanged(lib):
    bm = binding.BlockManager(3, 4)
    sim = Sim(bm, 3, 4, 4)
    sim.add(0, list(range(12)))  # all 3 blocks, each full
    free, cached = bm.num_free_blocks(), bm.num_cached_blocks()
    for call in (lambda: bm.add_sequence(1, [100, 101, 102, 103, 104]),  # needs 2 blocks
                 lambda: bm.append_token(0, 7)):                          # needs a 4th block
        with pytest.raises(binding.WllmError) as e:
            call()
        assert e.value.status == binding.WLLM_ERR_OUT_OF_RANGE
    assert bm.num_free_blocks() == free and bm.num_cached_blocks() == cached
    sim.check()


def test_bad_ids_raise(lib):
    bm = binding.BlockManager(8, 4)
    bm.add_sequence(1, [1, 2])
    for call in (lambda: bm.add_sequence(1, [3]), lambda: bm.append_token(9, 1), lambda: bm.fork(9, 10),
                 lambda: bm.fork(1, 1), lambda: bm.free_sequence(9), lambda: bm.block_table(9, 4),
                 lambda: bm.block_table(1, 0)):
        with pytest.raises(binding.WllmError):
            call()


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_keep_every_sequence_consistent(lib, seed):
    rng = random.Random(seed)
    bs = rng.choice([4, 8, 16])
    nb = rng.choice([24, 48, 96])
    bm = binding.BlockManager(nb, bs)
    sim = Sim(bm, nb, bs, nb)
    prompts = [[rng.randrange(6) for _ in range(rng.randrange(1, 5 * bs))] for _ in range(4)]
    next_id = 0
    for _ in range(400):
        op = rng.random()
        live = list(sim.seqs)
        try:
            if op < 0.3 or not live:
                base = rng.choice(prompts)
                toks = base[:rng.randrange(0, len(base) + 1)] + [rng.randrange(6) for _ in range(rng.randrange(0, 2 * bs))]
                if not toks:
                    toks = [1]
                sim.add(next_id, toks)
                next_id += 1
            elif op < 0.7:
                sim.append(rng.choice(live), rng.randrange(6))
            elif op < 0.8:
                sim.fork(rng.choice(live), next_id)
                next_id += 1
            else:
                sim.free(rng.choice(live))
        except binding.WllmError as e:
            assert e.status == binding.WLLM_ERR_OUT_OF_RANGE  # pool full: nothing changed
            if live:
                sim.free(rng.choice(live))
        sim.check()
    for sid in list(sim.seqs):
        sim.free(sid)
    assert bm.num_free_blocks() == nb
