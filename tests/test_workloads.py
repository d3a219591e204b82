"""Structure of the seeded synthetic workloads (CPU only)."""
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_185_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_paged_decode.txt")


def _check_tables(case):
    bt, cl, bs = case.block_tables, case.context_lens, case.block_size
    for i in range(case.num_seqs):
        n = (int(cl[i]) + bs - 1) // bs
        row = bt[i]
        assert (row[:n] >= 0).all() and (row[:n] < case.num_blocks).all()
        assert (row[n:] == -1).all()


def test_tiny_workload_shape():
    c = workloads.make_case("c0")
    assert c.context_lens.tolist() == [7, 16, 33, 50]
    assert (c.num_q_heads, c.num_kv_heads, c.head_dim, c.block_size, c.num_blocks) == (4, 2, 64, 16, 32)
    assert c.dtype == torch.float32
    assert c.used_blocks.numel() == 1 + 1 + 3 + 4
    assert len(set(c.used_blocks.tolist())) == 9
    _check_tables(c)
    # append at position L-1 of each sequence
    bs = c.block_size
    for i, L in enumerate(c.context_lens.tolist()):
        pos = L - 1
        assert int(c.slot_mapping[i]) == int(c.block_tables[i, pos // bs]) * bs + pos % bs


def test_workload_is_deterministic():
    a, b = workloads.make_case("c0"), workloads.make_case("c0")
    for name in ("q", "k_used", "v_used", "key", "value", "block_tables", "slot_mapping"):
        x, y = getattr(a, name), getattr(b, name)
        assert torch.equal(x.view(torch.uint8) if x.is_floating_point() else x,
                           y.view(torch.uint8) if y.is_floating_point() else y)


def test_tinyllama_workload():
    c = workloads.make_case("c1")
    assert c.num_seqs == 64 and c.group == 8 and c.head_dim == 64 and c.dtype == torch.float16
    L = c.context_lens
    assert int(L.min()) >= 128 and int(L.max()) <= 2048
    # pool sized to fit: every block is used exactly once
    assert c.num_blocks == c.used_blocks.numel()
    assert sorted(c.used_blocks.tolist()) == list(range(c.num_blocks))
    _check_tables(c)


def test_shared_prefix_workload_shares_blocks():
    c = workloads.custom_case("prefix", lens=[70, 90, 65, 100, 80, 66], num_q_heads=4,
                              num_kv_heads=2, head_dim=16, block_size=16, groups=(3, 4), seed=5)
    bt = c.block_tables
    assert torch.equal(bt[0, :4], bt[1, :4]) and torch.equal(bt[0, :4], bt[2, :4])
    assert torch.equal(bt[3, :4], bt[5, :4])
    assert not set(bt[0, :4].tolist()) & set(bt[3, :4].tolist())
    private = [int(x) for i in range(6) for x in bt[i, 4:] if x >= 0]
    assert len(private) == len(set(private))
    # unique tokens count shared blocks once
    assert c.meta["unique_tokens"] == 2 * 64 + sum(L - 64 for L in [70, 90, 65, 100, 80, 66])


def test_free_slot_append_never_hits_read_slots():
    c = workloads.custom_case("free", lens=[5, 16, 20], num_q_heads=2, num_kv_heads=2,
                              head_dim=8, block_size=8, spare_blocks=2, append="free",
                              n_append=10, seed=3)
    bs = c.block_size
    read = set()
    for i, L in enumerate(c.context_lens.tolist()):
        for j in range(L):
            read.add(int(c.block_tables[i, j // bs]) * bs + j % bs)
    slots = c.slot_mapping.tolist()
    assert len(set(slots)) == len(slots) == 10
    assert not read & set(slots)


def test_unread_slots_are_nan():
    c = workloads.make_case("c0")
    kc, vc = c.pool()
    bs = c.block_size
    read = torch.zeros(c.num_blocks, bs, dtype=torch.bool)
    appended = set(c.slot_mapping.tolist())
    for i, L in enumerate(c.context_lens.tolist()):
        for j in range(L):
            s = int(c.block_tables[i, j // bs]) * bs + j % bs
            if s not in appended:
                read[s // bs, s % bs] = True
    k_nan = torch.isnan(kc).all(dim=-1).all(dim=1)  # [N_b, bs]
    assert torch.equal(k_nan, ~read)
    assert not torch.isnan(kc[read.unsqueeze(1).expand(-1, 2, -1)]).any()


def test_heavy_keys_fraction():
    c = workloads.custom_case("heavy", lens=[4000, 3000], num_q_heads=4, num_kv_heads=2,
                              head_dim=32, block_size=16, heavy_key_frac=0.01, seed=8,
                              dtype=torch.float32, append="none")
    norms = c.k_used.float().norm(dim=-1)
    finite = norms[~torch.isnan(norms)]
    frac = float((finite > 3 * finite.median()).float().mean())
    assert 0.005 < frac < 0.02


def test_normal_is_thread_count_independent():
    a = workloads.normal(7, (1 << 22) * 2 + 17)
    b = workloads.normal(7, (1 << 22) * 2 + 17)
    assert np.array_equal(a, b)
    assert abs(float(a.mean())) < 1e-2 and abs(float(a.std()) - 1) < 1e-2


def test_compact_pool_matches_full_pool():
    c = workloads.custom_case("cmp", lens=[20, 33, 7], num_q_heads=4, num_kv_heads=2,
                              head_dim=16, block_size=8, num_blocks=40, seed=4)
    kc, vc = c.pool()
    oracle.reshape_and_cache(c.key, c.value, kc, vc, c.slot_mapping)
    full = oracle.paged_decode(c.q, kc, vc, c.block_tables, c.context_lens, 2, c.scale)
    k2, v2, bt2, s2 = c.compact()
    oracle.reshape_and_cache(c.key, c.value, k2, v2, s2)
    small = oracle.paged_decode(c.q, k2, v2, bt2, c.context_lens, 2, c.scale)
    assert torch.equal(full, small)


def test_golden_tiny_decode_matches_oracle():
    with open(GOLDEN) as f:
        lines = [ln for ln in f if not ln.startswith("#")]
    ref = torch.tensor([float.fromhex(x) for x in lines], dtype=torch.float64).reshape(4, 4, 64)
    c = workloads.make_case("c0")
    kc, vc = c.pool()
    oracle.reshape_and_cache(c.key, c.value, kc, vc, c.slot_mapping)
    got = oracle.paged_decode(c.q, kc, vc, c.block_tables, c.context_lens, 2, c.scale)
    torch.testing.assert_close(got, ref, rtol=0, atol=1e-14)


@pytest.mark.parametrize("name", ["c2", "c3"])
def test_large_workload_tables(name):
    c = workloads.make_case(name)
    _check_tables(c)
    if name == "c2":
        assert c.slot_mapping.numel() == 128 and c.num_kv_heads == 32
    else:
        L = c.context_lens
        assert int(L.min()) >= 1025 and int(L.max()) <= 32768
        bt = c.block_tables
        for g in range(0, 256, 8):
            assert (bt[g:g + 8, :64] == bt[g, :64]).all()


def test_e4m3_codes_draws_torch_codes_and_keeps_nan():
    from paged_kv_cache_185_gb300.workloads import e4m3_codes
    x = torch.tensor([[1.0, -2.5, float("nan")], [0.001, 100.0, -0.0]])
    got = e4m3_codes(x, 2.0)
    ref = (x.float() * 2.0).to(torch.float8_e4m3fn).view(torch.uint8)
    assert got.dtype == torch.uint8 and got.shape == x.shape
    assert torch.equal(got, ref)
    assert got[0, 2] & 0x7F == 0x7F
    with pytest.raises(ValueError):
        e4m3_codes(torch.tensor([300.0]), 2.0)  # 600 is outside E4M3
