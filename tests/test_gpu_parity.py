"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bars: the KV append is bit-exact over the whole pool (NaN-poisoned slots
included); attention is within max-abs 1e-5 for fp32 inputs and within
max-abs 2e-2 with relative L2 5e-3 for fp16/bf16 inputs.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_185_gb300 as wllm
from paged_kv_cache_185_gb300 import workloads
from tests.gpu_common import assert_attention_close, gpu_step, int_view, oracle_step

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_paged_decode.txt")


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_kv_cache_185_gb300 import build
    build.build()
    wllm.load_library()
    yield
    assert wllm.device_errors() == 0


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

def test_tiny_workload_matches_oracle_and_golden():
    case = workloads.make_case("c0")
    got, kc, vc = gpu_step(case)
    ref, kr, vr = oracle_step(case)
    assert torch.equal(int_view(kc.cpu()), int_view(kr))
    assert torch.equal(int_view(vc.cpu()), int_view(vr))
    assert_attention_close(got, ref, case.dtype, "c0")
    with open(GOLDEN) as f:
        gold = torch.tensor([float.fromhex(x) for x in f if not x.startswith("#")],
                            dtype=torch.float64).reshape(ref.shape)
    assert_attention_close(got, gold, case.dtype, "c0 golden")


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "gemma_mqa", "bs32"])
def test_workload_matches_oracle(name):
    case = workloads.make_case(name)
    got, kc, vc = gpu_step(case)
    ref, kr, vr = oracle_step(case)
    assert torch.equal(int_view(kc.cpu()), int_view(kr)), "K append not bit-exact"
    assert torch.equal(int_view(vc.cpu()), int_view(vr)), "V append not bit-exact"
    del kc, vc
    torch.cuda.empty_cache()
    assert_attention_close(got, ref, case.dtype, name)


def test_long_context_workload_sampled():
    """32K-128K tokens per sequence, ~120 GB pool, 1% keys x8: sampled rows
    against the oracle, the append checked bit for bit on every used block."""
    case = workloads.make_case("c4")
    free = torch.cuda.mem_get_info()[0]
    need = 2 * case.pool_bytes() + (4 << 30)
    assert free > need, f"needs {need / 2**30:.0f} GiB of device memory, {free / 2**30:.0f} free"
    got, kc, vc = gpu_step(case)
    ids = case.used_blocks.cuda()
    k_used, v_used = kc[ids].cpu(), vc[ids].cpu()
    del kc, vc
    torch.cuda.empty_cache()
    g = torch.Generator().manual_seed(4)
    B, Hq = case.num_seqs, case.num_q_heads
    rows = sorted(set(torch.randint(0, B * Hq, (40,), generator=g).tolist()) |
                  {b * Hq + (b * 5) % Hq for b in range(B)})
    ref, kr, vr = oracle_step(case, rows=rows, compact=True)
    assert torch.equal(int_view(k_used), int_view(kr))
    assert torch.equal(int_view(v_used), int_view(vr))
    flat = got.reshape(B * Hq, -1)[rows]
    assert_attention_close(flat, ref, case.dtype, "c4 sampled rows")


def test_long_context_fused_step_sampled():
    """The long-context batch through the fused step (append, grid barrier,
    decode, in-launch merge of up to 128 partitions per sequence) over the full
    ~120 GB pool, as the benchmark times it: sampled rows against the oracle
    (which reads only the referenced blocks), the append bit for bit."""
    case = workloads.make_case("c4")
    free = torch.cuda.mem_get_info()[0]
    need = 2 * case.pool_bytes() + (4 << 30)
    assert free > need, f"needs {need / 2**30:.0f} GiB of device memory, {free / 2**30:.0f} free"
    kc, vc = case.pool("cuda")
    q = case.q.cuda()
    out = torch.full_like(q, float("nan"))
    wllm.decode_step(out, q, case.key.cuda(), case.value.cuda(), kc, vc, case.slot_mapping.cuda(),
                     case.block_tables.cuda(), case.context_lens.cuda(), case.num_kv_heads, case.scale,
                     case.block_size)
    torch.cuda.synchronize()
    ids = case.used_blocks.cuda()
    k_used, v_used = kc[ids].cpu(), vc[ids].cpu()
    del kc, vc
    torch.cuda.empty_cache()
    B, Hq = case.num_seqs, case.num_q_heads
    g = torch.Generator().manual_seed(44)
    rows = sorted(set(torch.randint(0, B * Hq, (40,), generator=g).tolist()) |
                  {b * Hq + (b * 3 + 1) % Hq for b in range(B)})
    ref, kr, vr = oracle_step(case, rows=rows, compact=True)
    assert torch.equal(int_view(k_used), int_view(kr))
    assert torch.equal(int_view(v_used), int_view(vr))
    got = out.cpu()
    assert torch.isfinite(got).all(), "every row written"
    assert_attention_close(got.reshape(B * Hq, -1)[rows], ref, case.dtype, "c4 fused step, sampled rows")


# ---------------------------------------------------------------------------
# shape sweep: dtype x head_dim x block_size x GQA group, ragged lengths
# ---------------------------------------------------------------------------

SHAPES = [
    # (dtype, Hq, Hkv, D, bs)
    (torch.float32, 4, 2, 64, 16), (torch.float32, 8, 1, 128, 8), (torch.float32, 12, 2, 256, 32),
    (torch.float16, 32, 4, 64, 16), (torch.float16, 8, 8, 128, 8), (torch.float16, 28, 4, 128, 32),
    (torch.float16, 8, 1, 256, 16), (torch.float16, 24, 2, 128, 16), (torch.float16, 32, 1, 64, 64),
    (torch.bfloat16, 32, 32, 128, 16), (torch.bfloat16, 28, 4, 128, 16), (torch.bfloat16, 32, 8, 128, 8),
    (torch.bfloat16, 16, 1, 256, 32), (torch.bfloat16, 2, 2, 64, 128), (torch.bfloat16, 48, 4, 64, 16),
    (torch.bfloat16, 40, 2, 256, 16), (torch.bfloat16, 4, 4, 256, 256),
]
LENS = [1, 15, 16, 17, 33, 0, 64, 100, 255, 256, 257, 700, 1031]


@pytest.mark.parametrize("dtype,Hq,Hkv,D,bs", SHAPES)
def test_shape_sweep(dtype, Hq, Hkv, D, bs):
    case = workloads.custom_case("sweep", lens=LENS, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                                 block_size=bs, dtype=dtype, seed=Hq * 7 + D + bs,
                                 spare_blocks=3, max_blocks=(max(LENS) + bs - 1) // bs + 2)
    got, kc, vc = gpu_step(case)
    ref, kr, vr = oracle_step(case)
    assert torch.equal(int_view(kc.cpu()), int_view(kr))
    assert torch.equal(int_view(vc.cpu()), int_view(vr))
    assert_attention_close(got, ref, dtype, f"{dtype} {Hq}/{Hkv} D{D} bs{bs}")
    assert torch.equal(got[LENS.index(0)], torch.zeros_like(got[0]))


@pytest.mark.parametrize("part", [64, 128, 320])
@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_forced_split_kv(monkeypatch, part, dtype):
    """Many partitions per sequence: exercises the cross-CTA combine."""
    monkeypatch.setenv("WLLM_PARTITION_TOKENS", str(part))
    lens = [1, 63, 64, 65, 500, 1000, 2049, 0, 3000]
    case = workloads.custom_case("split", lens=lens, num_q_heads=8, num_kv_heads=2, head_dim=128,
                                 block_size=16, dtype=dtype, seed=part, heavy_key_frac=0.02)
    got, _, _ = gpu_step(case)
    ref, _, _ = oracle_step(case)
    assert_attention_close(got, ref, dtype, f"split {part}")
    # the same with a fresh table layout: counters must have been left at zero
    got2, _, _ = gpu_step(case)
    assert torch.equal(got, got2)


@pytest.mark.parametrize("B,part", [(300, 256), (1024, 512)])
def test_split_schedule_with_tied_lengths(monkeypatch, B, part):
    """Many sequences sharing few distinct lengths (ties in the partition
    count) split over several partitions: every CTA must derive the same unit
    order, so each (sequence, partition, kv head) is computed exactly once."""
    monkeypatch.setenv("WLLM_PARTITION_TOKENS", str(part))
    rng = torch.Generator().manual_seed(B)
    lens = [int(x) for x in torch.tensor([part - 3, 2 * part, 2 * part + 5, 3 * part - 1])[
        torch.randint(0, 4, (B,), generator=rng)]]
    case = workloads.custom_case("ties", lens=lens, num_q_heads=4, num_kv_heads=2, head_dim=64,
                                 block_size=16, dtype=torch.float16, seed=B)
    got, _, _ = gpu_step(case)
    rows = list(range(0, B * 4, 7)) + [B * 4 - 1]
    ref, _, _ = oracle_step(case, rows=rows)
    assert_attention_close(got.reshape(B * 4, -1)[rows], ref, case.dtype, f"ties {B}")


def test_fma_variant_matches_oracle(monkeypatch):
    monkeypatch.setenv("WLLM_FORCE_FMA", "1")
    case = workloads.custom_case("fma", lens=LENS, num_q_heads=28, num_kv_heads=4, head_dim=128,
                                 block_size=16, dtype=torch.bfloat16, seed=77)
    got, _, _ = gpu_step(case)
    ref, _, _ = oracle_step(case)
    assert_attention_close(got, ref, case.dtype, "fma bf16")


# ---------------------------------------------------------------------------
# invariants and closed forms on the GPU
# ---------------------------------------------------------------------------

def test_block_permutation_is_bitwise_invariant():
    case = workloads.custom_case("perm", lens=[5, 300, 77, 1024], num_q_heads=16, num_kv_heads=2,
                                 head_dim=128, block_size=16, dtype=torch.bfloat16, seed=3,
                                 spare_blocks=11, append="none")
    kc, vc = case.pool("cuda")
    q = case.q.cuda()
    out1 = torch.empty_like(q)
    wllm.paged_attention_decode(out1, q, kc, vc, case.block_tables.cuda(), case.context_lens.cuda(),
                                2, case.scale, 16)
    perm = torch.randperm(case.num_blocks, generator=torch.Generator().manual_seed(1))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(case.num_blocks)
    bt2 = torch.where(case.block_tables >= 0, inv[case.block_tables.clamp(min=0).long()].int(),
                      case.block_tables)
    kc2, vc2 = kc[perm.cuda()], vc[perm.cuda()]
    out2 = torch.empty_like(q)
    wllm.paged_attention_decode(out2, q, kc2, vc2, bt2.cuda(), case.context_lens.cuda(), 2,
                                case.scale, 16)
    torch.cuda.synchronize()
    assert torch.equal(int_view(out1), int_view(out2))


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_single_token_returns_value_exactly(dtype):
    case = workloads.custom_case("one", lens=[1] * 8, num_q_heads=8, num_kv_heads=2, head_dim=64,
                                 block_size=16, dtype=dtype, seed=5, append="tail")
    got, _, _ = gpu_step(case)
    expect = case.value.repeat_interleave(4, dim=1)  # every head of the group sees the one token
    assert torch.equal(int_view(got.to(dtype)), int_view(expect))


def test_equal_keys_give_mean_of_values():
    L, D = 300, 128
    case = workloads.custom_case("mean", lens=[L], num_q_heads=4, num_kv_heads=1, head_dim=D,
                                 block_size=16, dtype=torch.float32, seed=6, append="none")
    case.k_used[:] = case.k_used[0, 0, 0]  # every key equal
    got, _, _ = gpu_step(case)
    kc, vc = case.pool("cpu")
    v = torch.cat([vc[int(case.block_tables[0, j])][0] for j in range((L + 15) // 16)])[:L]
    mean = v.double().mean(dim=0)
    for h in range(4):
        assert (got[0, h].double() - mean).abs().max().item() < 1e-5


# ---------------------------------------------------------------------------
# append variants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_append_strided_int32_and_padding(dtype):
    g = torch.Generator().manual_seed(9)
    T, Hkv, D, bs, N_b = 37, 4, 128, 16, 20
    qkv = torch.randn(T, 3 * Hkv + 1, D, generator=g).to(dtype)  # fused-projection-like layout
    key, value = qkv[:, 1:1 + Hkv], qkv[:, 1 + Hkv:1 + 2 * Hkv]
    slots = torch.randperm(N_b * bs, generator=g)[:T]
    slots[[3, 10, 30]] = -1
    kc = torch.full((N_b, Hkv, bs, D), float("nan"), dtype=dtype)
    vc = kc.clone()
    kr, vr = kc.clone(), vc.clone()
    oracle.reshape_and_cache(key.contiguous(), value.contiguous(), kr, vr, slots.long())
    kd, vd = kc.cuda(), vc.cuda()
    wllm.reshape_and_cache(key.cuda(), value.cuda(), kd, vd, slots.int().cuda())
    torch.cuda.synchronize()
    assert torch.equal(int_view(kd.cpu()), int_view(kr))
    assert torch.equal(int_view(vd.cpu()), int_view(vr))


def test_append_unaligned_rows_use_scalar_path():
    g = torch.Generator().manual_seed(10)
    T, Hkv, D = 9, 2, 64
    buf = torch.randn(T * Hkv * D + 1, generator=g).to(torch.float16)
    key = buf[1:].view(T, Hkv, D)  # 2-byte aligned only
    value = torch.randn(T, Hkv, D, generator=g).to(torch.float16)
    slots = torch.arange(T) * 3
    kc = torch.zeros(4, Hkv, 8, D, dtype=torch.float16)
    vc = kc.clone()
    kr, vr = kc.clone(), vc.clone()
    oracle.reshape_and_cache(key.contiguous(), value, kr, vr, slots)
    kd, vd = kc.cuda(), vc.cuda()
    wllm.reshape_and_cache(key.cuda(), value.cuda(), kd, vd, slots.cuda())
    torch.cuda.synchronize()
    assert torch.equal(int_view(kd.cpu()), int_view(kr))
    assert torch.equal(int_view(vd.cpu()), int_view(vr))


# ---------------------------------------------------------------------------
# check mode, workspace, streams, errors
# ---------------------------------------------------------------------------

def test_check_mode_reports_bad_indices(monkeypatch):
    monkeypatch.setenv("WLLM_CHECK", "1")
    case = workloads.custom_case("chk", lens=[40, 17], num_q_heads=4, num_kv_heads=2, head_dim=64,
                                 block_size=16, dtype=torch.float16, seed=2, spare_blocks=2)
    got, _, _ = gpu_step(case)  # valid inputs pass
    kc, vc = case.pool("cuda")
    q = case.q.cuda()
    out = torch.empty_like(q)
    bt = case.block_tables.clone()
    bt[0, 1] = case.num_blocks + 5
    with pytest.raises(wllm.WllmError) as e:
        wllm.paged_attention_decode(out, q, kc, vc, bt.cuda(), case.context_lens.cuda(), 2,
                                    case.scale, 16)
    assert e.value.status == 3
    cl = case.context_lens.clone()
    cl[1] = case.max_blocks * 16 + 1
    with pytest.raises(wllm.WllmError) as e:
        wllm.paged_attention_decode(out, q, kc, vc, case.block_tables.cuda(), cl.cuda(), 2,
                                    case.scale, 16)
    assert e.value.status == 3
    key, value = case.key.cuda(), case.value.cuda()
    for bad in ([0, case.num_blocks * 16], [5, 5]):
        with pytest.raises(wllm.WllmError) as e:
            wllm.reshape_and_cache(key, value, kc, vc, torch.tensor(bad).cuda())
        assert e.value.status == 3
    assert wllm.device_errors() == 0


def test_out_of_range_slot_is_skipped_without_check_mode():
    kc = torch.zeros(2, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    key = torch.ones(2, 1, 64, dtype=torch.bfloat16, device="cuda")
    wllm.reshape_and_cache(key, key, kc, vc, torch.tensor([3, 16], device="cuda"))
    torch.cuda.synchronize()
    assert wllm.device_errors() & 1
    assert kc.sum().item() == 64 and vc.sum().item() == 64


def test_caller_workspace_and_stream(monkeypatch):
    monkeypatch.setenv("WLLM_PARTITION_TOKENS", "128")
    case = workloads.custom_case("ws", lens=[900, 1500, 33], num_q_heads=8, num_kv_heads=2,
                                 head_dim=128, block_size=16, dtype=torch.bfloat16, seed=8)
    ref, _, _ = gpu_step(case)
    need = wllm.workspace_bytes(3, 8, 2, 128, case.max_blocks, 16)
    assert need > 0
    buf = torch.empty(need, dtype=torch.uint8, device="cuda")
    try:
        wllm.set_workspace(buf)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            got, _, _ = gpu_step(case)
        assert torch.equal(int_view(got), int_view(ref))
        wllm.set_workspace(buf[: 256])
        kc, vc = case.pool("cuda")
        q = case.q.cuda()
        with pytest.raises(wllm.WllmError) as e:
            wllm.paged_attention_decode(torch.empty_like(q), q, kc, vc, case.block_tables.cuda(),
                                        case.context_lens.cuda(), 2, case.scale, 16)
        assert e.value.status == 1
    finally:
        wllm.set_workspace(None)


def test_invalid_arguments_raise():
    q = torch.zeros(2, 4, 64, dtype=torch.float16, device="cuda")
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.float16, device="cuda")
    bt = torch.zeros(2, 2, dtype=torch.int32, device="cuda")
    cl = torch.ones(2, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    cases = [
        dict(kv=3),                       # num_kv_heads mismatch
        dict(bs=8),                       # block_size mismatch
        dict(cl=cl.long()),               # wrong dtype
        dict(q=q.float()),                # dtype mismatch
    ]
    for c in cases:
        with pytest.raises(wllm.WllmError) as e:
            wllm.paged_attention_decode(out, c.get("q", q), kc, kc, bt, c.get("cl", cl),
                                        c.get("kv", 2), 0.125, c.get("bs", 16))
        assert e.value.status == 1
    with pytest.raises(wllm.WllmError) as e:  # unsupported head_dim
        q96 = torch.zeros(2, 4, 96, dtype=torch.float16, device="cuda")
        k96 = torch.zeros(4, 2, 16, 96, dtype=torch.float16, device="cuda")
        wllm.paged_attention_decode(torch.empty_like(q96), q96, k96, k96, bt, cl, 2, 0.1, 16)
    assert e.value.status == 2


def test_empty_batch_is_a_no_op():
    q = torch.zeros(0, 4, 64, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    wllm.paged_attention_decode(torch.empty_like(q), q, kc, kc, torch.zeros(0, 3, dtype=torch.int32,
                                device="cuda"), torch.zeros(0, dtype=torch.int32, device="cuda"),
                                2, 0.125, 16)
    key = torch.zeros(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    wllm.reshape_and_cache(key, key, kc, kc, torch.zeros(0, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# kernel selection: persistent (default for f16/bf16) vs one-CTA-per-unit grid
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,Hq,Hkv,D,bs", [s for s in SHAPES if s[0] != torch.float32][::2])
def test_grid_kernel_variant(monkeypatch, dtype, Hq, Hkv, D, bs):
    monkeypatch.setenv("WLLM_DECODE_KERNEL", "grid")
    case = workloads.custom_case("grid", lens=LENS, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                                 block_size=bs, dtype=dtype, seed=Hq + D, spare_blocks=2)
    got, _, _ = gpu_step(case)
    ref, _, _ = oracle_step(case)
    assert_attention_close(got, ref, dtype, f"grid {Hq}/{Hkv} D{D} bs{bs}")


def test_unaligned_query_rows_fall_back():
    """q rows only 4-byte aligned: the bulk-copy path is skipped, result unchanged."""
    case = workloads.custom_case("qalign", lens=[5, 200, 1500], num_q_heads=8, num_kv_heads=2,
                                 head_dim=128, block_size=16, dtype=torch.bfloat16, seed=12)
    kc, vc = case.pool("cuda")
    wllm.reshape_and_cache(case.key.cuda(), case.value.cuda(), kc, vc, case.slot_mapping.cuda())
    buf = torch.zeros(3, 8, 128 + 2, dtype=torch.bfloat16, device="cuda")
    q = buf[:, :, 2:]
    q.copy_(case.q.cuda())
    out = torch.empty(3, 8, 128, dtype=torch.bfloat16, device="cuda")
    wllm.paged_attention_decode(out, q, kc, vc, case.block_tables.cuda(), case.context_lens.cuda(), 2,
                                case.scale, 16)
    torch.cuda.synchronize()
    ref, _, _ = oracle_step(case)
    assert_attention_close(out.cpu(), ref, case.dtype, "unaligned q")


def test_large_batch_is_sliced():
    """More sequences than one persistent launch takes (1024): the host slices the batch."""
    g = torch.Generator().manual_seed(13)
    lens = torch.randint(1, 40, (4300,), generator=g).tolist()
    case = workloads.custom_case("big", lens=lens, num_q_heads=4, num_kv_heads=1, head_dim=64,
                                 block_size=16, dtype=torch.float16, seed=13)
    got, _, _ = gpu_step(case)
    ref, _, _ = oracle_step(case)
    assert_attention_close(got, ref, case.dtype, "4300 sequences")


def test_large_batch_fused_step_with_splits(monkeypatch):
    """A fused step over more sequences than one launch takes, split into
    partitions: the first slice's launch appends every sequence's rows, the
    later slices decode after it, each slice merges its split rows."""
    monkeypatch.setenv("WLLM_PARTITION_TOKENS", "256")
    g = torch.Generator().manual_seed(15)
    lens = torch.randint(1, 1500, (1100,), generator=g).tolist()
    case = workloads.custom_case("big_step", lens=lens, num_q_heads=4, num_kv_heads=1, head_dim=64,
                                 block_size=16, dtype=torch.float16, seed=15)
    got, kc, vc = fused_step(case)
    ref, kr, vr = oracle_step(case)
    assert torch.equal(int_view(kc.cpu()), int_view(kr)), "K append not bit-exact"
    assert torch.equal(int_view(vc.cpu()), int_view(vr)), "V append not bit-exact"
    del kc, vc
    assert_attention_close(got, ref, case.dtype, "1100 sequences, fused step")
    assert wllm.device_errors() == 0


def test_repeated_launches_leave_scheduler_clean():
    case = workloads.custom_case("rep", lens=[3000, 17, 900], num_q_heads=28, num_kv_heads=4,
                                 head_dim=128, block_size=16, dtype=torch.bfloat16, seed=14)
    first, kc, vc = gpu_step(case)
    q = case.q.cuda()
    for _ in range(5):
        out = torch.empty_like(q)
        wllm.paged_attention_decode(out, q, kc, vc, case.block_tables.cuda(), case.context_lens.cuda(),
                                    4, case.scale, 16)
        torch.cuda.synchronize()
        assert torch.equal(int_view(out.cpu()), int_view(first))


# ---------------------------------------------------------------------------
# the fused decode step (append + decode + combine in one launch)
# ---------------------------------------------------------------------------

def fused_step(case, pools=None):
    kc, vc = pools if pools is not None else case.pool("cuda")
    q = case.q.cuda()
    out = torch.empty_like(q)
    wllm.decode_step(out, q, case.key.cuda(), case.value.cuda(), kc, vc, case.slot_mapping.cuda(),
                     case.block_tables.cuda(), case.context_lens.cuda(), case.num_kv_heads, case.scale,
                     case.block_size)
    torch.cuda.synchronize()
    return out.cpu(), kc, vc


@pytest.mark.parametrize("name", ["c0", "c1", "c2", "c3"])
def test_fused_step_matches_oracle(name):
    case = workloads.make_case(name)
    got, kc, vc = fused_step(case)
    ref, kr, vr = oracle_step(case)
    assert torch.equal(int_view(kc.cpu()), int_view(kr)), "K append not bit-exact"
    assert torch.equal(int_view(vc.cpu()), int_view(vr)), "V append not bit-exact"
    del kc, vc
    assert_attention_close(got, ref, case.dtype, f"fused {name}")


@pytest.mark.parametrize("part", [64, 256])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_fused_step_split(monkeypatch, part, dtype):
    monkeypatch.setenv("WLLM_PARTITION_TOKENS", str(part))
    lens = [1, 63, 64, 65, 500, 1000, 2049, 0, 3000]
    case = workloads.custom_case("fsplit", lens=lens, num_q_heads=28, num_kv_heads=4, head_dim=128,
                                 block_size=16, dtype=dtype, seed=part + 5, heavy_key_frac=0.02)
    got, _, _ = fused_step(case)
    ref, _, _ = oracle_step(case)
    assert_attention_close(got, ref, dtype, f"fused split {part}")
    got2, _, _ = fused_step(case)  # scheduler and barrier words left clean
    assert torch.equal(int_view(got), int_view(got2))


@pytest.mark.parametrize("dtype,Hq,Hkv,D,bs", [SHAPES[0], SHAPES[4], SHAPES[8], SHAPES[12], SHAPES[15]])
def test_fused_step_shapes(dtype, Hq, Hkv, D, bs):
    case = workloads.custom_case("fshape", lens=LENS, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                                 block_size=bs, dtype=dtype, seed=Hq + D + bs + 1, spare_blocks=2)
    got, kc, vc = fused_step(case)
    ref, kr, vr = oracle_step(case)
    assert torch.equal(int_view(kc.cpu()), int_view(kr))
    assert_attention_close(got, ref, dtype, f"fused {dtype} {Hq}/{Hkv} D{D} bs{bs}")


@pytest.mark.parametrize("D,Hq,Hkv,dtype", [(64, 32, 4, torch.float16), (256, 8, 1, torch.bfloat16),
                                           (128, 32, 32, torch.bfloat16)])
def test_split_merge_head_dims(monkeypatch, D, Hq, Hkv, dtype):
    """In-launch merge of split sequences at every head_dim, twice in a row
    (scheduler and barrier words must be back at zero after each launch)."""
    monkeypatch.setenv("WLLM_PARTITION_TOKENS", "128")
    lens = [1, 129, 700, 2049, 0, 1300, 128, 257]
    case = workloads.custom_case("merge", lens=lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                                 block_size=16, dtype=dtype, seed=D + Hq, heavy_key_frac=0.02)
    got, _, _ = gpu_step(case)
    ref, _, _ = oracle_step(case)
    assert_attention_close(got, ref, dtype, f"merge D{D}")
    got2, _, _ = fused_step(case)
    assert torch.equal(int_view(got), int_view(got2))


@pytest.mark.parametrize("value", ["1", "0"])
def test_other_combine_modes(monkeypatch, value):
    """Split partitions merged by a second kernel (=1) or inside the launch
    (=0), forced against the default for the batch size."""
    monkeypatch.setenv("WLLM_SEPARATE_COMBINE", value)
    monkeypatch.setenv("WLLM_PARTITION_TOKENS", "128")
    lens = [5, 900, 2500, 1] if value == "1" else [5, 900, 2500, 1] * 160  # 640 x 8 rows: above the switch
    case = workloads.custom_case("sep", lens=lens, num_q_heads=8, num_kv_heads=2,
                                 head_dim=64, block_size=16, dtype=torch.float16, seed=44)
    got, _, _ = gpu_step(case)
    ref, _, _ = oracle_step(case)
    what = f"WLLM_SEPARATE_COMBINE={value}"
    assert_attention_close(got, ref, case.dtype, what)
    got2, _, _ = fused_step(case)
    assert_attention_close(got2, ref, case.dtype, what + ", step")


def test_fused_steps_of_different_grid_sizes():
    """Fused steps whose launches have very different grids (4 CTAs, then a
    full persistent grid), alternated on one device: the grid barrier's count
    stays consistent across grid sizes, so every step appends bit for bit and
    decodes against the oracle, with no error reported."""
    small = workloads.custom_case("grid_small", lens=[40, 17], num_q_heads=4, num_kv_heads=2, head_dim=64,
                                  block_size=16, dtype=torch.bfloat16, seed=46)
    rng = np.random.default_rng(47)
    big = workloads.custom_case("grid_big", lens=rng.integers(300, 1200, 64).tolist(), num_q_heads=32,
                                num_kv_heads=4, head_dim=64, block_size=16, dtype=torch.float16, seed=48)
    refs = {c.name: oracle_step(c) for c in (small, big)}
    assert wllm.device_errors() == 0
    for case in (small, big, small, big, big, small, big):
        got, kc, vc = fused_step(case)
        ref, kr, vr = refs[case.name]
        assert torch.equal(int_view(kc.cpu()), int_view(kr)), f"{case.name}: K append not bit-exact"
        assert torch.equal(int_view(vc.cpu()), int_view(vr)), f"{case.name}: V append not bit-exact"
        assert_attention_close(got, ref, case.dtype, f"{case.name} after a launch of another grid size")
        assert wllm.device_errors() == 0


def test_fused_step_without_tokens_or_sequences():
    case = workloads.custom_case("noapp", lens=[40, 17], num_q_heads=4, num_kv_heads=2, head_dim=64,
                                 block_size=16, dtype=torch.bfloat16, seed=45, append="none")
    got, _, _ = fused_step(case)
    ref, _, _ = oracle_step(case)
    assert_attention_close(got, ref, case.dtype, "no append")
    # attention over nothing, append only
    kc = torch.zeros(2, 1, 16, 64, dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    key = torch.ones(1, 1, 64, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(0, 1, 64, dtype=torch.bfloat16, device="cuda")
    wllm.decode_step(torch.empty_like(q), q, key, key, kc, vc, torch.tensor([17], device="cuda"),
                     torch.zeros(0, 2, dtype=torch.int32, device="cuda"),
                     torch.zeros(0, dtype=torch.int32, device="cuda"), 1, 0.1, 16)
    torch.cuda.synchronize()
    assert kc[1, 0, 1].float().sum().item() == 64


# ---------------------------------------------------------------------------
# prefix groups: sequences sharing a partition's blocks are processed once
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("gsize,shared,part", [(8, 64, 512), (12, 40, 128), (3, 33, 256), (5, 16, 256),
                                               (1, 20, 128), (9, 8, 128)])
@pytest.mark.parametrize("dtype,Hq,Hkv,D", [(torch.bfloat16, 28, 4, 128), (torch.float16, 16, 4, 64)])
def test_prefix_groups(monkeypatch, gsize, shared, part, dtype, Hq, Hkv, D):
    monkeypatch.setenv("WLLM_PARTITION_TOKENS", str(part))
    monkeypatch.setenv("WLLM_PREFIX_GROUPS", "1")
    g = torch.Generator().manual_seed(gsize * 100 + shared)
    n_groups = 3
    lens = [shared * 16 + int(x) for x in torch.randint(1, 700, (gsize * n_groups,), generator=g)]
    lens[0] = shared * 16 + 1  # a member whose only private token is the appended one
    case = workloads.custom_case("groups", lens=lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                                 block_size=16, dtype=dtype, seed=gsize + shared, groups=(gsize, shared))
    got, _, _ = gpu_step(case)
    ref, _, _ = oracle_step(case)
    assert_attention_close(got, ref, dtype, f"groups {gsize}x{shared} P{part}")
    got_f, _, _ = fused_step(case)
    assert_attention_close(got_f, ref, dtype, f"groups fused {gsize}x{shared} P{part}")
    monkeypatch.setenv("WLLM_PREFIX_GROUPS", "0")
    got0, _, _ = gpu_step(case)
    assert_attention_close(got0, ref, dtype, "groups off")
