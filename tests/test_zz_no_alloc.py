"""The allocation-free decode entry point, through the C ABI.

Some callers cannot let the library allocate device memory: an engine whose
memory manager already owns all device memory, or a latency-critical caller
that cannot take cudaMalloc's implicit synchronisation.  For them the library
offers a decode call whose scratch is a fixed array in its device image.  This
file checks that call against the fp64 oracle and against the regular entry
point on two calls in a row, that device-detected index errors reach
wllm_device_errors(), that batches cut into several launches reuse the array
correctly, and that sizes beyond the fixed array are refused without
launching anything.  It is collected last so that a failure here leaves every
other test run.
"""
import pytest
import torch

import paged_kv_cache_185_gb300 as wllm
from paged_kv_cache_185_gb300 import workloads
from tests.gpu_common import assert_attention_close, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_kv_cache_185_gb300 import build
    build.build()
    wllm.load_library()
    yield
    assert wllm.device_errors() == 0


def _inputs(case):
    kc, vc = case.pool("cuda")
    if case.slot_mapping.numel():
        wllm.reshape_and_cache(case.key.cuda(), case.value.cuda(), kc, vc, case.slot_mapping.cuda())
    return kc, vc, case.q.cuda(), case.block_tables.cuda(), case.context_lens.cuda()


@pytest.mark.parametrize("part_tokens", ["", "256"])
def test_noalloc_matches_oracle_and_regular_decode_twice(monkeypatch, part_tokens):
    if part_tokens:
        monkeypatch.setenv("WLLM_PARTITION_TOKENS", part_tokens)  # several partitions: scratch in use
    case = workloads.custom_case("noalloc", lens=[1, 17, 300, 1000, 2500, 0, 4000], num_q_heads=28,
                                 num_kv_heads=4, head_dim=128, block_size=16, dtype=torch.bfloat16,
                                 seed=21, heavy_key_frac=0.01)
    kc, vc, q, bt, cl = _inputs(case)
    regular = torch.empty_like(q)
    wllm.paged_attention_decode(regular, q, kc, vc, bt, cl, case.num_kv_heads, case.scale, case.block_size)
    outs = []
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        wllm.paged_attention_decode_noalloc(out, q, kc, vc, bt, cl, case.num_kv_heads, case.scale,
                                            case.block_size)
        outs.append(out)
    torch.cuda.synchronize()
    ref, _, _ = oracle_step(case)
    for i, out in enumerate(outs):
        assert_attention_close(out.cpu(), ref, case.dtype, f"no-alloc call {i} vs oracle")
        assert_attention_close(out.cpu(), regular.cpu().double(), case.dtype, f"no-alloc call {i} vs regular")
    assert wllm.device_errors() == 0


def test_noalloc_second_call_with_other_inputs():
    """The array keeps the previous call's partials; a new call must not depend on them."""
    for seed in (31, 32):
        case = workloads.custom_case("noalloc2", lens=[700, 3000, 64], num_q_heads=32, num_kv_heads=8,
                                     head_dim=64, block_size=16, dtype=torch.float16, seed=seed)
        kc, vc, q, bt, cl = _inputs(case)
        out = torch.empty_like(q)
        wllm.paged_attention_decode_noalloc(out, q, kc, vc, bt, cl, 8, case.scale, 16)
        torch.cuda.synchronize()
        ref, _, _ = oracle_step(case)
        assert_attention_close(out.cpu(), ref, case.dtype, f"seed {seed}")


def test_noalloc_batch_over_several_launches(monkeypatch):
    """More sequences than one launch takes: the slices run one after another
    on the same stream and reuse the one array."""
    monkeypatch.setenv("WLLM_PARTITION_TOKENS", "64")
    g = torch.Generator().manual_seed(5)
    lens = torch.randint(0, 200, (1100,), generator=g).tolist()
    case = workloads.custom_case("noalloc_slices", lens=lens, num_q_heads=8, num_kv_heads=2, head_dim=64,
                                 block_size=16, dtype=torch.float16, seed=51)
    kc, vc, q, bt, cl = _inputs(case)
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        wllm.paged_attention_decode_noalloc(out, q, kc, vc, bt, cl, 2, case.scale, 16)
        torch.cuda.synchronize()
        ref, _, _ = oracle_step(case)
        assert_attention_close(out.cpu(), ref, case.dtype, "1100 sequences")


def test_noalloc_reports_clamped_indices():
    """Out-of-range block ids and lengths are clamped on the device (no stray
    access) and reported through wllm_device_errors(), like the regular call;
    the other sequences' outputs are unaffected."""
    case = workloads.custom_case("noalloc_err", lens=[40, 500, 33, 900], num_q_heads=8, num_kv_heads=2,
                                 head_dim=128, block_size=16, dtype=torch.bfloat16, seed=61, append="none")
    kc, vc, q, bt, cl = _inputs(case)
    ref, _, _ = oracle_step(case)
    assert wllm.device_errors() == 0
    bad = bt.clone()
    bad[1, 3] = case.num_blocks + 5      # inside sequence 1's used range
    bad[3, 0] = -7                       # first block of sequence 3
    out = torch.empty_like(q)
    wllm.paged_attention_decode_noalloc(out, q, kc, vc, bad, cl, 2, case.scale, 16)
    torch.cuda.synchronize()
    word = wllm.device_errors()
    assert word & 2, f"block-id bit not reported: 0x{word:x}"
    assert wllm.device_errors() == 0, "reading the word clears it"
    got = out.cpu()
    for b in (0, 2):
        assert_attention_close(got[b], ref[b], case.dtype, f"untouched sequence {b}")
    # a length above the table's reach is clamped and reported too
    long_cl = cl.clone()
    long_cl[2] = case.max_blocks * 16 + 100
    wllm.paged_attention_decode_noalloc(out, q, kc, vc, bt, long_cl, 2, case.scale, 16)
    torch.cuda.synchronize()
    assert wllm.device_errors() & 4
    # the array is usable again afterwards
    wllm.paged_attention_decode_noalloc(out, q, kc, vc, bt, cl, 2, case.scale, 16)
    torch.cuda.synchronize()
    assert wllm.device_errors() == 0
    assert_attention_close(out.cpu(), ref, case.dtype, "after the errors")


def test_noalloc_refuses_sizes_beyond_its_array(monkeypatch):
    monkeypatch.setenv("WLLM_PARTITION_TOKENS", "16")
    B, Hq, Hkv, D, M_b = 1024, 32, 8, 128, 256
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(2, Hkv, 16, D, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(B, M_b, dtype=torch.int32, device="cuda")
    cl = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 7.0)
    with pytest.raises(wllm.WllmError) as e:
        wllm.paged_attention_decode_noalloc(out, q, kc, kc, bt, cl, Hkv, 0.1, 16)
    assert e.value.status == 2 and "scratch" in str(e.value)
    torch.cuda.synchronize()
    assert (out == 7.0).all()  # nothing launched
