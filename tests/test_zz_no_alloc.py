"""The allocation-free decode entry point, through the C ABI.

For callers that cannot let the library allocate device memory (a CUDA-graph
capture in progress, a memory manager that owns all device memory, a caller
that cannot take cudaMalloc's implicit synchronisation), the library offers a
decode call whose scratch is a fixed array in its device image.  This file
checks that call against the regular entry point on two calls in a row, and
that sizes beyond the fixed array are refused without launching anything.
It is collected last so that a failure here leaves every other test run.
"""
import pytest
import torch

import paged_kv_cache_185_gb300 as wllm
from paged_kv_cache_185_gb300 import workloads
from tests.gpu_common import LOWP_MAX_ABS, LOWP_REL_L2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_kv_cache_185_gb300 import build
    build.build()
    wllm.load_library()


def _close(a, b):
    a, b = a.double(), b.double()
    assert torch.isfinite(a).all()
    err = (a - b).abs().max().item()
    rel = ((a - b).norm() / b.norm()).item()
    assert err <= LOWP_MAX_ABS and rel <= LOWP_REL_L2, (err, rel)


@pytest.mark.parametrize("part_tokens", ["", "256"])
def test_noalloc_matches_regular_decode_twice(monkeypatch, part_tokens):
    if part_tokens:
        monkeypatch.setenv("WLLM_PARTITION_TOKENS", part_tokens)  # several partitions: scratch in use
    case = workloads.custom_case("noalloc", lens=[1, 17, 300, 1000, 2500, 0, 4000], num_q_heads=28,
                                 num_kv_heads=4, head_dim=128, block_size=16, dtype=torch.bfloat16,
                                 seed=21, heavy_key_frac=0.01)
    kc, vc = case.pool("cuda")
    wllm.reshape_and_cache(case.key.cuda(), case.value.cuda(), kc, vc, case.slot_mapping.cuda())
    q, bt, cl = case.q.cuda(), case.block_tables.cuda(), case.context_lens.cuda()
    ref = torch.empty_like(q)
    wllm.paged_attention_decode(ref, q, kc, vc, bt, cl, case.num_kv_heads, case.scale, case.block_size)
    outs = []
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        wllm.paged_attention_decode_noalloc(out, q, kc, vc, bt, cl, case.num_kv_heads, case.scale,
                                            case.block_size)
        outs.append(out)
    torch.cuda.synchronize()
    for out in outs:
        _close(out.cpu(), ref.cpu())


def test_noalloc_second_call_with_other_inputs():
    """The array keeps the previous call's partials; a new call must not depend on them."""
    for seed in (31, 32):
        case = workloads.custom_case("noalloc2", lens=[700, 3000, 64], num_q_heads=32, num_kv_heads=8,
                                     head_dim=64, block_size=16, dtype=torch.float16, seed=seed)
        kc, vc = case.pool("cuda")
        wllm.reshape_and_cache(case.key.cuda(), case.value.cuda(), kc, vc, case.slot_mapping.cuda())
        q, bt, cl = case.q.cuda(), case.block_tables.cuda(), case.context_lens.cuda()
        ref = torch.empty_like(q)
        wllm.paged_attention_decode(ref, q, kc, vc, bt, cl, 8, case.scale, 16)
        out = torch.empty_like(q)
        wllm.paged_attention_decode_noalloc(out, q, kc, vc, bt, cl, 8, case.scale, 16)
        torch.cuda.synchronize()
        _close(out.cpu(), ref.cpu())


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
