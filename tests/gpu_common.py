"""Shared helpers of the GPU parity tests: run a workload through the C ABI
(via the Python binding) and through the oracle, and compare."""
import torch

import oracle
import paged_kv_cache_185_gb300 as wllm

# Tolerances of the attention output against the fp64 oracle.
FP32_MAX_ABS = 1e-5
LOWP_MAX_ABS = 2e-2
LOWP_REL_L2 = 5e-3


def int_view(t: torch.Tensor) -> torch.Tensor:
    return t.view({4: torch.int32, 2: torch.int16}[t.element_size()])


def gpu_step(case, device="cuda", pools=None):
    """Append + decode on the GPU.  Returns (out on host, k_pool, v_pool on device)."""
    kc, vc = pools if pools is not None else case.pool(device)
    q = case.q.to(device)
    out = torch.empty_like(q)
    if case.slot_mapping.numel():
        wllm.reshape_and_cache(case.key.to(device), case.value.to(device), kc, vc,
                               case.slot_mapping.to(device))
    wllm.paged_attention_decode(out, q, kc, vc, case.block_tables.to(device),
                                case.context_lens.to(device), case.num_kv_heads, case.scale,
                                case.block_size)
    torch.cuda.synchronize()
    return out.cpu(), kc, vc


def oracle_step(case, rows=None, compact=False):
    """Append + decode in the oracle.  Returns (out float64, k_pool, v_pool) on the host."""
    if compact:
        kc, vc, bt, slots = case.compact()
    else:
        kc, vc = case.pool("cpu")
        bt, slots = case.block_tables, case.slot_mapping
    if slots.numel():
        oracle.reshape_and_cache(case.key, case.value, kc, vc, slots)
    out = oracle.paged_decode(case.q, kc, vc, bt, case.context_lens, case.num_kv_heads,
                              case.scale, rows=rows)
    return out, kc, vc


def assert_attention_close(got: torch.Tensor, ref: torch.Tensor, dtype: torch.dtype, what=""):
    got = got.to(torch.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert torch.isfinite(got).all(), f"{what}: non-finite output"
    err = (got - ref).abs().max().item()
    if dtype == torch.float32:
        assert err <= FP32_MAX_ABS, f"{what}: max-abs {err:.3e} > {FP32_MAX_ABS}"
    else:
        rel = ((got - ref).norm() / ref.norm().clamp_min(1e-30)).item()
        assert err <= LOWP_MAX_ABS, f"{what}: max-abs {err:.3e} > {LOWP_MAX_ABS}"
        assert rel <= LOWP_REL_L2, f"{what}: rel-L2 {rel:.3e} > {LOWP_REL_L2}"
    return err
