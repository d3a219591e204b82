"""Chunked-prefill paged attention on the GPU, through the C ABI, against the
oracle: packed query chunks (fresh prompts, continued prompts, one-token and
empty chunks), GQA/MHA, head dims 64/128, block sizes 8..64, and a large
sampled case.  16-bit caches run on the tcgen05 kernel when the q/out rows are
16-byte aligned; the mma.sync kernel (WLLM_PREFILL_KERNEL=mma, misaligned rows,
fp8 caches) is covered by the same cases."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_185_gb300 as wllm
from paged_kv_cache_185_gb300.workloads import custom_case
from tests.gpu_common import assert_attention_close

pytestmark = pytest.mark.gpu


def prefill_case(lens, chunks, Hq, Hkv, D, bs, dtype, seed, **kw):
    """Pools holding every sequence's L tokens (the chunk's K/V appended) and packed query chunks."""
    case = custom_case("prefill", lens=lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                       dtype=dtype, seed=seed, spare_blocks=2, append="none", **kw)
    gen = torch.Generator().manual_seed(seed + 7)
    T = int(sum(chunks))
    q = torch.randn(T, Hq, D, generator=gen).to(dtype)
    qsl = torch.tensor(np.concatenate([[0], np.cumsum(chunks)]), dtype=torch.int32)
    return case, q, qsl


def run_gpu(case, q, qsl, out=None):
    dev = "cuda"
    kc, vc = case.pool(dev)
    qd = q.to(dev)
    o = torch.empty_like(qd) if out is None else out
    wllm.paged_attention_prefill(o, qd, kc, vc, case.block_tables.to(dev), case.context_lens.to(dev), qsl.to(dev),
                                 case.num_kv_heads, case.scale, case.block_size)
    torch.cuda.synchronize()
    return o.cpu()


def run_oracle(case, q, qsl, rows=None):
    kc, vc = case.pool("cpu")
    return oracle.paged_prefill(q, kc, vc, case.block_tables, case.context_lens, qsl, case.num_kv_heads,
                                case.scale, rows=rows)


CASES = [
    # (Hq, Hkv, D, bs, lens, chunks)
    (8, 8, 128, 16, [200, 64, 1, 77, 500, 33], [200, 64, 1, 13, 129, 0]),    # MHA: fresh, continued, 1, 0
    (32, 8, 128, 16, [300, 1000, 17, 65], [300, 255, 17, 1]),                 # GQA 4
    (28, 4, 128, 32, [513, 90, 1200], [513, 90, 70]),                         # GQA 7, bs 32
    (12, 1, 64, 8, [100, 257, 31], [100, 200, 9]),                            # MQA, D 64, bs 8
    (16, 2, 64, 64, [640, 1, 129], [128, 1, 129]),                            # D 64, bs 64
    (64, 4, 128, 16, [150, 333], [150, 20]),                                  # GQA 16
]


@pytest.fixture(params=["tcgen05", "mma"])
def kernel(request, monkeypatch):
    if request.param == "mma":
        monkeypatch.setenv("WLLM_PREFILL_KERNEL", "mma")
    return request.param


@pytest.mark.parametrize("Hq,Hkv,D,bs,lens,chunks", CASES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_prefill_matches_oracle(Hq, Hkv, D, bs, lens, chunks, dtype, kernel):
    case, q, qsl = prefill_case(lens, chunks, Hq, Hkv, D, bs, dtype, seed=Hq * 3 + D + bs)
    got = run_gpu(case, q, qsl)
    ref = run_oracle(case, q, qsl)
    assert_attention_close(got, ref, dtype, f"prefill {Hq}/{Hkv} D{D} bs{bs}")


@pytest.mark.parametrize("nseq", [64, 70])
def test_prefill_many_sequences_in_either_launch_order(nseq, kernel):
    """Up to 64 sequences the tcgen05 kernel launches its CTAs longest context
    first (equal lengths in sequence order); above 64, in sequence order: every
    row block is covered exactly once either way."""
    rng = np.random.default_rng(nseq)
    lens = rng.integers(1, 400, size=nseq)
    lens[::5] = 300  # ties in the ranking
    chunks = np.minimum(lens, rng.integers(0, 40, size=nseq))
    case, q, qsl = prefill_case(lens, chunks, 16, 4, 64, 16, torch.float16, seed=nseq + 3)
    assert_attention_close(run_gpu(case, q, qsl), run_oracle(case, q, qsl), torch.float16, f"{nseq} sequences")


def test_prefill_one_token_chunks_match_decode(kernel):
    # n_b = 1 everywhere: the decode's answer
    rng = np.random.default_rng(2)
    lens = rng.integers(1, 3000, size=20)
    case, q, qsl = prefill_case(lens, [1] * 20, 28, 4, 128, 16, torch.bfloat16, seed=21)
    got = run_gpu(case, q, qsl)
    dev = "cuda"
    kc, vc = case.pool(dev)
    dec = torch.empty(20, 28, 128, dtype=torch.bfloat16, device=dev)
    wllm.paged_attention_decode(dec, q.to(dev), kc, vc, case.block_tables.to(dev), case.context_lens.to(dev), 4,
                                case.scale, 16)
    ref = run_oracle(case, q, qsl)
    assert_attention_close(got, ref, torch.bfloat16, "prefill n=1")
    assert_attention_close(dec.cpu(), ref, torch.bfloat16, "decode")


def test_prefill_strided_output_and_query(kernel):
    # q and out as slices of wider buffers (a fused QKV projection and a padded output)
    case, q, qsl = prefill_case([90, 40], [90, 15], 8, 2, 64, 16, torch.float16, seed=31)
    dev = "cuda"
    wide_q = torch.zeros(q.shape[0], 12, 64, dtype=q.dtype, device=dev)
    wide_q[:, 2:10] = q.to(dev)
    wide_o = torch.full((q.shape[0], 10, 64), 7.0, dtype=q.dtype, device=dev)
    kc, vc = case.pool(dev)
    wllm.paged_attention_prefill(wide_o[:, 1:9], wide_q[:, 2:10], kc, vc, case.block_tables.to(dev),
                                 case.context_lens.to(dev), qsl.to(dev), 2, case.scale, 16)
    torch.cuda.synchronize()
    assert_attention_close(wide_o[:, 1:9].cpu(), run_oracle(case, q, qsl), torch.float16, "strided")
    assert (wide_o[:, 0] == 7).all() and (wide_o[:, 9] == 7).all()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_prefill_heavy_keys_move_the_running_max(dtype, kernel):
    """3% of the keys scaled x8: scores jump by far more than 2^8 in the log2
    domain deep into the context, so the running maximum moves mid-row and O
    is rescaled (in TMEM, for the tcgen05 kernel)."""
    case, q, qsl = prefill_case([1500, 900, 2100], [300, 900, 64], 28, 4, 128, 16, dtype, seed=71,
                                heavy_key_frac=0.03, heavy_key_factor=8.0)
    got = run_gpu(case, q, qsl)
    assert_attention_close(got, run_oracle(case, q, qsl), dtype, f"heavy keys {kernel}")


def test_prefill_misaligned_rows_use_the_mma_kernel():
    """q rows only 4-byte aligned: the call still succeeds (mma.sync kernel)."""
    case, q, qsl = prefill_case([70, 200], [70, 33], 8, 2, 64, 16, torch.float16, seed=72)
    dev = "cuda"
    buf = torch.zeros(q.numel() + 2, dtype=q.dtype, device=dev)
    qd = buf[2:].view(q.shape)
    qd.copy_(q.to(dev))
    kc, vc = case.pool(dev)
    out = torch.empty(q.shape, dtype=q.dtype, device=dev)
    wllm.paged_attention_prefill(out, qd, kc, vc, case.block_tables.to(dev), case.context_lens.to(dev), qsl.to(dev),
                                 2, case.scale, 16)
    torch.cuda.synchronize()
    assert_attention_close(out.cpu(), run_oracle(case, q, qsl), torch.float16, "misaligned q")


def test_prefill_long_chunks_sampled(kernel):
    # four sequences, 1024-token chunks after 0..3000 tokens of context: sampled rows
    rng = np.random.default_rng(4)
    prior = rng.integers(0, 3000, size=4)
    chunks = [1024] * 4
    lens = [int(p) + 1024 for p in prior]
    case, q, qsl = prefill_case(lens, chunks, 32, 8, 128, 16, torch.bfloat16, seed=41)
    got = run_gpu(case, q, qsl)
    rows = np.sort(rng.choice(q.shape[0] * 32, size=256, replace=False))
    ref = run_oracle(case, q, qsl, rows=torch.from_numpy(rows))
    assert_attention_close(got.reshape(-1, 128)[torch.from_numpy(rows)], ref, torch.bfloat16, "long chunks")


def test_prefill_reports_inconsistent_query_starts(monkeypatch):
    monkeypatch.setenv("WLLM_CHECK", "1")
    case, q, qsl = prefill_case([40, 40], [20, 20], 8, 2, 64, 16, torch.bfloat16, seed=51)
    bad = qsl.clone()
    bad[1] = 30  # sequence 0 now claims 30 query rows ...
    cl = case.context_lens.clone()
    cl[0] = 25  # ... but holds 25 tokens: a chunk longer than its context
    dev = "cuda"
    kc, vc = case.pool(dev)
    out = torch.zeros(q.shape, dtype=q.dtype, device=dev)
    with pytest.raises(wllm.WllmError):
        wllm.paged_attention_prefill(out, q.to(dev), kc, vc, case.block_tables.to(dev), cl.to(dev), bad.to(dev), 2,
                                     case.scale, 16)
    assert wllm.device_errors() == 0  # the failing call cleared the word


FP8_CASES = [c for c in CASES if not (c[2] == 64 and c[3] < 16)]  # D 64 needs blocks of >= 16 tokens


@pytest.mark.parametrize("Hq,Hkv,D,bs,lens,chunks", FP8_CASES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_prefill_fp8_matches_oracle(Hq, Hkv, D, bs, lens, chunks, dtype):
    from paged_kv_cache_185_gb300.workloads import e4m3_codes
    case, q, qsl = prefill_case(lens, chunks, Hq, Hkv, D, bs, dtype, seed=Hq * 5 + D + bs)
    kc, vc = case.pool("cpu")
    k8, v8 = e4m3_codes(kc, 4.0), e4m3_codes(vc, 4.0)
    dev = "cuda"
    out = torch.empty(q.shape, dtype=dtype, device=dev)
    wllm.paged_attention_prefill_fp8(out, q.to(dev), k8.to(dev), v8.to(dev), case.block_tables.to(dev),
                                     case.context_lens.to(dev), qsl.to(dev), Hkv, case.scale, 0.25, 0.3, bs)
    torch.cuda.synchronize()
    ref = oracle.paged_prefill(q, k8, v8, case.block_tables, case.context_lens, qsl, Hkv, case.scale,
                               k_scale=0.25, v_scale=0.3)
    assert_attention_close(out.cpu(), ref, dtype, f"fp8 prefill {Hq}/{Hkv} D{D} bs{bs}")


def test_prefill_fp8_long_chunks_sampled_and_refusals():
    from paged_kv_cache_185_gb300.workloads import e4m3_codes
    rng = np.random.default_rng(6)
    prior = rng.integers(0, 2500, size=3)
    lens = [int(p) + 700 for p in prior]
    case, q, qsl = prefill_case(lens, [700] * 3, 28, 4, 128, 16, torch.bfloat16, seed=61)
    kc, vc = case.pool("cpu")
    k8, v8 = e4m3_codes(kc, 4.0), e4m3_codes(vc, 4.0)
    dev = "cuda"
    out = torch.empty(q.shape, dtype=q.dtype, device=dev)
    wllm.paged_attention_prefill_fp8(out, q.to(dev), k8.to(dev), v8.to(dev), case.block_tables.to(dev),
                                     case.context_lens.to(dev), qsl.to(dev), 4, case.scale, 0.25, 0.25, 16)
    torch.cuda.synchronize()
    rows = np.sort(rng.choice(q.shape[0] * 28, size=200, replace=False))
    ref = oracle.paged_prefill(q, k8, v8, case.block_tables, case.context_lens, qsl, 4, case.scale,
                               rows=torch.from_numpy(rows), k_scale=0.25, v_scale=0.25)
    assert_attention_close(out.cpu().reshape(-1, 128)[torch.from_numpy(rows)], ref, torch.bfloat16, "fp8 long")
    # head_dim 64 with 8-token blocks is refused on the host
    c8, q8, qsl8 = prefill_case([40], [40], 4, 2, 64, 8, torch.float16, seed=62)
    k8, v8 = e4m3_codes(c8.pool("cpu")[0], 4.0), e4m3_codes(c8.pool("cpu")[1], 4.0)
    with pytest.raises(wllm.WllmError):
        wllm.paged_attention_prefill_fp8(torch.empty(q8.shape, dtype=q8.dtype, device=dev), q8.to(dev), k8.to(dev),
                                         v8.to(dev), c8.block_tables.to(dev), c8.context_lens.to(dev),
                                         qsl8.to(dev), 2, c8.scale, 1.0, 1.0, 8)
