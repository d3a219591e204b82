"""FP8 (E4M3) KV cache on the GPU, against the oracle: the quantising append
byte for byte, the decode over E4M3 codes within the low-precision tolerance,
and the fused step."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_185_gb300 as wllm
from paged_kv_cache_185_gb300.workloads import custom_case, e4m3_codes, make_case
from tests.gpu_common import assert_attention_close

pytestmark = pytest.mark.gpu

AMP = 4.0        # codes hold 4 x the drawn normal values ...
K_SCALE = 0.25   # ... so the dequantised K and V are back on the drawn scale
V_SCALE = 0.25


def fp8_pools(case, amp=AMP):
    kc, vc = case.pool("cpu")
    return e4m3_codes(kc, amp), e4m3_codes(vc, amp)


def gpu_decode_fp8(case, kc, vc, k_scale=K_SCALE, v_scale=V_SCALE):
    dev = "cuda"
    q = case.q.to(dev)
    out = torch.empty_like(q)
    wllm.paged_attention_decode_fp8(out, q, kc.to(dev), vc.to(dev), case.block_tables.to(dev),
                                    case.context_lens.to(dev), case.num_kv_heads, case.scale, k_scale, v_scale,
                                    case.block_size)
    torch.cuda.synchronize()
    return out.cpu()


def oracle_decode_fp8(case, kc, vc, k_scale=K_SCALE, v_scale=V_SCALE, rows=None):
    return oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, case.num_kv_heads,
                               case.scale, rows=rows, k_scale=k_scale, v_scale=v_scale)


# --------------------------------------------------------------------------
# append
# --------------------------------------------------------------------------

@pytest.mark.parametrize("src", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("slot_dtype", [torch.int64, torch.int32])
def test_fp8_append_is_bit_exact(src, slot_dtype):
    gen = torch.Generator().manual_seed(41)
    T, Hkv, D, nb, bs = 75, 4, 128, 24, 16
    # a fused QKV row [T][3*Hkv][D]: key and value are strided slices of it
    qkv = (torch.randn(T, 3 * Hkv, D, generator=gen) * 6).to(src)
    key, value = qkv[:, Hkv:2 * Hkv], qkv[:, 2 * Hkv:]
    slots = torch.randperm(nb * bs, generator=gen)[:T].to(torch.int64)
    slots[::9] = -1  # padding tokens
    k0 = torch.randint(0, 256, (nb, Hkv, bs, D), dtype=torch.uint8, generator=gen)
    v0 = torch.randint(0, 256, (nb, Hkv, bs, D), dtype=torch.uint8, generator=gen)
    ks, vs = 0.013, 0.021  # |x| / scale reaches past 448: the saturating path runs too
    kc, vc = k0.cuda(), v0.cuda()
    wllm.reshape_and_cache_fp8(key.cuda(), value.cuda(), kc, vc, slots.to(slot_dtype).cuda(), ks, vs)
    kr, vr = k0.clone(), v0.clone()
    oracle.reshape_and_cache_e4m3(key.contiguous(), value.contiguous(), kr, vr, slots, ks, vs)
    assert (kr == 0x7E).any() or (kr == 0xFE).any(), "the saturating case is exercised"
    assert torch.equal(kc.cpu(), kr)
    assert torch.equal(vc.cpu(), vr)


def test_fp8_append_accepts_float8_tensors_and_empty_input():
    gen = torch.Generator().manual_seed(42)
    key = torch.randn(5, 2, 256, generator=gen).half()
    value = torch.randn(5, 2, 256, generator=gen).half()
    kc = torch.zeros(4, 2, 8, 256, dtype=torch.float8_e4m3fn, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.tensor([0, 9, 31, 17, 3])
    wllm.reshape_and_cache_fp8(key.cuda(), value.cuda(), kc, vc, slots.cuda(), 1.0, 0.5)
    kr = torch.zeros(4, 2, 8, 256, dtype=torch.uint8)
    vr = torch.zeros_like(kr)
    oracle.reshape_and_cache_e4m3(key, value, kr, vr, slots, 1.0, 0.5)
    assert torch.equal(kc.view(torch.uint8).cpu(), kr) and torch.equal(vc.view(torch.uint8).cpu(), vr)
    e = torch.empty(0, 2, 256, dtype=torch.float16, device="cuda")
    wllm.reshape_and_cache_fp8(e, e, kc, vc, torch.empty(0, dtype=torch.int64, device="cuda"), 1.0, 1.0)


# --------------------------------------------------------------------------
# decode
# --------------------------------------------------------------------------

DECODE_CASES = [
    # (Hq, Hkv, D, bs, dtype, lens)
    (32, 32, 128, 16, torch.bfloat16, [0, 1, 15, 16, 17, 300, 1000, 5000, 64, 2049]),  # MHA, split
    (28, 4, 128, 16, torch.float16, [1, 33, 511, 512, 513, 4100, 70, 9000]),           # GQA 7
    (32, 8, 256, 8, torch.bfloat16, [5, 8, 9, 1500, 3333, 0, 100]),                    # D 256, bs 8
    (64, 4, 128, 32, torch.bfloat16, [31, 32, 33, 2500, 777]),                          # GQA 16: two head tiles
    (8, 1, 128, 64, torch.float16, [1, 127, 128, 129, 6000]),                           # one kv head
    (16, 2, 256, 16, torch.float16, [4097, 12, 900]),
    (32, 4, 64, 16, torch.float16, [1, 15, 16, 17, 700, 2048, 129]),                   # D 64 (two tokens a row)
    (16, 16, 64, 32, torch.bfloat16, [33, 1000, 5, 64]),                                # D 64 MHA, bs 32
]


@pytest.mark.parametrize("Hq,Hkv,D,bs,dtype,lens", DECODE_CASES)
def test_fp8_decode_matches_oracle(Hq, Hkv, D, bs, dtype, lens):
    case = custom_case("fp8", lens=lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                       dtype=dtype, seed=Hq * 7 + D + bs, spare_blocks=3, append="none")
    kc, vc = fp8_pools(case)
    got = gpu_decode_fp8(case, kc, vc)
    ref = oracle_decode_fp8(case, kc, vc)
    assert_attention_close(got, ref, dtype, f"fp8 {Hq}/{Hkv} D{D} bs{bs}")


@pytest.mark.parametrize("env", [{"WLLM_SEPARATE_COMBINE": "1"}, {"WLLM_PARTITION_TOKENS": "256"},
                                 {"WLLM_PARTITION_TOKENS": "4096"}])
def test_fp8_decode_merge_modes(env, monkeypatch):
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    rng = np.random.default_rng(7)
    lens = rng.integers(1, 6000, size=40)
    case = custom_case("fp8_modes", lens=lens, num_q_heads=28, num_kv_heads=4, head_dim=128, block_size=16,
                       dtype=torch.bfloat16, seed=77, append="none")
    kc, vc = fp8_pools(case)
    got = gpu_decode_fp8(case, kc, vc)
    assert_attention_close(got, oracle_decode_fp8(case, kc, vc), torch.bfloat16, str(env))


@pytest.mark.parametrize("env", [{}, {"WLLM_PARTITION_TOKENS": "256"}, {"WLLM_PARTITION_TOKENS": "2048"},
                                 {"WLLM_PREFIX_GROUPS": "0"}, {"WLLM_SEPARATE_COMBINE": "1"}])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_fp8_decode_with_shared_prefix_blocks(env, dtype, monkeypatch):
    # groups of 8 sequences share 64 blocks (1024 tokens); the last group is
    # ragged (5 members) and one member ends inside the shared prefix's partition
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    rng = np.random.default_rng(8)
    lens = 1024 + rng.integers(1, 3000, size=29)
    lens[9] = 1024
    case = custom_case("fp8_prefix", lens=lens, num_q_heads=28, num_kv_heads=4, head_dim=128, block_size=16,
                       dtype=dtype, seed=88, groups=(8, 64), append="none")
    kc, vc = fp8_pools(case)
    got = gpu_decode_fp8(case, kc, vc, 0.3, 0.7)
    assert_attention_close(got, oracle_decode_fp8(case, kc, vc, 0.3, 0.7), dtype, f"shared prefixes {env}")


def test_fp8_scales_enter_as_binary32_factors():
    # the same codes read with other scales: the output moves as the oracle says
    case = custom_case("fp8_scales", lens=[700, 1, 2000], num_q_heads=8, num_kv_heads=2, head_dim=128,
                       block_size=16, dtype=torch.float16, seed=5, append="none")
    kc, vc = fp8_pools(case, amp=1.0)
    for ks, vs in [(1.0, 1.0), (0.37, 3.1), (2.0 ** -6, 0.75)]:
        got = gpu_decode_fp8(case, kc, vc, ks, vs)
        assert_attention_close(got, oracle_decode_fp8(case, kc, vc, ks, vs), torch.float16, f"{ks},{vs}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_fp8_decode_step_fused(dtype):
    rng = np.random.default_rng(9)
    lens = rng.integers(1, 5000, size=33)
    case = custom_case("fp8_step", lens=lens, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                       dtype=dtype, seed=99, append="tail")
    kc, vc = fp8_pools(case)
    dev = "cuda"
    kd, vd = kc.cuda(), vc.cuda()
    q = case.q.cuda()
    out = torch.empty_like(q)
    ks, vs = 0.21, 0.27
    wllm.decode_step_fp8(out, q, case.key.cuda(), case.value.cuda(), kd, vd, case.slot_mapping.cuda(),
                         case.block_tables.cuda(), case.context_lens.cuda(), case.num_kv_heads, case.scale, ks, vs,
                         case.block_size)
    torch.cuda.synchronize()
    oracle.reshape_and_cache_e4m3(case.key, case.value, kc, vc, case.slot_mapping, ks, vs)
    assert torch.equal(kd.cpu(), kc) and torch.equal(vd.cpu(), vc)
    ref = oracle_decode_fp8(case, kc, vc, ks, vs)
    assert_attention_close(out.to(dev).cpu(), ref, dtype, "fused fp8 step")


def test_fp8_fused_steps_of_different_grid_sizes():
    """fp8 fused steps whose launches have very different grids (2 CTAs, then
    a full persistent grid), alternated with a 16-bit one on the same device:
    the grid barrier stays consistent, every step's append is bit-exact and
    its decode matches the oracle, with no error reported."""
    ks, vs = 0.23, 0.29
    small = custom_case("fp8_grid_small", lens=[37, 16], num_q_heads=8, num_kv_heads=1, head_dim=128,
                        block_size=16, dtype=torch.bfloat16, seed=61, append="tail")
    rng = np.random.default_rng(62)
    big = custom_case("fp8_grid_big", lens=rng.integers(200, 3000, 96).tolist(), num_q_heads=28, num_kv_heads=4,
                      head_dim=128, block_size=16, dtype=torch.bfloat16, seed=63, append="tail")
    refs = {}
    for c in (small, big):
        kc, vc = fp8_pools(c)
        oracle.reshape_and_cache_e4m3(c.key, c.value, kc, vc, c.slot_mapping, ks, vs)
        refs[c.name] = (kc, vc, oracle_decode_fp8(c, kc, vc, ks, vs))
    b16 = custom_case("b16_grid", lens=[5, 900], num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                      dtype=torch.float16, seed=64)
    assert wllm.device_errors() == 0
    for case in (small, big, b16, small, big, big, small):
        q = case.q.cuda()
        out = torch.empty_like(q)
        if case is b16:
            kd, vd = case.pool("cuda")
            wllm.decode_step(out, q, case.key.cuda(), case.value.cuda(), kd, vd, case.slot_mapping.cuda(),
                             case.block_tables.cuda(), case.context_lens.cuda(), case.num_kv_heads, case.scale,
                             case.block_size)
            torch.cuda.synchronize()
            assert wllm.device_errors() == 0
            continue
        kd, vd = (x.cuda() for x in fp8_pools(case))
        wllm.decode_step_fp8(out, q, case.key.cuda(), case.value.cuda(), kd, vd, case.slot_mapping.cuda(),
                             case.block_tables.cuda(), case.context_lens.cuda(), case.num_kv_heads, case.scale, ks,
                             vs, case.block_size)
        torch.cuda.synchronize()
        kr, vr, ref = refs[case.name]
        assert torch.equal(kd.cpu(), kr) and torch.equal(vd.cpu(), vr), f"{case.name}: append not bit-exact"
        assert_attention_close(out.cpu(), ref, case.dtype, f"{case.name} after a launch of another grid size")
        assert wllm.device_errors() == 0


def test_fp8_rejects_unsupported_shapes():
    case = custom_case("fp8_d64", lens=[10], num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=8,
                       dtype=torch.float16, seed=1, append="none")
    kc, vc = fp8_pools(case)
    with pytest.raises(wllm.WllmError):
        gpu_decode_fp8(case, kc, vc)


# --------------------------------------------------------------------------
# the Llama-2-7B-shaped workload at full size, sampled rows
# --------------------------------------------------------------------------

def test_fp8_full_size_llama2_7b_sampled():
    case = make_case("c2")
    kc, vc, bt, _ = case.compact()
    kc, vc = e4m3_codes(kc, AMP), e4m3_codes(vc, AMP)
    dev = "cuda"
    q = case.q.to(dev)
    out = torch.empty_like(q)
    wllm.paged_attention_decode_fp8(out, q, kc.to(dev), vc.to(dev), bt.to(dev), case.context_lens.to(dev),
                                    case.num_kv_heads, case.scale, K_SCALE, V_SCALE, case.block_size)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(case.num_seqs * case.num_q_heads, size=96, replace=False))
    ref = oracle.paged_decode(case.q, kc, vc, bt, case.context_lens, case.num_kv_heads, case.scale,
                              rows=torch.from_numpy(rows), k_scale=K_SCALE, v_scale=V_SCALE)
    got = out.cpu().reshape(-1, case.head_dim)[torch.from_numpy(rows)]
    assert_attention_close(got, ref, case.dtype, "c2 fp8 sampled")


def test_fp8_head_dim_64_step_with_shared_prefixes():
    # TinyLlama-shaped heads (32/4, D 64) over an fp8 cache: the fused step, groups of 8 sharing 16 blocks
    rng = np.random.default_rng(12)
    lens = 256 + rng.integers(1, 1800, size=21)
    case = custom_case("fp8_d64_step", lens=lens, num_q_heads=32, num_kv_heads=4, head_dim=64, block_size=16,
                       dtype=torch.float16, seed=121, groups=(8, 16), append="tail")
    kc, vc = fp8_pools(case)
    kd, vd = kc.cuda(), vc.cuda()
    q = case.q.cuda()
    out = torch.empty_like(q)
    wllm.decode_step_fp8(out, q, case.key.cuda(), case.value.cuda(), kd, vd, case.slot_mapping.cuda(),
                         case.block_tables.cuda(), case.context_lens.cuda(), case.num_kv_heads, case.scale, 0.2, 0.3,
                         case.block_size)
    torch.cuda.synchronize()
    oracle.reshape_and_cache_e4m3(case.key, case.value, kc, vc, case.slot_mapping, 0.2, 0.3)
    assert torch.equal(kd.cpu(), kc) and torch.equal(vd.cpu(), vc)
    assert_attention_close(out.cpu(), oracle_decode_fp8(case, kc, vc, 0.2, 0.3), torch.float16, "fp8 D64 step")


# --------------------------------------------------------------------------
# the Qwen2.5-shaped prefix batch and the long-context batch at full size,
# through the fused step the benchmark times
# --------------------------------------------------------------------------

def _fp8_fused_full_size(name, rows=None):
    """decode_step_fp8 over E4M3 codes of the workload's referenced blocks (the
    compact pool: the same tokens and sharing, renumbered), against the
    oracle's E4M3 append and its attention over the dequantised codes."""
    case = make_case(name)
    kc, vc, bt, slots = case.compact()
    kc, vc = e4m3_codes(kc, AMP), e4m3_codes(vc, AMP)
    kd, vd = kc.cuda(), vc.cuda()
    q = case.q.cuda()
    out = torch.full_like(q, float("nan"))
    wllm.decode_step_fp8(out, q, case.key.cuda(), case.value.cuda(), kd, vd, slots.cuda(), bt.cuda(),
                         case.context_lens.cuda(), case.num_kv_heads, case.scale, K_SCALE, V_SCALE, case.block_size)
    torch.cuda.synchronize()
    oracle.reshape_and_cache_e4m3(case.key, case.value, kc, vc, slots, K_SCALE, V_SCALE)
    assert torch.equal(kd.cpu(), kc) and torch.equal(vd.cpu(), vc), "E4M3 append not bit-exact"
    del kd, vd
    ref = oracle.paged_decode(case.q, kc, vc, bt, case.context_lens, case.num_kv_heads, case.scale,
                              rows=rows, k_scale=K_SCALE, v_scale=V_SCALE)
    got = out.cpu()
    assert torch.isfinite(got).all(), "every row written"
    if rows is not None:
        got = got.reshape(-1, case.head_dim)[rows]
    return got, ref, case


def test_fp8_full_size_qwen25_prefix_step():
    """256 sequences in groups of 8 sharing a 1024-token prompt: prefix-group
    units over E4M3 codes, every row."""
    got, ref, case = _fp8_fused_full_size("c3")
    assert_attention_close(got, ref, case.dtype, "c3 fp8 fused step")


def test_fp8_full_size_long_context_step_sampled():
    """32K-128K tokens per sequence, up to 128 partitions merged per sequence,
    1% keys x8: sampled rows."""
    case = make_case("c4")
    B, Hq = case.num_seqs, case.num_q_heads
    g = torch.Generator().manual_seed(45)
    rows = torch.tensor(sorted(set(torch.randint(0, B * Hq, (40,), generator=g).tolist()) |
                               {b * Hq + (b * 7 + 2) % Hq for b in range(B)}))
    got, ref, case = _fp8_fused_full_size("c4", rows=rows)
    assert_attention_close(got, ref, case.dtype, "c4 fp8 fused step, sampled rows")
