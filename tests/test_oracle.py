"""Pins for the fp64 CPU oracle: each test ties it to something other than itself.

* 16-bit decoding: every f16 / bf16 bit pattern against numpy / torch.
* Dense equivalence ("mini-vLLM" README, "Results / Correctness": paged attention
  equals dense attention over scattered blocks, grouped-query heads and
  non-power-of-two tables included): torch's float64 scaled_dot_product_attention
  on the dense tokens, with K/V heads expanded by repeat_interleave (the
  grouped-query order "query head h reads KV head h // G").
* Closed forms: one token, equal keys, two tokens (logistic form), one dominant
  key (fails without the max subtraction), empty sequence.
* Invariants: physical block permutation, block-size re-layout and sequence
  permutation leave the result bitwise unchanged.
* Brute force: pure-Python loops with math.fsum on the tiny workload.
* Append: gather-by-slot returns the input bits; nothing else changes.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_185_gb300 import workloads
from tests.paged_helpers import paged_from_dense

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


# --------------------------------------------------------------------------
# element decoding
# --------------------------------------------------------------------------

def test_widen_every_f16_pattern():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.widen(torch.from_numpy(bits.view(np.int16).copy()).view(torch.float16)).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    # sign of zero kept
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_widen_every_bf16_pattern():
    bits = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16)
    ref = x.to(torch.float64).numpy()
    got = oracle.widen(x).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()


def test_widen_f32_identity():
    x = torch.randn(1000, dtype=torch.float32)
    assert torch.equal(oracle.widen(x), x.to(torch.float64))


# --------------------------------------------------------------------------
# dense equivalence
# --------------------------------------------------------------------------

def _dense_sdpa(q, dense_k, dense_v, scale):
    """Library reference: float64 SDPA per sequence, K/V heads repeated per group."""
    B, Hq, D = q.shape
    outs = []
    for i in range(B):
        k = dense_k[i].to(torch.float64).transpose(0, 1)  # [Hkv, L, D]
        v = dense_v[i].to(torch.float64).transpose(0, 1)
        G = Hq // k.shape[0]
        k = k.repeat_interleave(G, dim=0)
        v = v.repeat_interleave(G, dim=0)
        qi = q[i].to(torch.float64).unsqueeze(1)          # [Hq, 1, D]
        if k.shape[1] == 0:
            outs.append(torch.zeros(Hq, D, dtype=torch.float64))
            continue
        o = F.scaled_dot_product_attention(qi.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0),
                                           scale=float(np.float32(scale)))
        outs.append(o[0, :, 0, :])
    return torch.stack(outs)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("Hq,Hkv,D,bs", [
    (4, 2, 64, 16), (8, 8, 64, 8), (28, 4, 128, 16), (7, 1, 32, 32), (6, 3, 256, 8), (32, 8, 128, 16)])
def test_matches_dense_sdpa(dtype, Hq, Hkv, D, bs):
    gen = torch.Generator().manual_seed(Hq * 1000 + D + bs)
    lens = [1, 5, bs, bs + 1, 3 * bs - 1, 70]
    dense_k = [torch.randn(L, Hkv, D, generator=gen).to(dtype) for L in lens]
    dense_v = [torch.randn(L, Hkv, D, generator=gen).to(dtype) for L in lens]
    q = torch.randn(len(lens), Hq, D, generator=gen).to(dtype)
    scale = float(np.float32(1 / math.sqrt(D)))
    nb = sum((L + bs - 1) // bs for L in lens) + 5
    kp, vp, bt = paged_from_dense(dense_k, dense_v, bs, nb, gen, pad_blocks=2)
    cl = torch.tensor(lens, dtype=torch.int32)
    got = oracle.paged_decode(q, kp, vp, bt, cl, Hkv, scale)
    ref = _dense_sdpa(q, dense_k, dense_v, scale)
    assert not torch.isnan(got).any()
    torch.testing.assert_close(got, ref, rtol=1e-12, atol=1e-12)


def test_gqa_mapping_is_contiguous_groups():
    """Query head h must read KV head h // G, not h % G (HF repeat_kv order)."""
    gen = torch.Generator().manual_seed(5)
    Hq, Hkv, D, bs, L = 8, 2, 16, 4, 9
    k = [torch.randn(L, Hkv, D, generator=gen)]
    v = [torch.zeros(L, Hkv, D)]
    v[0][:, 0, :] = 1.0   # KV head 0 -> all ones
    v[0][:, 1, :] = -1.0  # KV head 1 -> all minus ones
    q = torch.randn(1, Hq, D, generator=gen)
    kp, vp, bt = paged_from_dense(k, v, bs, 6, gen)
    out = oracle.paged_decode(q, kp, vp, bt, torch.tensor([L], dtype=torch.int32), Hkv, 0.25)
    expect = torch.tensor([1.0] * 4 + [-1.0] * 4, dtype=torch.float64)
    assert torch.equal(out[0, :, 0], expect)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def _single_seq(k, v, q, bs=4, scale=0.125):
    gen = torch.Generator().manual_seed(0)
    L = k.shape[0]
    nb = (L + bs - 1) // bs + 3
    kp, vp, bt = paged_from_dense([k], [v], bs, nb, gen)
    return oracle.paged_decode(q, kp, vp, bt, torch.tensor([L], dtype=torch.int32),
                               k.shape[1], scale)


def test_one_token_returns_its_value_exactly():
    gen = torch.Generator().manual_seed(1)
    for dtype in (torch.float32, torch.float16, torch.bfloat16):
        k = torch.randn(1, 2, 64, generator=gen).to(dtype)
        v = torch.randn(1, 2, 64, generator=gen).to(dtype)
        q = torch.randn(1, 4, 64, generator=gen).to(dtype)
        out = _single_seq(k, v, q)
        expect = v[0].to(torch.float64).repeat_interleave(2, dim=0)
        assert torch.equal(out[0], expect)


def test_equal_keys_give_mean_of_values():
    gen = torch.Generator().manual_seed(2)
    L, D = 37, 32
    k = torch.randn(1, 1, D, generator=gen).expand(L, 1, D).contiguous()
    v = torch.randn(L, 1, D, generator=gen)
    q = torch.randn(1, 3, D, generator=gen)
    out = _single_seq(k, v, q)
    mean = torch.tensor([math.fsum(v[:, 0, d].double().tolist()) / L for d in range(D)],
                        dtype=torch.float64)
    for h in range(3):
        torch.testing.assert_close(out[0, h], mean, rtol=0, atol=1e-14)


def test_two_tokens_logistic_form():
    gen = torch.Generator().manual_seed(3)
    D, scale = 16, 0.3
    k = torch.randn(2, 1, D, generator=gen)
    v = torch.randn(2, 1, D, generator=gen)
    q = torch.randn(1, 1, D, generator=gen)
    out = _single_seq(k, v, q, scale=scale)
    sc = float(np.float32(scale))
    s0 = sc * math.fsum(float(a) * float(b) for a, b in zip(q[0, 0], k[0, 0]))
    s1 = sc * math.fsum(float(a) * float(b) for a, b in zip(q[0, 0], k[1, 0]))
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    expect = torch.tensor([w0 * float(v[0, 0, d]) + w1 * float(v[1, 0, d]) for d in range(D)],
                          dtype=torch.float64)
    torch.testing.assert_close(out[0, 0], expect, rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value():
    """Scores near 1e4: exp overflows unless the running max is subtracted."""
    gen = torch.Generator().manual_seed(4)
    L, D = 50, 64
    q = torch.randn(1, 1, D, generator=gen)
    k = torch.randn(L, 1, D, generator=gen)
    k[17, 0] = q[0, 0] * 2000.0
    v = torch.randn(L, 1, D, generator=gen)
    out = _single_seq(k, v, q, scale=1.0)
    assert torch.equal(out[0, 0], v[17, 0].double())


def test_empty_sequence_gives_zeros():
    gen = torch.Generator().manual_seed(6)
    dense = [torch.randn(5, 2, 8, generator=gen), torch.randn(0, 2, 8)]
    kp, vp, bt = paged_from_dense(dense, dense, 4, 4, gen, pad_blocks=1)
    q = torch.randn(2, 2, 8, generator=gen)
    out = oracle.paged_decode(q, kp, vp, bt, torch.tensor([5, 0], dtype=torch.int32), 2, 0.5)
    assert torch.equal(out[1], torch.zeros(2, 8, dtype=torch.float64))
    assert not torch.isnan(out).any()


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

def _case_pool(case):
    kc, vc = case.pool()
    oracle.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping)
    return kc, vc


def test_block_permutation_invariance():
    case = workloads.custom_case("perm", lens=[3, 40, 17, 64, 1], num_q_heads=6, num_kv_heads=2,
                                 head_dim=32, block_size=8, dtype=torch.bfloat16, seed=11,
                                 spare_blocks=7)
    kc, vc = _case_pool(case)
    ref = oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, 2, case.scale)
    perm = torch.randperm(case.num_blocks, generator=torch.Generator().manual_seed(9))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(case.num_blocks)
    # new physical block inv[p] holds what old block p held
    kc2, vc2 = kc[perm], vc[perm]
    bt2 = torch.where(case.block_tables >= 0, inv[case.block_tables.clamp(min=0).long()].int(),
                      case.block_tables)
    got = oracle.paged_decode(case.q, kc2, vc2, bt2, case.context_lens, 2, case.scale)
    assert torch.equal(got, ref)


@pytest.mark.parametrize("bs2", [4, 16, 32])
def test_block_size_relayout_invariance(bs2):
    gen = torch.Generator().manual_seed(12)
    lens = [1, 9, 31, 64, 100]
    dk = [torch.randn(L, 2, 64, generator=gen).to(torch.float16) for L in lens]
    dv = [torch.randn(L, 2, 64, generator=gen).to(torch.float16) for L in lens]
    q = torch.randn(5, 8, 64, generator=gen).to(torch.float16)
    cl = torch.tensor(lens, dtype=torch.int32)
    kp, vp, bt = paged_from_dense(dk, dv, 8, 40, gen)
    ref = oracle.paged_decode(q, kp, vp, bt, cl, 2, 0.125)
    nb2 = sum((L + bs2 - 1) // bs2 for L in lens) + 3
    kp2, vp2, bt2 = paged_from_dense(dk, dv, bs2, nb2, gen, pad_blocks=1)
    got = oracle.paged_decode(q, kp2, vp2, bt2, cl, 2, 0.125)
    assert torch.equal(got, ref)


def test_sequence_permutation_permutes_outputs():
    case = workloads.make_case("c0")
    kc, vc = _case_pool(case)
    ref = oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, 2, case.scale)
    p = torch.tensor([2, 0, 3, 1])
    got = oracle.paged_decode(case.q[p], kc, vc, case.block_tables[p], case.context_lens[p],
                              2, case.scale)
    assert torch.equal(got, ref[p])


def test_row_subset_equals_full():
    case = workloads.make_case("c0")
    kc, vc = _case_pool(case)
    full = oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, 2, case.scale)
    rows = [15, 0, 6, 9]
    sub = oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, 2,
                              case.scale, rows=rows)
    flat = full.reshape(-1, full.shape[-1])
    assert torch.equal(sub, flat[rows])


# --------------------------------------------------------------------------
# brute force on the tiny workload
# --------------------------------------------------------------------------

def _brute_force(case, kc, vc):
    """Pure-Python loops: gather token j via the table, fsum dot products."""
    B, Hq, D = case.q.shape
    G = case.group
    bs = case.block_size
    qf = case.q.double().tolist()
    kf = kc.double().tolist()
    vf = vc.double().tolist()
    sc = float(np.float32(case.scale))
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        L = int(case.context_lens[b])
        for h in range(Hq):
            c = h // G
            toks = []
            for j in range(L):
                pb = int(case.block_tables[b, j // bs])
                toks.append((kf[pb][c][j % bs], vf[pb][c][j % bs]))
            s = [sc * math.fsum(qf[b][h][d] * kk[d] for d in range(D)) for kk, _ in toks]
            m = max(s)
            w = [math.exp(x - m) for x in s]
            den = math.fsum(w)
            for d in range(D):
                out[b][h][d] = math.fsum(w[j] * toks[j][1][d] for j in range(L)) / den
    return torch.tensor(out, dtype=torch.float64)


def test_brute_force_tiny_workload():
    case = workloads.make_case("c0")
    kc, vc = _case_pool(case)
    got = oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, 2, case.scale)
    ref = _brute_force(case, kc, vc)
    torch.testing.assert_close(got, ref, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# KV append
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_append_gather_returns_input_and_touches_nothing_else(dtype):
    gen = torch.Generator().manual_seed(21)
    N_b, Hkv, bs, D, T = 12, 3, 8, 32, 20
    kc = torch.randn(N_b, Hkv, bs, D, generator=gen).to(dtype)
    vc = torch.randn(N_b, Hkv, bs, D, generator=gen).to(dtype)
    key = torch.randn(T, Hkv, D, generator=gen).to(dtype)
    val = torch.randn(T, Hkv, D, generator=gen).to(dtype)
    slots = torch.randperm(N_b * bs, generator=gen)[:T].long()
    slots[3] = -1
    slots[11] = -7
    kc0, vc0 = kc.clone(), vc.clone()
    oracle.reshape_and_cache(key, val, kc, vc, slots)
    # gather back through the slots
    flat_k = kc.view(torch.int16 if dtype != torch.float32 else torch.int32) \
        .permute(0, 2, 1, 3).reshape(N_b * bs, Hkv, D)
    flat_v = vc.view(torch.int16 if dtype != torch.float32 else torch.int32) \
        .permute(0, 2, 1, 3).reshape(N_b * bs, Hkv, D)
    itype = torch.int16 if dtype != torch.float32 else torch.int32
    ok = slots >= 0
    assert torch.equal(flat_k[slots[ok]], key.view(itype)[ok])
    assert torch.equal(flat_v[slots[ok]], val.view(itype)[ok])
    # everything else bit-identical
    touched = torch.zeros(N_b * bs, dtype=torch.bool)
    touched[slots[ok]] = True
    f0k = kc0.view(itype).permute(0, 2, 1, 3).reshape(N_b * bs, Hkv, D)
    f0v = vc0.view(itype).permute(0, 2, 1, 3).reshape(N_b * bs, Hkv, D)
    assert torch.equal(flat_k[~touched], f0k[~touched])
    assert torch.equal(flat_v[~touched], f0v[~touched])


def test_append_copies_nan_bits_unchanged():
    key = torch.tensor([0x7FC1, 0x7C00, 0xFC00, 0x8000], dtype=torch.int32).to(torch.int16) \
        .view(torch.float16).reshape(1, 1, 4)
    kc = torch.zeros(2, 1, 2, 4, dtype=torch.float16)
    vc = torch.zeros_like(kc)
    oracle.reshape_and_cache(key, key, kc, vc, torch.tensor([3]))
    assert torch.equal(kc[1, 0, 1].view(torch.int16), key[0, 0].view(torch.int16))


def test_append_out_of_range_slot_writes_nothing():
    kc = torch.zeros(2, 1, 2, 4)
    vc = torch.zeros_like(kc)
    key = torch.ones(2, 1, 4)
    with pytest.raises(oracle.OracleError):
        oracle.reshape_and_cache(key, key, kc, vc, torch.tensor([0, 4]))
    assert torch.equal(kc, torch.zeros_like(kc))


def test_decode_rejects_bad_tables():
    kc = torch.zeros(2, 1, 2, 4)
    q = torch.zeros(1, 1, 4)
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(q, kc, kc, torch.tensor([[0, 2]], dtype=torch.int32),
                            torch.tensor([4], dtype=torch.int32), 1, 1.0)
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(q, kc, kc, torch.tensor([[0, 1]], dtype=torch.int32),
                            torch.tensor([5], dtype=torch.int32), 1, 1.0)


# --------------------------------------------------------------------------
# FP8 (E4M3) KV cache: codes, the scaled append, attention over scaled codes
# --------------------------------------------------------------------------

def test_e4m3_decode_every_code_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    got = oracle.widen_e4m3(codes)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64)
    assert ((got == ref) | (got.isnan() & ref.isnan())).all()
    assert got[0x7E] == 448 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_e4m3_encode_rounds_like_torch_in_range():
    gen = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(200000, generator=gen) * s for s in (1e-3, 1.0, 30.0, 200.0)])
    # every midpoint between neighbouring finite codes (ties go to the even code)
    v = oracle.widen_e4m3(torch.arange(0x7F, dtype=torch.uint8))
    mids = ((v[1:] + v[:-1]) / 2).to(torch.float32)
    x = torch.cat([x, mids, -mids])
    keep = x.abs() < 464  # torch turns larger magnitudes into NaN, E4M3 here saturates
    got = oracle.e4m3_encode(x[keep])
    ref = x[keep].to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(got, ref)


def test_e4m3_encode_saturates_and_keeps_nan():
    x = torch.tensor([448.0, 463.9, 464.0, 1e6, -1e6, float("inf"), float("-inf"), float("nan"), -0.0])
    got = oracle.e4m3_encode(x).tolist()
    assert got[:7] == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE]
    assert got[7] & 0x7F == 0x7F and got[8] == 0x80


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_e4m3_append_stores_scaled_codes(dtype):
    gen = torch.Generator().manual_seed(9)
    T, Hkv, D, nb, bs = 7, 2, 64, 6, 8
    key = (torch.randn(T, Hkv, D, generator=gen) * 3).to(dtype)
    value = (torch.randn(T, Hkv, D, generator=gen) * 3).to(dtype)
    kc = torch.full((nb, Hkv, bs, D), 0x55, dtype=torch.uint8)
    vc = kc.clone()
    slots = torch.tensor([3, 17, -1, 40, 0, 47, 9], dtype=torch.int64)
    ks, vs = 0.0371, 2.5
    oracle.reshape_and_cache_e4m3(key, value, kc, vc, slots, ks, vs)
    inv_k = torch.tensor(oracle.inv_scale(ks), dtype=torch.float32)
    inv_v = torch.tensor(oracle.inv_scale(vs), dtype=torch.float32)
    for t, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        yk = key[t].to(torch.float32) * inv_k
        yv = value[t].to(torch.float32) * inv_v
        assert (yk.abs() < 464).all() and (yv.abs() < 464).all()
        assert torch.equal(kc[s // bs, :, s % bs], yk.to(torch.float8_e4m3fn).view(torch.uint8))
        assert torch.equal(vc[s // bs, :, s % bs], yv.to(torch.float8_e4m3fn).view(torch.uint8))
    written = {(s // bs, s % bs) for s in slots.tolist() if s >= 0}
    for b in range(nb):
        for o in range(bs):
            if (b, o) not in written:
                assert (kc[b, :, o] == 0x55).all() and (vc[b, :, o] == 0x55).all()


@pytest.mark.parametrize("qdtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("Hq,Hkv,D,bs", [(8, 2, 128, 16), (32, 32, 128, 16), (28, 4, 256, 8)])
def test_e4m3_decode_matches_dense_sdpa_on_scaled_codes(qdtype, Hq, Hkv, D, bs):
    gen = torch.Generator().manual_seed(Hq + D + bs)
    lens = [1, 9, bs, 3 * bs + 2, 50]
    dk = [torch.randn(L, Hkv, D, generator=gen).to(torch.float8_e4m3fn) for L in lens]
    dv = [torch.randn(L, Hkv, D, generator=gen).to(torch.float8_e4m3fn) for L in lens]
    q = torch.randn(len(lens), Hq, D, generator=gen).to(qdtype)
    ks, vs, scale = 0.731, 1.0 / 3.0, float(np.float32(1 / math.sqrt(D)))
    nb = sum((L + bs - 1) // bs for L in lens) + 3
    kp, vp, bt = paged_from_dense(dk, dv, bs, nb, gen, pad_blocks=1)
    got = oracle.paged_decode(q, kp.view(torch.uint8), vp.view(torch.uint8), bt,
                              torch.tensor(lens, dtype=torch.int32), Hkv, scale, k_scale=ks, v_scale=vs)
    k64 = [k.to(torch.float64) * float(np.float32(ks)) for k in dk]
    v64 = [v.to(torch.float64) * float(np.float32(vs)) for v in dv]
    ref = _dense_sdpa(q, k64, v64, scale)
    torch.testing.assert_close(got, ref, rtol=1e-12, atol=1e-12)


def test_e4m3_one_token_returns_scaled_value_exactly():
    v = torch.tensor([[[0.5, -3.0, 448.0, 2.0 ** -9]]]).to(torch.float8_e4m3fn)  # [1 token, 1 head, 4]
    k = torch.ones(1, 1, 4).to(torch.float8_e4m3fn)
    kp, vp, bt = paged_from_dense([k], [v], 4, 2, torch.Generator().manual_seed(0))
    q = torch.ones(1, 2, 4, dtype=torch.float16)
    got = oracle.paged_decode(q, kp.view(torch.uint8), vp.view(torch.uint8), bt, torch.tensor([1], dtype=torch.int32),
                              1, 0.5, k_scale=3.0, v_scale=0.1)
    vs = float(np.float32(0.1))
    assert got[0, 0].tolist() == [0.5 * vs, -3.0 * vs, 448.0 * vs, 2.0 ** -9 * vs]
