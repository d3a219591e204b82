"""Pins of the oracle's chunked-prefill paged attention against things other
than itself: torch float64 SDPA with the causal offset mask on the dense
tokens, closed forms, invariances of causal attention, and a brute force."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tests.paged_helpers import paged_from_dense


def _setup(lens, chunks, Hq, Hkv, D, bs, dtype, seed, pad_blocks=1):
    """Dense K/V per sequence, the paged pools, and the packed query chunks."""
    gen = torch.Generator().manual_seed(seed)
    dk = [torch.randn(L, Hkv, D, generator=gen).to(dtype) for L in lens]
    dv = [torch.randn(L, Hkv, D, generator=gen).to(dtype) for L in lens]
    nb = sum((L + bs - 1) // bs for L in lens) + 3
    kp, vp, bt = paged_from_dense(dk, dv, bs, nb, gen, pad_blocks=pad_blocks)
    T = sum(chunks)
    q = torch.randn(T, Hq, D, generator=gen).to(dtype)
    qsl = torch.tensor(np.concatenate([[0], np.cumsum(chunks)]), dtype=torch.int32)
    return dk, dv, kp, vp, bt, q, qsl


def _dense_causal_sdpa(q, qsl, dk, dv, lens, scale):
    """torch float64 SDPA per sequence; chunk token i (position L-n+i) sees keys 0..L-n+i."""
    T, Hq, D = q.shape
    out = torch.empty(T, Hq, D, dtype=torch.float64)
    for b, L in enumerate(lens):
        s0, s1 = int(qsl[b]), int(qsl[b + 1])
        n = s1 - s0
        if n == 0:
            continue
        k = dk[b].to(torch.float64).transpose(0, 1)  # [Hkv, L, D]
        v = dv[b].to(torch.float64).transpose(0, 1)
        G = Hq // k.shape[0]
        k, v = k.repeat_interleave(G, 0), v.repeat_interleave(G, 0)
        qb = q[s0:s1].to(torch.float64).transpose(0, 1)  # [Hq, n, D]
        pos = torch.arange(L - n, L)[:, None]
        allowed = torch.arange(L)[None, :] <= pos  # [n, L]
        o = F.scaled_dot_product_attention(qb[None], k[None], v[None], attn_mask=allowed,
                                           scale=float(np.float32(scale)))
        out[s0:s1] = o[0].transpose(0, 1)
    return out


GEOMS = [(4, 4, 64), (8, 2, 128), (28, 4, 128), (12, 1, 64)]


@pytest.mark.parametrize("Hq,Hkv,D", GEOMS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("bs", [8, 16])
def test_prefill_matches_dense_causal_sdpa(Hq, Hkv, D, dtype, bs):
    # fresh prompts (n = L), continued prompts (n < L), a decode-like n = 1, an empty chunk
    lens = [37, 50, 64, 9, 21, 3]
    chunks = [37, 13, 16, 1, 0, 3]
    dk, dv, kp, vp, bt, q, qsl = _setup(lens, chunks, Hq, Hkv, D, bs, dtype, seed=Hq + D + bs)
    scale = float(np.float32(1 / math.sqrt(D)))
    got = oracle.paged_prefill(q, kp, vp, bt, torch.tensor(lens, dtype=torch.int32), qsl, Hkv, scale)
    ref = _dense_causal_sdpa(q, qsl, dk, dv, lens, scale)
    torch.testing.assert_close(got, ref, rtol=1e-12, atol=1e-12)


def test_prefill_first_prompt_token_returns_its_value_exactly():
    lens, chunks = [20, 7], [20, 7]
    dk, dv, kp, vp, bt, q, qsl = _setup(lens, chunks, 4, 2, 64, 16, torch.float32, seed=3)
    got = oracle.paged_prefill(q, kp, vp, bt, torch.tensor(lens, dtype=torch.int32), qsl, 2, 0.125)
    for b in range(2):
        t0 = int(qsl[b])
        for h in range(4):
            assert torch.equal(got[t0, h], dv[b][0, h // 2].to(torch.float64))


def test_prefill_equal_keys_give_running_means_of_values():
    # all keys equal: chunk token at position P gets the mean of values 0..P
    L, n, Hkv, D = 40, 25, 2, 64
    gen = torch.Generator().manual_seed(4)
    k = torch.randn(1, Hkv, D, generator=gen).expand(L, Hkv, D).contiguous()
    v = torch.randn(L, Hkv, D, generator=gen)
    kp, vp, bt = paged_from_dense([k], [v], 16, 8, gen)
    q = torch.randn(n, 4, D, generator=gen)
    qsl = torch.tensor([0, n], dtype=torch.int32)
    got = oracle.paged_prefill(q, kp, vp, bt, torch.tensor([L], dtype=torch.int32), qsl, Hkv, 0.3)
    for i in range(n):
        P = L - n + i
        ref = v[: P + 1].to(torch.float64).mean(0)  # [Hkv, D]
        torch.testing.assert_close(got[i], ref.repeat_interleave(2, 0), rtol=1e-13, atol=1e-13)


def test_prefill_is_independent_of_the_chunking():
    # causal attention: a prompt processed as one chunk or as two gives the same rows
    L, Hq, Hkv, D = 70, 8, 2, 64
    dk, dv, kp, vp, bt, q, _ = _setup([L], [L], Hq, Hkv, D, 16, torch.bfloat16, seed=5)
    whole = oracle.paged_prefill(q, kp, vp, bt, torch.tensor([L], dtype=torch.int32),
                                 torch.tensor([0, L], dtype=torch.int32), Hkv, 0.1)
    for cut in (1, 29, 64, 69):
        first = oracle.paged_prefill(q[:cut], kp, vp, bt, torch.tensor([cut], dtype=torch.int32),
                                     torch.tensor([0, cut], dtype=torch.int32), Hkv, 0.1)
        second = oracle.paged_prefill(q[cut:], kp, vp, bt, torch.tensor([L], dtype=torch.int32),
                                      torch.tensor([0, L - cut], dtype=torch.int32), Hkv, 0.1)
        assert torch.equal(torch.cat([first, second]), whole)


def test_prefill_with_one_token_chunks_is_decode():
    # the decode definition pinned elsewhere (dense SDPA) is the n = 1 case
    lens = [5, 33, 17]
    dk, dv, kp, vp, bt, q, qsl = _setup(lens, [1, 1, 1], 8, 2, 64, 8, torch.float16, seed=6)
    cl = torch.tensor(lens, dtype=torch.int32)
    pre = oracle.paged_prefill(q, kp, vp, bt, cl, qsl, 2, 0.125)
    dec = oracle.paged_decode(q, kp, vp, bt, cl, 2, 0.125)
    assert torch.equal(pre, dec)


def test_prefill_block_relayout_is_bitwise_invariant():
    lens, chunks = [45, 30], [20, 30]
    dk, dv, kp, vp, bt, q, qsl = _setup(lens, chunks, 8, 4, 64, 16, torch.float32, seed=7)
    cl = torch.tensor(lens, dtype=torch.int32)
    a = oracle.paged_prefill(q, kp, vp, bt, cl, qsl, 4, 0.2)
    kp2, vp2, bt2 = paged_from_dense(dk, dv, 8, 12, torch.Generator().manual_seed(99), pad_blocks=2)
    b = oracle.paged_prefill(q, kp2, vp2, bt2, cl, qsl, 4, 0.2)
    assert torch.equal(a, b)


def test_prefill_brute_force_fsum():
    lens, chunks = [6, 4], [3, 4]
    dk, dv, kp, vp, bt, q, qsl = _setup(lens, chunks, 2, 1, 64, 8, torch.float32, seed=8)
    scale = 0.37
    got = oracle.paged_prefill(q, kp, vp, bt, torch.tensor(lens, dtype=torch.int32), qsl, 1, scale)
    s32 = float(np.float32(scale))
    for b, (L, n) in enumerate(zip(lens, chunks)):
        for i in range(n):
            t = int(qsl[b]) + i
            P = L - n + i
            for h in range(2):
                qv = [float(x) for x in q[t, h]]
                s = [s32 * math.fsum(qv[d] * float(dk[b][j, 0, d]) for d in range(64)) for j in range(P + 1)]
                m = max(s)
                w = [math.exp(x - m) for x in s]
                den = math.fsum(w)
                ref = [math.fsum(w[j] * float(dv[b][j, 0, d]) for j in range(P + 1)) / den for d in range(64)]
                assert np.allclose(got[t, h].numpy(), ref, rtol=1e-13, atol=1e-13)


def test_prefill_rows_and_validation():
    lens, chunks = [30, 12], [10, 12]
    dk, dv, kp, vp, bt, q, qsl = _setup(lens, chunks, 4, 2, 64, 16, torch.float16, seed=9)
    cl = torch.tensor(lens, dtype=torch.int32)
    full = oracle.paged_prefill(q, kp, vp, bt, cl, qsl, 2, 0.125)
    rows = [0, 5, 39, 87]
    part = oracle.paged_prefill(q, kp, vp, bt, cl, qsl, 2, 0.125, rows=rows)
    assert torch.equal(part, full.reshape(-1, 64)[rows])
    with pytest.raises(oracle.OracleError):  # chunk longer than the context
        oracle.paged_prefill(q, kp, vp, bt, torch.tensor([5, 12], dtype=torch.int32), qsl, 2, 0.125)
    with pytest.raises(oracle.OracleError):  # last start != T
        oracle.paged_prefill(q, kp, vp, bt, cl, torch.tensor([0, 10, 21], dtype=torch.int32), 2, 0.125)


@pytest.mark.parametrize("qdtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 128), (4, 4, 64)])
def test_prefill_over_e4m3_codes_matches_dense_causal_sdpa(qdtype, Hq, Hkv, D):
    lens, chunks = [40, 70, 5], [40, 22, 1]
    gen = torch.Generator().manual_seed(Hq + D)
    dk = [torch.randn(L, Hkv, D, generator=gen).to(torch.float8_e4m3fn) for L in lens]
    dv = [torch.randn(L, Hkv, D, generator=gen).to(torch.float8_e4m3fn) for L in lens]
    kp, vp, bt = paged_from_dense(dk, dv, 16, 12, gen, pad_blocks=1)
    q = torch.randn(sum(chunks), Hq, D, generator=gen).to(qdtype)
    qsl = torch.tensor(np.concatenate([[0], np.cumsum(chunks)]), dtype=torch.int32)
    ks, vs, scale = 0.61, 1.7, float(np.float32(1 / math.sqrt(D)))
    got = oracle.paged_prefill(q, kp.view(torch.uint8), vp.view(torch.uint8), bt, torch.tensor(lens, dtype=torch.int32),
                               qsl, Hkv, scale, k_scale=ks, v_scale=vs)
    k64 = [k.to(torch.float64) * float(np.float32(ks)) for k in dk]
    v64 = [v.to(torch.float64) * float(np.float32(vs)) for v in dv]
    ref = _dense_causal_sdpa(q, qsl, k64, v64, lens, scale)
    torch.testing.assert_close(got, ref, rtol=1e-12, atol=1e-12)
