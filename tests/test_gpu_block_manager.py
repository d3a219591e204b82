"""The block manager's tables driving the GPU path: prompts with shared
prefixes are registered (shared full blocks hold K/V written once), decode
steps append through the manager (copy-on-write included), and the attention
read through the manager's tables must equal the oracle's attention over each
sequence's own tokens laid out densely -- a mapping that pointed a sequence at
the wrong blocks would read other tokens' K/V and fail."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_185_gb300 as wllm
from tests.gpu_common import assert_attention_close

pytestmark = pytest.mark.gpu

BS, HQ, HKV, D, VOCAB, MAXPOS = 16, 8, 2, 64, 50, 512


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    wllm.load_library()
    yield


def kv_rows(tokens, positions, emb):
    """K and V rows [T, Hkv, D] of tokens at positions (depend on both only)."""
    ek, ev, pk, pv = emb
    t = torch.as_tensor(tokens, dtype=torch.long)
    p = torch.as_tensor(positions, dtype=torch.long)
    return (ek[t] + pk[p]).half(), (ev[t] + pv[p]).half()


def dense_reference(seqs, q, emb):
    """Oracle attention over each sequence's own tokens in a private dense layout."""
    B = len(seqs)
    lens = [len(s) for s in seqs]
    mb = max((n + BS - 1) // BS for n in lens)
    kc = torch.zeros(B * mb, HKV, BS, D, dtype=torch.float16)
    vc = torch.zeros_like(kc)
    bt = torch.full((B, mb), -1, dtype=torch.int32)
    for i, toks in enumerate(seqs):
        k, v = kv_rows(toks, range(len(toks)), emb)
        for t in range(len(toks)):
            kc[i * mb + t // BS, :, t % BS] = k[t]
            vc[i * mb + t // BS, :, t % BS] = v[t]
        bt[i, :(len(toks) + BS - 1) // BS] = torch.arange(i * mb, i * mb + (len(toks) + BS - 1) // BS)
    return oracle.paged_decode(q, kc, vc, bt, torch.tensor(lens, dtype=torch.int32), HKV, 0.125)


def test_block_manager_tables_drive_decode():
    g = torch.Generator().manual_seed(11)
    emb = (torch.randn(VOCAB, HKV, D, generator=g), torch.randn(VOCAB, HKV, D, generator=g),
           0.5 * torch.randn(MAXPOS, HKV, D, generator=g), 0.5 * torch.randn(MAXPOS, HKV, D, generator=g))
    nb = 256
    bm = wllm.BlockManager(nb, BS)
    kc = torch.zeros(nb, HKV, BS, D, dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    rng = np.random.default_rng(5)
    prefixes = [list(rng.integers(0, VOCAB, 40)) for _ in range(3)]
    seqs = []
    for i in range(12):
        toks = prefixes[i % 3] + list(rng.integers(0, VOCAB, int(rng.integers(1, 60))))
        slots, cached = bm.add_sequence(i, toks)
        if i >= 3:
            assert cached == 32, "two full prefix blocks should be shared"
        k, v = kv_rows(toks[cached:], range(cached, len(toks)), emb)
        wllm.reshape_and_cache(k.cuda(), v.cuda(), kc, vc, slots[cached:].cuda())
        seqs.append(list(toks))
    bm.fork(1, 12)  # a second sample of prompt 1 (41 tokens): shares its partial last block
    seqs.append(list(seqs[1]))
    B = len(seqs)
    mb = 16
    copies = 0
    for step in range(3):
        new = [int(rng.integers(0, VOCAB)) for _ in range(B)]
        slot_map = []
        for i in range(B):
            slot, copy = bm.append_token(i, new[i])
            if copy is not None:  # copy-on-write: the caller copies the filled slots
                src, dst = copy
                n = len(seqs[i]) % BS
                kc[dst, :, :n] = kc[src, :, :n]
                vc[dst, :, :n] = vc[src, :, :n]
                copies += 1
            slot_map.append(slot)
            seqs[i].append(new[i])
        k, v = kv_rows(new, [len(s) - 1 for s in seqs], emb)
        rows = [bm.block_table(i, mb) for i in range(B)]
        bt = torch.stack([r for r, _ in rows]).cuda()
        cl = torch.tensor([n for _, n in rows], dtype=torch.int32).cuda()
        q = torch.randn(B, HQ, D, generator=g).half()
        out = torch.empty(B, HQ, D, dtype=torch.float16, device="cuda")
        wllm.decode_step(out, q.cuda(), k.cuda(), v.cuda(), kc, vc, torch.tensor(slot_map).cuda(), bt, cl, HKV,
                         0.125, BS)
        torch.cuda.synchronize()
        ref = dense_reference(seqs, q, emb)
        assert_attention_close(out.cpu(), ref, torch.float16, f"block manager step {step}")
    assert copies >= 1, "the fork should have needed a copy-on-write"
    assert wllm.device_errors() == 0
