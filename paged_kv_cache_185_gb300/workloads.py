"""Seeded synthetic decode-step inputs for the paged KV cache.

This module only draws inputs: it holds none of the attention or append
arithmetic, and both the CUDA path and the CPU oracle consume what it makes.

A case describes one decode step of a continuously batched engine:

* a fixed pool of ``num_blocks`` physical KV blocks, K and V each laid out
  ``[num_blocks, num_kv_heads, block_size, head_dim]``;
* per sequence a block table (int32, ``-1`` past the blocks it uses) and a
  context length (int32, the number of tokens it attends to, this step's
  token included);
* one query token per sequence ``[B, Hq, D]``;
* the step's KV append: ``key``/``value`` ``[T, Hkv, D]`` and an int64
  ``slot_mapping`` (slot = physical_block * block_size + offset).

Only the blocks some sequence references carry data (drawn once per physical
block, so blocks shared by several tables really hold the same bytes).  Every
other slot is NaN, as are the slots the append is about to fill and the slots of
a sequence's last block past its length, so that a kernel that reads anything it
should not turns its output into NaN.

Shapes follow the page workloads: TinyLlama / Llama-2 / Qwen2.5 / Gemma head
geometries, block size 16 ("mini-vLLM" README, "Configuration" table default),
ragged context lengths, shared prefix blocks ("wLLM: Native Windows LLM
Inference Server", ADR-001: prefix sharing is a block-table operation).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = ["DecodeCase", "make_case", "custom_case", "CASE_NAMES", "normal", "e4m3_codes"]


def normal(seed: int, n: int) -> np.ndarray:
    """``n`` i.i.d. N(0,1) float32 values from ``seed``.

    Drawn in fixed chunks of 2**22 values, chunk ``i`` from the i-th child of
    ``SeedSequence(seed)``, so the values do not depend on the thread count.
    """
    chunk = 1 << 22
    out = np.empty(n, np.float32)
    nchunks = max(1, (n + chunk - 1) // chunk)
    children = np.random.SeedSequence(seed).spawn(nchunks)

    def fill(i: int) -> None:
        lo, hi = i * chunk, min(n, (i + 1) * chunk)
        if hi > lo:
            g = np.random.Generator(np.random.PCG64(children[i]))
            g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])

    workers = min(nchunks, os.cpu_count() or 1)
    if workers <= 1:
        for i in range(nchunks):
            fill(i)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


@dataclass
class DecodeCase:
    name: str
    dtype: torch.dtype
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float                    # a binary32 value
    q: torch.Tensor                 # [B, Hq, D]
    context_lens: torch.Tensor      # int32 [B]
    block_tables: torch.Tensor      # int32 [B, M_b], -1 past the used blocks
    used_blocks: torch.Tensor       # int64 [n_used], physical ids holding data
    k_used: torch.Tensor            # [n_used, Hkv, bs, D]  (K of those blocks)
    v_used: torch.Tensor            # [n_used, Hkv, bs, D]
    key: torch.Tensor               # [T, Hkv, D]   this step's new K
    value: torch.Tensor             # [T, Hkv, D]   this step's new V
    slot_mapping: torch.Tensor      # int64 [T]
    meta: dict = field(default_factory=dict)

    # --- sizes -----------------------------------------------------------
    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def elt(self) -> int:
        return torch.empty((), dtype=self.dtype).element_size()

    def pool_bytes(self) -> int:
        """Bytes of one of the two (K or V) pools."""
        return self.num_blocks * self.num_kv_heads * self.block_size * self.head_dim * self.elt

    # --- materialisation ---------------------------------------------------
    def pool(self, device="cpu"):
        """Full K and V pools on ``device``: NaN everywhere but the used blocks."""
        shape = (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)
        ids = self.used_blocks.to(device)
        out = []
        for data in (self.k_used, self.v_used):
            p = torch.full(shape, float("nan"), dtype=self.dtype, device=device)
            p[ids] = data.to(device)
            out.append(p)
        return out[0], out[1]

    def compact(self):
        """(k_pool, v_pool, block_tables) holding only the used blocks.

        Same tokens, renumbered physical ids: decode over this compact pool
        reads exactly the bytes it reads over the full one.  The append slots
        are renumbered too and returned as the fourth item (-1 where a slot
        falls in a block no table uses).
        """
        ids = self.used_blocks.numpy()
        order = np.argsort(ids)
        sorted_ids = ids[order]

        def remap(phys: np.ndarray) -> np.ndarray:
            pos = np.searchsorted(sorted_ids, phys)
            pos = np.clip(pos, 0, len(sorted_ids) - 1)
            hit = sorted_ids[pos] == phys
            return np.where(hit, order[pos], -1)

        bt = self.block_tables.numpy().astype(np.int64)
        new_bt = np.where(bt >= 0, remap(np.where(bt >= 0, bt, 0)), -1).astype(np.int32)
        slots = self.slot_mapping.numpy()
        blk = np.where(slots >= 0, slots // self.block_size, 0)
        nb = remap(blk)
        new_slots = np.where((slots >= 0) & (nb >= 0), nb * self.block_size + slots % self.block_size, -1)
        return (self.k_used.clone(), self.v_used.clone(), torch.from_numpy(new_bt),
                torch.from_numpy(new_slots.astype(np.int64)))

    def kv_bytes_read(self) -> int:
        """Algorithmic K+V bytes of one decode: tokens used per distinct (block, kv head)."""
        return int(self.meta["unique_tokens"]) * self.num_kv_heads * self.head_dim * self.elt * 2

    def algorithmic_bytes(self) -> int:
        """Unique K/V bytes read + q + out + block-table entries used + context lengths."""
        qo = 2 * self.num_seqs * self.num_q_heads * self.head_dim * self.elt
        used_entries = int(sum((int(L) + self.block_size - 1) // self.block_size
                               for L in self.context_lens.tolist()))
        return self.kv_bytes_read() + qo + 4 * used_entries + 4 * self.num_seqs

    def append_bytes(self) -> int:
        """Append: key+value read, the same written, slots read."""
        T = int(self.slot_mapping.numel())
        valid = int((self.slot_mapping >= 0).sum())
        row = self.num_kv_heads * self.head_dim * self.elt
        return 2 * valid * row * 2 + 8 * T


def _cast(x: np.ndarray, dtype: torch.dtype, shape) -> torch.Tensor:
    return torch.from_numpy(x).reshape(shape).to(dtype)


def custom_case(name: str, *, lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                block_size: int = 16, dtype=torch.bfloat16, seed: int = 0,
                num_blocks: int | None = None, spare_blocks: int = 0,
                groups: tuple[int, int] | None = None, append: str = "tail",
                n_append: int | None = None, heavy_key_frac: float = 0.0,
                heavy_key_factor: float = 8.0, max_blocks: int | None = None) -> DecodeCase:
    """Build one seeded decode step.

    lens: context length of every sequence (this step's token included).
    groups: (group_size, shared_blocks): consecutive sequences in groups of
      ``group_size`` share their first ``shared_blocks`` physical blocks.
    num_blocks: pool size (default: exactly the blocks used + ``spare_blocks``).
    append: "tail" -- each sequence appends its token at position L-1;
            "free" -- ``n_append`` tokens go to distinct slots nobody reads;
            "none" -- no append.
    heavy_key_frac: fraction of key vectors (per block, slot, kv head) scaled
      by ``heavy_key_factor`` before the cast.
    """
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int64)
    B, Hq, Hkv, D, bs = len(lens), num_q_heads, num_kv_heads, head_dim, block_size
    assert Hq % Hkv == 0 and (lens >= 0).all()
    nblk = (lens + bs - 1) // bs
    M_b = int(max(1, nblk.max() if B else 1)) if max_blocks is None else int(max_blocks)
    assert (nblk <= M_b).all()

    # logical block ids: shared prefix blocks first, then private ones
    logical = np.full((B, M_b), -1, np.int64)
    n_logical = 0
    if groups is not None:
        gsize, shared = groups
        for g0 in range(0, B, gsize):
            members = range(g0, min(B, g0 + gsize))
            assert all(nblk[i] >= shared for i in members)
            logical[g0:g0 + gsize, :shared] = np.arange(n_logical, n_logical + shared)
            n_logical += shared
    for i in range(B):
        start = 0 if groups is None else groups[1]
        k = int(nblk[i]) - start
        logical[i, start:start + k] = np.arange(n_logical, n_logical + k)
        n_logical += k

    N_b = n_logical + spare_blocks if num_blocks is None else int(num_blocks)
    assert N_b >= n_logical
    if N_b <= 4_000_000:
        phys_of_logical = rng.permutation(N_b)[:n_logical]
    else:
        phys_of_logical = rng.choice(N_b, size=n_logical, replace=False)
    bt = np.where(logical >= 0, phys_of_logical[np.maximum(logical, 0)], -1).astype(np.int32)

    # valid slots per logical block = max over its readers of tokens it holds
    valid = np.zeros(n_logical, np.int64)
    for i in range(B):
        for jb in range(int(nblk[i])):
            lb = logical[i, jb]
            valid[lb] = max(valid[lb], min(bs, int(lens[i]) - jb * bs))

    n_elem = n_logical * Hkv * bs * D
    kd = normal(seed * 16 + 1, n_elem).reshape(n_logical, Hkv, bs, D)
    if heavy_key_frac > 0:
        heavy = rng.random((n_logical, Hkv, bs)) < heavy_key_frac
        kd[heavy] *= np.float32(heavy_key_factor)
    vd = normal(seed * 16 + 2, n_elem).reshape(n_logical, Hkv, bs, D)
    slot_idx = np.arange(bs)
    tail_mask = slot_idx[None, :] >= valid[:, None]           # [n_logical, bs]
    kd[np.broadcast_to(tail_mask[:, None, :], (n_logical, Hkv, bs))] = np.nan
    vd[np.broadcast_to(tail_mask[:, None, :], (n_logical, Hkv, bs))] = np.nan

    # this step's append
    if append == "tail":
        T = int((lens > 0).sum())
        seqs = np.nonzero(lens > 0)[0]
        pos = lens[seqs] - 1
        slots = bt[seqs, pos // bs].astype(np.int64) * bs + pos % bs
        # the slot is still empty before the append
        lb = logical[seqs, pos // bs]
        kd[lb, :, pos % bs, :] = np.nan
        vd[lb, :, pos % bs, :] = np.nan
    elif append == "free":
        T = int(n_append if n_append is not None else B)
        used_phys = set(phys_of_logical.tolist())
        spare = np.array([p for p in range(N_b) if p not in used_phys], np.int64) \
            if N_b <= 4_000_000 else np.zeros(0, np.int64)
        free = [spare[:, None] * bs + slot_idx[None, :]]
        for lb in range(n_logical):
            if valid[lb] < bs:
                free.append(phys_of_logical[lb] * bs + np.arange(valid[lb], bs)[None, :])
        free = np.concatenate([f.reshape(-1) for f in free]) if free else np.zeros(0, np.int64)
        assert len(free) >= T
        slots = np.sort(rng.choice(free, size=T, replace=False)).astype(np.int64)
        slots = slots[rng.permutation(T)]
    elif append == "none":
        T = 0
        slots = np.zeros(0, np.int64)
    else:
        raise ValueError(append)

    q = normal(seed * 16 + 3, B * Hq * D)
    key = normal(seed * 16 + 4, T * Hkv * D)
    value = normal(seed * 16 + 5, T * Hkv * D)

    unique_tokens = int(valid.sum())
    return DecodeCase(
        name=name, dtype=dtype, num_seqs=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
        block_size=bs, num_blocks=N_b,
        scale=float(np.float32(1.0 / math.sqrt(D))),
        q=_cast(q, dtype, (B, Hq, D)),
        context_lens=torch.from_numpy(lens.astype(np.int32)),
        block_tables=torch.from_numpy(bt),
        used_blocks=torch.from_numpy(phys_of_logical.astype(np.int64)),
        k_used=_cast(kd, dtype, (n_logical, Hkv, bs, D)),
        v_used=_cast(vd, dtype, (n_logical, Hkv, bs, D)),
        key=_cast(key, dtype, (T, Hkv, D)),
        value=_cast(value, dtype, (T, Hkv, D)),
        slot_mapping=torch.from_numpy(slots),
        meta={"unique_tokens": unique_tokens, "seed": seed, "groups": groups,
              "append": append, "heavy_key_frac": heavy_key_frac},
    )


# ---------------------------------------------------------------------------
# The five workloads.  Seeds are 1000 + index.
# ---------------------------------------------------------------------------

def _c0(r=0):
    # 4 sequences, 4/2 heads, D 64, fp32, pool of 32 blocks; append 1 token each
    return custom_case("tiny_paged_decode", lens=[7, 16, 33, 50], num_q_heads=4, num_kv_heads=2,
                       head_dim=64, block_size=16, dtype=torch.float32, seed=1000 + 100000 * r,
                       num_blocks=32, append="tail")


def _c1(r=0):
    rng = np.random.default_rng(1001 + 100000 * r)
    lens = rng.integers(128, 2048, size=64, endpoint=True)
    return custom_case("tinyllama_1.1b_decode", lens=lens, num_q_heads=32, num_kv_heads=4,
                       head_dim=64, block_size=16, dtype=torch.float16, seed=1001 + 100000 * r, append="tail")


def _c2(r=0):
    rng = np.random.default_rng(1002 + 100000 * r)
    lens = rng.integers(1024, 4096, size=128, endpoint=True)
    return custom_case("llama2_7b_mha_decode", lens=lens, num_q_heads=32, num_kv_heads=32,
                       head_dim=128, block_size=16, dtype=torch.bfloat16, seed=1002 + 100000 * r,
                       spare_blocks=64, append="free", n_append=128)


def _c3(r=0):
    rng = np.random.default_rng(1003 + 100000 * r)
    z = rng.standard_normal(256)
    tails = np.clip(np.rint(1500.0 * np.exp(0.5 * z)), 1, 32768 - 1024).astype(np.int64)
    lens = 1024 + tails
    return custom_case("qwen2.5_7b_gqa_prefix_decode", lens=lens, num_q_heads=28, num_kv_heads=4,
                       head_dim=128, block_size=16, dtype=torch.bfloat16, seed=1003 + 100000 * r,
                       groups=(8, 64), append="tail")


def _c4(r=0):
    rng = np.random.default_rng(1004 + 100000 * r)
    lens = rng.integers(32768, 131072, size=8, endpoint=True)
    n_b = (120 * 10**9) // (2 * 8 * 16 * 128 * 2)
    return custom_case("long_context_splitkv_decode", lens=lens, num_q_heads=32, num_kv_heads=8,
                       head_dim=128, block_size=16, dtype=torch.bfloat16, seed=1004 + 100000 * r,
                       num_blocks=n_b, append="tail", heavy_key_frac=0.01, heavy_key_factor=8.0)


# Report-only rows: a Gemma-shaped multi-query geometry (one kv head, head_dim
# 256) and the Llama-2-shaped batch over 32-token blocks.
def _gemma_mqa(r=0):
    rng = np.random.default_rng(1005 + 100000 * r)
    lens = rng.integers(1024, 4096, size=128, endpoint=True)
    return custom_case("gemma_mqa_decode", lens=lens, num_q_heads=8, num_kv_heads=1, head_dim=256,
                       block_size=16, dtype=torch.bfloat16, seed=1005 + 100000 * r, append="tail")


def _bs32(r=0):
    rng = np.random.default_rng(1006 + 100000 * r)
    lens = rng.integers(1024, 4096, size=128, endpoint=True)
    return custom_case("llama2_7b_bs32_decode", lens=lens, num_q_heads=32, num_kv_heads=32, head_dim=128,
                       block_size=32, dtype=torch.bfloat16, seed=1006 + 100000 * r, spare_blocks=32,
                       append="free", n_append=128)


_BUILDERS = {"c0": _c0, "c1": _c1, "c2": _c2, "c3": _c3, "c4": _c4, "gemma_mqa": _gemma_mqa, "bs32": _bs32}
CASE_NAMES = tuple(_BUILDERS)


def make_case(name: str, replica: int = 0) -> DecodeCase:
    """One of the workloads: c0 (tiny, fp32), c1 (TinyLlama-1.1B-shaped),
    c2 (Llama-2-7B-shaped MHA), c3 (Qwen2.5-7B-shaped GQA with shared prefixes),
    c4 (long-context, 32K-128K tokens, ~120 GB pool), and the report-only rows
    gemma_mqa (8/1 heads, head_dim 256) and bs32 (c2's shape over 32-token
    blocks).  ``replica`` > 0 draws an
    independent batch of the same recipe (another seed)."""
    return _BUILDERS[name](replica)


def e4m3_codes(x: torch.Tensor, amp: float = 1.0) -> torch.Tensor:
    """Input codes for an fp8 (E4M3) cache: PyTorch's float8_e4m3fn cast of
    float32(x) * amp, returned as uint8 (NaN slots stay NaN codes).  This draws
    inputs only; the library's own append rule (which saturates) is not used
    here, so finite values must stay below 448 in magnitude."""
    flat = x.reshape(-1)
    out = torch.empty(flat.shape, dtype=torch.uint8)
    step = 1 << 26
    for i in range(0, flat.numel(), step):
        y = flat[i:i + step].to(torch.float32) * amp
        fin = y[torch.isfinite(y)]
        if fin.numel() and fin.abs().max().item() >= 448:
            raise ValueError("values out of the E4M3 range: lower amp")
        out[i:i + step] = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return out.reshape(x.shape)
