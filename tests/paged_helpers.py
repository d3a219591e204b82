"""Test-side helpers: lay dense per-sequence K/V out in a paged pool.

Used to pin the oracle against dense attention.  Written with plain torch
indexing, independent of both the oracle and the CUDA library.
"""
import torch


def paged_from_dense(dense_k, dense_v, block_size, num_blocks, gen, pad_blocks=0):
    """dense_k[i], dense_v[i]: [L_i, Hkv, D].  Returns (k_pool, v_pool, tables).

    Physical blocks are a random permutation of range(num_blocks); unused
    blocks and unused tail slots hold NaN.  ``pad_blocks`` extra table columns
    are filled with -1.
    """
    Hkv, D = dense_k[0].shape[1], dense_k[0].shape[2]
    dtype = dense_k[0].dtype
    nblk = [(k.shape[0] + block_size - 1) // block_size for k in dense_k]
    need = sum(nblk)
    assert need <= num_blocks
    perm = torch.randperm(num_blocks, generator=gen)
    k_pool = torch.full((num_blocks, Hkv, block_size, D), float("nan"), dtype=dtype)
    v_pool = torch.full_like(k_pool, float("nan"))
    width = max(max(nblk), 1) + pad_blocks
    tables = torch.full((len(dense_k), width), -1, dtype=torch.int32)
    nxt = 0
    for i, (k, v) in enumerate(zip(dense_k, dense_v)):
        for j in range(nblk[i]):
            pb = int(perm[nxt]); nxt += 1
            tables[i, j] = pb
            lo, hi = j * block_size, min(k.shape[0], (j + 1) * block_size)
            k_pool[pb, :, : hi - lo, :] = k[lo:hi].transpose(0, 1)
            v_pool[pb, :, : hi - lo, :] = v[lo:hi].transpose(0, 1)
    return k_pool, v_pool, tables
