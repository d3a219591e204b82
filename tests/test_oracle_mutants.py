"""The pins catch plausible oracle mistakes.

Each case plants one mistake in a copy of the oracle's C source (a wrong
grouped-query head map, no max subtraction, a dropped scale, an off-by-one
block index, a causal off-by-one, ties rounded away from even), builds it as a
separate library, and checks that an independent reference -- torch float64
attention on the dense tokens, a closed form, or torch's E4M3 cast -- now
disagrees with it.  The unmodified oracle agrees with the same references in
test_oracle.py / test_oracle_prefill.py.
"""
import math
import os
import subprocess

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tests.paged_helpers import paged_from_dense


def _build_mutant(tmp_path, old, new, count=1):
    src = open(oracle._SRC).read()
    assert src.count(old) >= count, old
    mutated = src.replace(old, new, count)
    path = tmp_path / "oracle_mutant.c"
    path.write_text(mutated)
    lib = tmp_path / "oracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math", "-o", str(lib),
                    str(path), "-lm"], check=True)
    return str(path), str(lib)


class _Using:
    """Point the oracle module at another compiled source for the duration."""

    def __init__(self, src, lib):
        self.src, self.lib = src, lib

    def __enter__(self):
        self.saved = (oracle._SRC, oracle._LIB, oracle._lib)
        oracle._SRC, oracle._LIB, oracle._lib = self.src, self.lib, None

    def __exit__(self, *exc):
        oracle._SRC, oracle._LIB, oracle._lib = self.saved


def _dense_attention(q_rows, k, v, scale, allowed=None):
    # q_rows [n, Hq, D]; k/v [L, Hkv, D]; GQA by repeat_interleave; returns [n, Hq, D] float64
    Hq = q_rows.shape[1]
    G = Hq // k.shape[1]
    kk = k.to(torch.float64).transpose(0, 1).repeat_interleave(G, 0)
    vv = v.to(torch.float64).transpose(0, 1).repeat_interleave(G, 0)
    qq = q_rows.to(torch.float64).transpose(0, 1)
    o = F.scaled_dot_product_attention(qq[None], kk[None], vv[None], attn_mask=allowed, scale=scale)
    return o[0].transpose(0, 1)


def decode_error():
    gen = torch.Generator().manual_seed(1)
    lens, Hq, Hkv, D = [5, 33, 17], 8, 2, 64
    dk = [torch.randn(L, Hkv, D, generator=gen) for L in lens]
    dv = [torch.randn(L, Hkv, D, generator=gen) for L in lens]
    kp, vp, bt = paged_from_dense(dk, dv, 16, 8, gen)
    q = torch.randn(3, Hq, D, generator=gen)
    scale = float(np.float32(0.125))
    got = oracle.paged_decode(q, kp, vp, bt, torch.tensor(lens, dtype=torch.int32), Hkv, scale)
    ref = torch.stack([_dense_attention(q[i:i + 1], dk[i], dv[i], scale)[0] for i in range(3)])
    return (got - ref).abs().max().item()


def dominant_key_error():
    # scores around 1e4: without the max subtraction exp overflows
    D = 64
    k = torch.zeros(3, 1, D)
    k[1, 0, 0] = 100.0
    v = torch.arange(3 * D, dtype=torch.float32).reshape(3, 1, D)
    kp, vp, bt = paged_from_dense([k], [v], 16, 2, torch.Generator().manual_seed(0))
    q = torch.zeros(1, 1, D)
    q[0, 0, 0] = 100.0
    got = oracle.paged_decode(q, kp, vp, bt, torch.tensor([3], dtype=torch.int32), 1, 1.0)
    err = (got[0, 0] - v[1, 0].double()).abs().max().item()
    return err if math.isfinite(err) else float("inf")


def prefill_error():
    gen = torch.Generator().manual_seed(2)
    L, n, Hq, Hkv, D = 40, 12, 4, 2, 64
    k = torch.randn(L, Hkv, D, generator=gen)
    v = torch.randn(L, Hkv, D, generator=gen)
    kp, vp, bt = paged_from_dense([k], [v], 16, 4, gen)
    q = torch.randn(n, Hq, D, generator=gen)
    scale = float(np.float32(0.125))
    got = oracle.paged_prefill(q, kp, vp, bt, torch.tensor([L], dtype=torch.int32),
                               torch.tensor([0, n], dtype=torch.int32), Hkv, scale)
    allowed = torch.arange(L)[None, :] <= torch.arange(L - n, L)[:, None]
    ref = _dense_attention(q, k, v, scale, allowed)
    return (got - ref).abs().max().item()


def e4m3_error():
    v = oracle.widen_e4m3(torch.arange(0x7F, dtype=torch.uint8))
    mids = ((v[1:] + v[:-1]) / 2).to(torch.float32)  # every tie between neighbouring codes
    got = oracle.e4m3_encode(mids)
    ref = mids.to(torch.float8_e4m3fn).view(torch.uint8)
    return float((got != ref).sum().item())


MUTANTS = [
    ("grouped-query head map", "    const int64_t c = h / G;", "    const int64_t c = h % num_kv_heads;", decode_error),
    ("no max subtraction", "      const double w = exp(s[j] - m);", "      const double w = exp(s[j]);",
     dominant_key_error),
    ("scale dropped", "      s[j] = scale_d * dot;", "      s[j] = dot;", decode_error),
    ("off-by-one block index", "      const int64_t pb = block_tables[b * max_blocks + j / block_size];",
     "      const int64_t pb = block_tables[b * max_blocks + (j + 1) / block_size];", decode_error),
    ("causal off-by-one", "    const int64_t P = L - n + (t - query_start_loc[b]);",
     "    const int64_t P = L - n + (t - query_start_loc[b]) - 1;", prefill_error),
    ("ties away from even", "if (d < best_d || (d == best_d && (c & 1) == 0)) {", "if (d < best_d) {", e4m3_error),
]


@pytest.mark.parametrize("what,old,new,check", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_a_planted_mistake(tmp_path, what, old, new, check):
    assert check() < 1e-9, "the unmodified oracle agrees with the reference"
    src, lib = _build_mutant(tmp_path, old, new)
    with _Using(src, lib):
        try:
            err = check()
        except oracle.OracleError:
            err = float("inf")
    assert not err < 1e-6, f"{what}: the planted mistake went unnoticed (error {err})"
