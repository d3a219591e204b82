"""Write tests/golden/tiny_paged_decode.txt from the fp64 oracle alone.

The tiny workload (4 sequences with context lengths 7, 16, 33, 50; 4 query /
2 KV heads; head_dim 64; block size 16; pool of 32 blocks; fp32) is drawn by
the seeded generator, the step's four new tokens are appended by the oracle,
and the oracle's decode output is stored as one hex float per line
(row-major [seq][head][dim]).  The pages print no worked example, so this file
is a regression fixture of the oracle, not a pin of it.

    python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from paged_kv_cache_185_gb300 import workloads  # noqa: E402


def compute():
    case = workloads.make_case("c0")
    kc, vc = case.pool()
    oracle.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping)
    return oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens,
                               case.num_kv_heads, case.scale)


def main():
    out = compute()
    path = os.path.join(HERE, "tiny_paged_decode.txt")
    with open(path, "w") as f:
        f.write("# fp64 oracle output, tiny paged decode workload, shape "
                + "x".join(str(s) for s in out.shape) + "\n")
        for x in out.reshape(-1).tolist():
            f.write(float(x).hex() + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
