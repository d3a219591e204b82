"""The benchmark's reference arm (the oracle on the host cores) prints the
contract's JSON line; runs without a GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == "decode-attn tokens/s" and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "long_context_splitkv_decode"
    assert d["cpu_baseline"]["cores"] <= os.cpu_count()


def test_oracle_sample_order_covers_every_row_once():
    import bench
    from paged_kv_cache_185_gb300 import workloads
    case = workloads.make_case("c0")
    order = bench.sample_rows(case)
    B, Hq = case.num_seqs, case.num_q_heads
    assert sorted(order) == list(range(B * Hq))
    assert [r // Hq for r in order[:B]] == list(range(B))  # the first B rows visit every sequence


def test_host_oracle_inputs_never_build_the_full_pool():
    """The long-context batch's oracle inputs hold only the referenced blocks."""
    import bench
    from paged_kv_cache_185_gb300 import workloads
    case = workloads.make_case("c4")
    kc, vc, bt = bench.host_oracle_inputs(case)
    assert kc.shape[0] == case.used_blocks.numel() < case.num_blocks // 50
    assert int(bt.max()) < kc.shape[0]
