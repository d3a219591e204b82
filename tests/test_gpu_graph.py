"""CUDA-graph capture of the decode step over several layers: the fused
append + decode (+ in-launch merge of split sequences) launches are recorded
once and replayed; the replay must reproduce the eager outputs bit for bit
and match the oracle."""
import pytest
import torch

import paged_kv_cache_185_gb300 as wllm
from paged_kv_cache_185_gb300 import workloads
from tests.gpu_common import assert_attention_close, int_view, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    wllm.load_library()
    yield


def _layers(n, dtype, Hq, Hkv, D):
    lens = [1, 17, 300, 1025, 2100, 64, 900, 4000]
    return [workloads.custom_case(f"graph{l}", lens=lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                                  block_size=16, dtype=dtype, seed=500 + l, heavy_key_frac=0.01)
            for l in range(n)]


def _inputs(case):
    kc, vc = case.pool("cuda")
    return dict(out=torch.empty(case.q.shape, dtype=case.q.dtype, device="cuda"), q=case.q.cuda(),
                key=case.key.cuda(), value=case.value.cuda(), kc=kc, vc=vc,
                slots=case.slot_mapping.cuda(), bt=case.block_tables.cuda(), cl=case.context_lens.cuda())


def _step(case, x):
    wllm.decode_step(x["out"], x["q"], x["key"], x["value"], x["kc"], x["vc"], x["slots"], x["bt"], x["cl"],
                     case.num_kv_heads, case.scale, case.block_size)


@pytest.mark.parametrize("dtype,Hq,Hkv,D,part", [(torch.float16, 32, 4, 64, 256),
                                                 (torch.bfloat16, 28, 4, 128, 1024),
                                                 (torch.bfloat16, 32, 32, 128, 4096)])
def test_decode_step_graph_replay(monkeypatch, dtype, Hq, Hkv, D, part):
    monkeypatch.setenv("WLLM_PARTITION_TOKENS", str(part))
    cases = _layers(3, dtype, Hq, Hkv, D)
    # eager reference, one layer after the other on one stream
    eager = []
    for c in cases:
        x = _inputs(c)
        _step(c, x)
        eager.append(x["out"])
    torch.cuda.synchronize()
    # a caller-owned workspace sized for the largest layer: nothing is allocated while capturing
    need = max(wllm.workspace_bytes(c.num_seqs, c.num_q_heads, c.num_kv_heads, c.head_dim, c.max_blocks,
                                    c.block_size) for c in cases)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    wllm.set_workspace(ws)
    try:
        xs = [_inputs(c) for c in cases]
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # warm-up outside the capture (function attributes, counters)
            for c, x in zip(cases, xs):
                _step(c, x)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for c, x in zip(cases, xs):
                _step(c, x)
        for x in xs:
            x["out"].fill_(float("nan"))
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        assert wllm.device_errors() == 0
        for l, (c, x) in enumerate(zip(cases, xs)):
            assert torch.equal(int_view(x["out"]), int_view(eager[l])), f"layer {l}: replay differs from eager"
        ref, kr, _ = oracle_step(cases[0])
        assert torch.equal(int_view(xs[0]["kc"].cpu()), int_view(kr)), "append under replay not bit-exact"
        assert_attention_close(xs[0]["out"].cpu(), ref, dtype, "graph layer 0")
    finally:
        wllm.set_workspace(None)


def test_fp8_step_and_prefill_graph_replay():
    # the fp8 fused step (two layers) and a chunked prefill, captured in one graph
    cases = _layers(2, torch.bfloat16, 32, 8, 128)
    xs = []
    for c in cases:
        x = _inputs(c)
        kh, vh = c.pool("cpu")
        x["kc"], x["vc"] = workloads.e4m3_codes(kh, 4.0).cuda(), workloads.e4m3_codes(vh, 4.0).cuda()
        xs.append(x)
    pc = workloads.custom_case("graph_prefill", lens=[300, 1500], num_q_heads=28, num_kv_heads=4, head_dim=128,
                               block_size=16, dtype=torch.bfloat16, seed=77, append="none")
    pk, pv = pc.pool("cuda")
    pq = torch.randn(700, 28, 128, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16).cuda()
    pqsl = torch.tensor([0, 300, 700], dtype=torch.int32, device="cuda")
    pbt, pcl = pc.block_tables.cuda(), pc.context_lens.cuda()
    pout = torch.empty_like(pq)

    def run():
        for c, x in zip(cases, xs):
            wllm.decode_step_fp8(x["out"], x["q"], x["key"], x["value"], x["kc"], x["vc"], x["slots"], x["bt"],
                                 x["cl"], c.num_kv_heads, c.scale, 0.25, 0.25, c.block_size)
        wllm.paged_attention_prefill(pout, pq, pk, pv, pbt, pcl, pqsl, 4, pc.scale, 16)

    need = max(wllm.workspace_bytes(c.num_seqs, c.num_q_heads, c.num_kv_heads, c.head_dim, c.max_blocks,
                                    c.block_size) for c in cases)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    wllm.set_workspace(ws)
    try:
        run()
        torch.cuda.synchronize()
        eager = [x["out"].clone() for x in xs] + [pout.clone()]
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            run()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            run()
        for t in [x["out"] for x in xs] + [pout]:
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert wllm.device_errors() == 0
        for t, e in zip([x["out"] for x in xs] + [pout], eager):
            assert torch.equal(int_view(t), int_view(e)), "replay differs from eager"
    finally:
        wllm.set_workspace(None)
