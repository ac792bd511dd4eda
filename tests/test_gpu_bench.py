"""GPU checks of the measurement harness itself: the pipelined end-to-end
leg with fewer steps than batches in flight, issued call by call or
replayed from a CUDA graph (every slot that runs is checked against a
one-step-at-a-time result), and a short default-style run of bench.py that
must print one JSON line with the contract's keys."""

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import bench
import workloads

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import load_build_module

    load_build_module().build()
    import combine_get_layout_gb300 as ep

    return ep


def _inputs(ep, wl, device):
    inp = workloads.make_inputs(wl, seed=0)
    T, H, K = wl.num_tokens, wl.hidden, wl.num_topk
    cfg = ep.Config(T, H, K, wl.num_experts, wl.num_ranks, wl.expert_alignment,
                    wl.use_fp8_dispatch)
    x_h = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    route_h = torch.empty(T * K * 12, dtype=torch.uint8).pin_memory()
    for v, a in zip(bench.route_views(route_h, T, K), (inp["topk_idx"], inp["topk_weights"])):
        v.copy_(torch.from_numpy(a))
    g = torch.Generator(device=device)
    g.manual_seed(7)
    Y_d = torch.randn((cfg.capacity, H), generator=g, device=device).to(torch.bfloat16)
    # one step at a time through the device entry points: the rows every
    # pipelined step must give back
    idx_d, w_d = bench.route_views(route_h.to(device), T, K)
    L = ep.get_layout(cfg, idx_d, sync=True)
    rx, _, _ = ep.dispatch(cfg, L, x_h.to(device), w_d)
    ident = Y_d if wl.use_fp8_dispatch else rx
    y_want = ep.combine(cfg, L, ident, w_d).cpu()
    torch.cuda.synchronize()
    return cfg, x_h, route_h, rx, Y_d, y_want


@pytest.mark.parametrize("name,chunks", [("tiny", 0), ("decode", 0), ("sweep1k", 2)])
@pytest.mark.parametrize("steps,warmup", [(1, 1), (2, 1), (3, 6)])
@pytest.mark.parametrize("graph_steps", [0, 64])
def test_pipelined_e2e_with_fewer_steps_than_depth(ep, name, chunks, steps, warmup, graph_steps):
    wl = workloads.WORKLOADS[name]
    device = torch.device("cuda", 0)
    cfg, x_h, route_h, rx, Y_d, y_want = _inputs(ep, wl, device)
    r = bench.pipelined_e2e(ep, cfg.c(), cfg, wl.num_tokens, wl.num_topk, wl.hidden, wl,
                            device, torch.cuda.current_stream(device), x_h, route_h,
                            None if wl.use_fp8_dispatch else rx, Y_d, chunks, steps, warmup,
                            1, y_want, depth=4, graph_steps=graph_steps)
    assert r["value"] > 0 and r["ms_per_step"] > 0
    depth = min(4, max(steps, warmup))
    assert r["pipelining"].startswith(f"{depth} batches in flight")
    if graph_steps:
        # whole replays of one graph of steps, a multiple of the depth
        G = depth * (graph_steps // depth)
        assert r["steps_timed"] == G and f"graph of {G} steps" in r["launch"]
    else:
        assert r["steps_timed"] == steps


def test_short_bench_run_prints_one_line(ep):
    out = subprocess.run([sys.executable, "bench.py", "--workload", "tiny", "--steps", "2",
                          "--warmup", "3", "--no-cpu-baseline"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "config", "roofline", "e2e",
                "clocks", "gpu_launches"):
        assert key in d, key
    assert d["steps"] == 2 and d["value"] > 0 and d["gpu_launches"] > 0
    assert d["e2e"]["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] > 0
