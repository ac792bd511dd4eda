"""GPU checks of the host-buffer entry points (ep_dispatch_from_host,
ep_combine_to_host): rows copied in token chunks on the library's copy
streams (one for host-to-device, one for device-to-host), each chunk's
kernel waiting for its own copy.  The results must equal the device-buffer
entry points bit for bit (which the parity suite holds to the oracle), for
one chunk (on the caller's stream) and several (on the copy streams) with a
ragged last chunk, FP8 rows and zero padding; one case is also compared with
the oracle directly, and one keeps two batches in flight on two streams.
With 0 chunks (direct) the kernels read and write the pinned host rows in
place, with no staging buffer."""

import mmap

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import load_build_module

    load_build_module().build()
    import combine_get_layout_gb300 as ep

    return ep


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def pinned_bf16(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(
        torch.bfloat16).pin_memory()


def u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


CASES = {
    # 2 MB of rows: one chunk whatever num_chunks is (chunks carry >= 4 MiB)
    "ragged": workloads.Workload("ragged", 1000, 1024, 64, 8, 8, False,
                                 expert_alignment=16, mask_frac=0.07),
    # 35.8 MB of rows: up to 8 chunks, the last ragged
    "wide": workloads.Workload("wide", 2500, 7168, 64, 8, 8, False,
                               expert_alignment=16, mask_frac=0.05),
    "wide_fp8": workloads.Workload("wide_fp8", 2500, 7168, 64, 8, 8, True,
                                   expert_alignment=16, mask_frac=0.05),
    "fp8": workloads.Workload("fp8", 333, 1024, 32, 4, 4, True, expert_alignment=8,
                              mask_frac=0.1),
    "few_tokens": workloads.Workload("few_tokens", 5, 256, 16, 2, 4, False,
                                     expert_alignment=4),
    "prefill": workloads.WORKLOADS["prefill"],
    # 2 MB rows: 12 MB of x, up to 3 chunks of 2 tokens
    "h_2p20": workloads.Workload("h_2p20", 6, 1 << 20, 4, 2, 2, False, expert_alignment=2),
    "h_2p20_fp8": workloads.Workload("h_2p20_fp8", 6, 1 << 20, 4, 2, 2, True, expert_alignment=2),
}


def _run(ep, wl, chunks, zp, seed=0):
    inp = workloads.make_inputs(wl, seed=seed)
    cfg = ep.Config(wl.num_tokens, wl.hidden, wl.num_topk, wl.num_experts, wl.num_ranks,
                    wl.expert_alignment, wl.use_fp8_dispatch, zp)
    L = ep.get_layout(cfg, dev(inp["topk_idx"]), sync=True)
    w = dev(inp["topk_weights"])
    x_h = pinned_bf16(inp["x"])
    x_d = x_h.cuda()
    ref = ep.dispatch(cfg, L, x_d, w)
    got_x, got_s, got_w, staged = ep.dispatch_from_host(cfg, L, x_h, topk_weights=w,
                                                        num_chunks=chunks)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 5)
    Y = torch.randn((cfg.capacity, wl.hidden), generator=g, device="cuda").to(torch.bfloat16)
    y_ref = ep.combine(cfg, L, Y, w)
    h_y, _ = ep.combine_to_host(cfg, L, Y, w, num_chunks=chunks)
    torch.cuda.current_stream().synchronize()
    return inp, cfg, L, ref, (got_x, got_s, got_w, staged), y_ref, h_y


def _rows(L, cfg, zp):
    es = L.expert_start.cpu().numpy()
    used = int(es[-1])
    if zp:
        return np.arange(used)
    src = L.src_info.cpu().numpy().reshape(-1, 2)[:used]
    return np.nonzero(src[:, 0] >= 0)[0]


@pytest.mark.parametrize("name,chunks,zp", [
    ("ragged", 1, False), ("ragged", 8, True), ("fp8", 7, False), ("fp8", 4, True),
    ("few_tokens", 8, False), ("wide", 3, False), ("wide", 8, True), ("wide", 64, False),
    ("wide_fp8", 5, False), ("wide_fp8", 8, True), ("prefill", 8, False),
    ("ragged", 0, False), ("fp8", 0, True), ("few_tokens", 0, False), ("wide", 0, True),
    ("wide_fp8", 0, False), ("prefill", 0, False),
    ("h_2p20", 3, True), ("h_2p20", 0, False), ("h_2p20_fp8", 3, False), ("h_2p20_fp8", 0, True)])
def test_host_buffers_equal_device_buffers(ep, name, chunks, zp):
    wl = CASES[name]
    inp, cfg, L, ref, got, y_ref, h_y = _run(ep, wl, chunks, zp)
    rows = torch.from_numpy(_rows(L, cfg, zp)).long().cuda()
    rx, rs, rw = ref
    gx, gs, gw, staged = got
    assert torch.equal(gx[rows].view(torch.uint8), rx[rows].view(torch.uint8))
    if cfg.use_fp8_dispatch:
        assert torch.equal(gs[rows].view(torch.int32), rs[rows].view(torch.int32))
    assert torch.equal(gw[rows].view(torch.int32), rw[rows].view(torch.int32))
    if chunks:
        # the staging buffer holds x afterwards
        assert np.array_equal(u16(staged), inp["x"])
    else:
        assert staged is None
    assert np.array_equal(u16(h_y), u16(y_ref))


def test_host_dispatch_matches_oracle(ep):
    wl = CASES["wide"]
    inp, cfg, L, ref, got, y_ref, h_y = _run(ep, wl, 5, True)
    ora = oracle.layout(inp["topk_idx"], wl.num_experts, wl.num_ranks, wl.expert_alignment,
                        cap=cfg.capacity)
    want_x, want_w = oracle.dispatch_bf16(inp["x"], inp["topk_weights"], ora, zero_padding=True)
    used = int(ora["expert_start"][-1])
    assert np.array_equal(u16(got[0])[:used], want_x[:used])
    rows = ora["src_info"][:used, 0] >= 0
    assert np.array_equal(got[2].cpu().numpy()[:used][rows], want_w[:used][rows])


def test_two_calls_in_a_row_reuse_the_events(ep):
    """Back-to-back calls with different inputs, no synchronisation between
    them: each result must be its own call's."""
    wl = CASES["wide"]
    outs = []
    for seed in (0, 1):
        inp = workloads.make_inputs(wl, seed=seed)
        cfg = ep.Config(wl.num_tokens, wl.hidden, wl.num_topk, wl.num_experts, wl.num_ranks,
                        wl.expert_alignment, False, False)
        L = ep.get_layout(cfg, dev(inp["topk_idx"]), sync=True)
        w = dev(inp["topk_weights"])
        x_h = pinned_bf16(inp["x"])
        recv, _, _, _ = ep.dispatch_from_host(cfg, L, x_h, topk_weights=w, num_chunks=6)
        h_y, _ = ep.combine_to_host(cfg, L, recv, w, num_chunks=6)
        outs.append((inp, cfg, L, x_h, w, h_y))
    torch.cuda.current_stream().synchronize()
    for inp, cfg, L, x_h, w, h_y in outs:
        recv, _, _ = ep.dispatch(cfg, L, x_h.cuda(), w)
        y_ref = ep.combine(cfg, L, recv, w)
        torch.cuda.synchronize()
        assert np.array_equal(u16(h_y), u16(y_ref))



def test_two_batches_in_flight_on_two_streams(ep):
    """Two batches, each on its own stream, calls interleaved with no host
    synchronisation: batch B's rows go up while batch A's results come down,
    through the same two copy streams.  Every step's y must be its own
    batch's, bit for bit, and batch A's must match the oracle."""
    wl = CASES["wide"]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    batches = []
    for seed, s in zip((2, 3), streams):
        inp = workloads.make_inputs(wl, seed=seed)
        cfg = ep.Config(wl.num_tokens, wl.hidden, wl.num_topk, wl.num_experts, wl.num_ranks,
                        wl.expert_alignment, False, False)
        idx = dev(inp["topk_idx"])
        w = dev(inp["topk_weights"])
        torch.cuda.synchronize()
        L = ep.get_layout(cfg, idx, sync=True, stream=s)
        batches.append(dict(inp=inp, cfg=cfg, L=L, w=w, x_h=pinned_bf16(inp["x"]),
                            s=s, recv=None, d_x=None, d_y=None, ys=[]))
    steps = 3
    for _ in range(steps):
        for b in batches:
            b["recv"], _, _, b["d_x"] = ep.dispatch_from_host(
                b["cfg"], b["L"], b["x_h"], d_x=b["d_x"], topk_weights=b["w"],
                recv_x=b["recv"], num_chunks=5, stream=b["s"])
        for b in batches:
            h_y, b["d_y"] = ep.combine_to_host(b["cfg"], b["L"], b["recv"], b["w"],
                                               d_y=b["d_y"], num_chunks=7, stream=b["s"])
            b["ys"].append(h_y)
    for s in streams:
        s.synchronize()
    for b in batches:
        assert ep.check_error(b["L"], stream=b["s"]) == 0
        recv, _, _ = ep.dispatch(b["cfg"], b["L"], b["x_h"].cuda(), b["w"])
        y_ref = u16(ep.combine(b["cfg"], b["L"], recv, b["w"]))
        torch.cuda.synchronize()
        for h_y in b["ys"]:
            assert np.array_equal(u16(h_y), y_ref)
    assert not np.array_equal(u16(batches[0]["ys"][0]), u16(batches[1]["ys"][0]))
    inp = batches[0]["inp"]
    ora = oracle.layout(inp["topk_idx"], wl.num_experts, wl.num_ranks, wl.expert_alignment,
                        cap=batches[0]["cfg"].capacity)
    rx, _ = oracle.dispatch_bf16(inp["x"], inp["topk_weights"], ora)
    y_or = oracle.combine(rx, inp["topk_weights"], ora["slot_of"])
    assert np.array_equal(u16(batches[0]["ys"][-1]), y_or)

def test_empty_batch(ep):
    wl = CASES["few_tokens"]
    cfg = ep.Config(wl.num_tokens, wl.hidden, wl.num_topk, wl.num_experts, wl.num_ranks,
                    wl.expert_alignment, False, True)
    L = ep.get_layout(cfg, torch.zeros((0, wl.num_topk), dtype=torch.int64, device="cuda"),
                      sync=True)
    x_h = torch.empty((0, wl.hidden), dtype=torch.bfloat16).pin_memory()
    recv, _, _, _ = ep.dispatch_from_host(cfg, L, x_h, num_chunks=4)
    h_y, _ = ep.combine_to_host(cfg, L, recv, num_chunks=4)
    torch.cuda.synchronize()
    assert h_y.shape == (0, wl.hidden)


def test_direct_mode_needs_page_locked_memory(ep):
    wl = CASES["few_tokens"]
    inp = workloads.make_inputs(wl, seed=0)
    cfg = ep.Config(wl.num_tokens, wl.hidden, wl.num_topk, wl.num_experts, wl.num_ranks,
                    wl.expert_alignment, False, False)
    L = ep.get_layout(cfg, dev(inp["topk_idx"]), sync=True)
    x_pageable = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16)
    with pytest.raises(RuntimeError):
        ep.dispatch_from_host(cfg, L, x_pageable, num_chunks=0)
    recv, _, _ = ep.dispatch(cfg, L, x_pageable.cuda())
    with pytest.raises(RuntimeError):
        ep.combine_to_host(cfg, L, recv, h_y=torch.empty_like(x_pageable), num_chunks=0)
    torch.cuda.synchronize()


@pytest.mark.parametrize("where", ["device", "host"])
def test_fp8_rows_at_16_byte_offset(ep, where):
    """x 16 bytes past a 32-byte boundary takes two 16-byte loads per thread
    instead of one 32-byte load: the same rows and scales either way, and
    the oracle's."""
    wl = CASES["fp8"]
    inp = workloads.make_inputs(wl, seed=3)
    T, H = wl.num_tokens, wl.hidden
    cfg = ep.Config(T, H, wl.num_topk, wl.num_experts, wl.num_ranks, wl.expert_alignment,
                    True, True)
    L = ep.get_layout(cfg, dev(inp["topk_idx"]), sync=True)
    w = dev(inp["topk_weights"])
    flat = torch.empty(T * H + 8, dtype=torch.bfloat16)
    flat = flat.pin_memory() if where == "host" else flat.cuda()
    x_off = flat[8:].view(T, H)          # 16 bytes past the allocation's start
    x_off.copy_(pinned_bf16(inp["x"]))
    assert x_off.data_ptr() % 32 == 16
    if where == "host":
        gx, gs, gw, _ = ep.dispatch_from_host(cfg, L, x_off, topk_weights=w, num_chunks=0)
    else:
        gx, gs, gw = ep.dispatch(cfg, L, x_off, w)
    rx, rs, rw = ep.dispatch(cfg, L, dev(inp["x"].view(np.int16)).view(torch.bfloat16), w)
    torch.cuda.synchronize()
    used = int(L.expert_start[-1].item())
    assert torch.equal(gx[:used], rx[:used])
    assert torch.equal(gs[:used].view(torch.int32), rs[:used].view(torch.int32))
    ora = oracle.layout(inp["topk_idx"], wl.num_experts, wl.num_ranks, wl.expert_alignment,
                        cap=cfg.capacity)
    want_q, want_s, _ = oracle.dispatch_fp8(inp["x"], inp["topk_weights"], ora,
                                            zero_padding=True)
    assert np.array_equal(gx.cpu().numpy()[:used], want_q[:used])
    assert np.array_equal(gs.cpu().numpy()[:used].view(np.uint32),
                          want_s[:used].astype(np.float32).view(np.uint32))


def test_direct_mode_on_registered_memory(ep):
    """Ordinary host arrays registered as page-locked and mapped
    (cudaHostRegister) serve the direct mode as pinned allocations do."""
    rt = torch.cuda.cudart()
    if not hasattr(rt, "cudaHostRegister"):
        pytest.skip("no cudaHostRegister binding in this torch")
    wl = CASES["fp8"]
    inp = workloads.make_inputs(wl, seed=4)
    T, H = wl.num_tokens, wl.hidden
    cfg = ep.Config(T, H, wl.num_topk, wl.num_experts, wl.num_ranks, wl.expert_alignment,
                    True, False)
    L = ep.get_layout(cfg, dev(inp["topk_idx"]), sync=True)
    w = dev(inp["topk_weights"])
    def page_aligned(shape):
        # whole pages of their own, so that the two registrations do not share one
        n = int(np.prod(shape)) * 2
        return np.frombuffer(mmap.mmap(-1, (n + 4095) // 4096 * 4096), np.uint16,
                             count=n // 2).reshape(shape)

    x_np = page_aligned((T, H))
    x_np[:] = inp["x"]
    y_np = page_aligned((T, H))
    mapped = 2  # cudaHostRegisterMapped
    for a in (x_np, y_np):
        assert int(rt.cudaHostRegister(a.ctypes.data, a.nbytes, mapped)) == 0
    try:
        x_h = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16)
        y_h = torch.from_numpy(y_np.view(np.int16)).view(torch.bfloat16)
        gx, gs, _, _ = ep.dispatch_from_host(cfg, L, x_h, topk_weights=w, num_chunks=0)
        g = torch.Generator(device="cuda")
        g.manual_seed(9)
        Y = torch.randn((cfg.capacity, H), generator=g, device="cuda").to(torch.bfloat16)
        ep.combine_to_host(cfg, L, Y, w, h_y=y_h, num_chunks=0)
        rx, rs, _ = ep.dispatch(cfg, L, dev(inp["x"].view(np.int16)).view(torch.bfloat16), w)
        y_ref = ep.combine(cfg, L, Y, w)
        torch.cuda.synchronize()
        rows = torch.from_numpy(_rows(L, cfg, False)).long().cuda()
        assert torch.equal(gx[rows], rx[rows])
        assert torch.equal(gs[rows].view(torch.int32), rs[rows].view(torch.int32))
        assert np.array_equal(y_np, u16(y_ref))
    finally:
        torch.cuda.synchronize()
        for a in (x_np, y_np):
            rt.cudaHostUnregister(a.ctypes.data)
