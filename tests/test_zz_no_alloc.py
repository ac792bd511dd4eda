"""The allocation-free layout entry point (ep_get_layout_noalloc), for
callers that cannot allocate device memory: it must give exactly what
ep_get_layout gives with a caller-allocated workspace, call after call, while
its scratch lives in the library's own device memory.

Kept in a file that pytest collects last, so that a run that stops at the
first failure has run every other test before this one."""

import ctypes

import numpy as np
import pytest
import torch

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


FIELDS = ("expert_count", "expert_start", "expert_end", "rank_start",
          "tokens_per_rank", "is_token_in_rank", "slot_of", "src_info")


def _host(L):
    return {f: getattr(L, f).cpu().numpy().copy() for f in FIELDS}


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", ["prefill", "skew", "decode"])
def test_noalloc_layout_matches_workspace_layout_twice(ep, name):
    wl = workloads.WORKLOADS[name]
    cfg = ep.Config(wl.num_tokens, wl.hidden, wl.num_topk, wl.num_experts,
                    wl.num_ranks, wl.expert_alignment, wl.use_fp8_dispatch, False)
    ref_L = ep.Layout(cfg)
    na_L = ep.Layout(cfg)
    na_L.c.workspace = None          # the entry point must not need one
    for seed in (0, 1):              # two calls in a row, different routes
        idx = torch.from_numpy(workloads.make_inputs(wl, seed=seed)["topk_idx"]).cuda()
        h_ref = np.zeros(wl.num_experts, np.int32)
        h_na = np.zeros(wl.num_experts, np.int32)
        st = ep.ep_get_layout(cfg.c(), wl.num_tokens, idx.data_ptr(), ref_L.c,
                              h_ref.ctypes.data_as(ctypes.c_void_p), _stream())
        assert st == ep.EP_OK
        st = ep.ep_get_layout_noalloc(cfg.c(), wl.num_tokens, idx.data_ptr(), na_L.c,
                                      h_na.ctypes.data_as(ctypes.c_void_p), _stream())
        assert st == ep.EP_OK, ep.ep_status_str(st)
        torch.cuda.synchronize()
        assert na_L.num_tokens == wl.num_tokens
        assert np.array_equal(h_na, h_ref)
        a, b = _host(na_L), _host(ref_L)
        used = int(b["expert_start"][-1])
        for f in FIELDS:
            if f == "src_info":
                assert np.array_equal(a[f][:used], b[f][:used]), f
            else:
                assert np.array_equal(a[f], b[f]), f
        assert ep.ep_check_error(na_L.c, _stream()) == ep.EP_OK


def test_noalloc_rejects_configs_beyond_its_scratch(ep):
    cfg = ep.Config(1024, 128, 8, 2048, 2048, 4)
    assert ep.ep_layout_workspace_bytes(cfg.c()) > (1 << 20)
    L = ep.Layout(ep.Config(1024, 128, 8, 64, 8, 4))   # any valid buffers
    idx = torch.zeros((1024, 8), dtype=torch.int64, device="cuda")
    st = ep.ep_get_layout_noalloc(cfg.c(), 1024, idx.data_ptr(), L.c, None, _stream())
    assert st == ep.EP_ERR_CAPACITY


def test_noalloc_small_layout_needs_no_scratch(ep):
    """A layout of at most 4096 (t, k) pairs takes one launch and uses no
    scratch, so the allocation-free entry point accepts it even where the
    two-launch scratch would exceed the array (2048 experts, 2048 ranks)."""
    cfg = ep.Config(512, 128, 8, 2048, 2048, 4)
    assert ep.ep_layout_workspace_bytes(cfg.c()) > (1 << 20)
    rng = np.random.default_rng(21)
    idx_np = workloads.random_routes(rng, 512, 2048, 8)
    idx = torch.from_numpy(idx_np).cuda()
    ref_L, na_L = ep.Layout(cfg), ep.Layout(cfg)
    na_L.c.workspace = None
    for _ in range(2):
        assert ep.ep_get_layout(cfg.c(), 512, idx.data_ptr(), ref_L.c, None, _stream()) == ep.EP_OK
        st = ep.ep_get_layout_noalloc(cfg.c(), 512, idx.data_ptr(), na_L.c, None, _stream())
        assert st == ep.EP_OK, ep.ep_status_str(st)
        torch.cuda.synchronize()
        a, b = _host(na_L), _host(ref_L)
        used = int(b["expert_start"][-1])
        for f in FIELDS:
            if f == "src_info":
                assert np.array_equal(a[f][:used], b[f][:used]), f
            else:
                assert np.array_equal(a[f], b[f]), f
        assert ep.ep_check_error(na_L.c, _stream()) == ep.EP_OK
