"""Host-side checks of the C ABI that need no GPU: the shared library loads,
exports every entry point include/ep.h declares, and the pure host functions
(sizing, status names, argument validation) behave as documented.  No call
here reaches a CUDA kernel."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep.h")


@pytest.fixture(scope="module")
def ep():
    from conftest import load_build_module

    load_build_module().build()
    import combine_get_layout_gb300 as ep

    return ep


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"EP_API\s+[\w\s\*]+?\b(ep_\w+)\s*\(", text)))


def test_header_declares_the_abi(ep):
    assert declared_symbols() == sorted(ep.ABI_SYMBOLS)


def test_library_exports_every_declared_symbol(ep):
    out = subprocess.run(["nm", "-D", "--defined-only", ep.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(ep_\w+)$", out, re.M))
    for name in declared_symbols():
        assert name in exported, name
        assert getattr(ep.lib(), name) is not None


def test_struct_layouts_match_header(ep):
    # 8 int32 fields; 13 pointers + 2 int32
    assert ctypes.sizeof(ep.EpConfig) == 32
    assert ctypes.sizeof(ep.EpLayout) == 13 * 8 + 8


def test_capacity_and_workspace(ep):
    cfg = ep.Config(4096, 7168, 8, 256, 8, 128)
    assert ep.ep_recv_capacity(cfg.c()) == 4096 * 8 + 256 * 127 == 65280
    ws = ep.ep_layout_workspace_bytes(cfg.c())
    assert ws > 0 and ws % 16 == 0
    # workspace covers every tile count a smaller T could produce
    small = ep.Config(100, 7168, 8, 256, 8, 128)
    assert ep.ep_layout_workspace_bytes(small.c()) > 0


@pytest.mark.parametrize("bad", [
    dict(hidden=12),                      # not a multiple of 8
    dict(hidden=1024, use_fp8_dispatch=True, max_tokens=8, num_topk=2,
         num_experts=8, num_ranks=2) | {"hidden": 1000},
    dict(num_topk=0), dict(num_topk=33), dict(num_experts=6, num_ranks=4),
    dict(num_topk=9, num_experts=8, num_ranks=2), dict(expert_alignment=0),
    dict(num_ranks=0), dict(max_tokens=-1), dict(max_tokens=2**28, num_topk=16),
    dict(hidden=2**20 + 8),               # bf16 rows past 2^20 channels
    dict(hidden=2**20 + 128, use_fp8_dispatch=True),  # E4M3 rows past 2^20
])
def test_invalid_configs_rejected(ep, bad):
    base = dict(max_tokens=64, hidden=256, num_topk=4, num_experts=16,
                num_ranks=4, expert_alignment=4)
    base.update(bad)
    cfg = ep.Config(**base)
    assert ep.ep_recv_capacity(cfg.c()) == -1
    assert ep.ep_layout_workspace_bytes(cfg.c()) == -1
    lay = ep.EpLayout()
    assert ep.ep_get_layout(cfg.c(), 1, None, lay, None, None) == ep.EP_ERR_INVALID_ARG
    assert ep.ep_dispatch(cfg.c(), lay, None, None, None, None, None, None) == ep.EP_ERR_INVALID_ARG
    assert ep.ep_combine(cfg.c(), lay, None, None, None, None) == ep.EP_ERR_INVALID_ARG


@pytest.mark.parametrize("edge", [dict(hidden=49160), dict(hidden=2**20),
                                  dict(hidden=2**20, use_fp8_dispatch=True)])
def test_widest_rows_accepted(ep, edge):
    base = dict(max_tokens=64, hidden=256, num_topk=4, num_experts=16,
                num_ranks=4, expert_alignment=4)
    base.update(edge)
    assert ep.ep_recv_capacity(ep.Config(**base).c()) == 64 * 4 + 16 * 3


def _has_gpu():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.mark.skipif(_has_gpu(), reason="uses fake device addresses: host-only check")
def test_null_and_misaligned_pointers_rejected(ep):
    cfg = ep.Config(16, 128, 2, 8, 2, 4).c()
    lay = ep.EpLayout()   # all NULL
    assert ep.ep_get_layout(cfg, 4, None, lay, None, None) == ep.EP_ERR_INVALID_ARG
    # fake, never dereferenced addresses: one misaligned
    fake = [0x10000 + 0x100 * i for i in range(10)]
    lay = ep.EpLayout(*fake, None, None, None, 0, 0)
    lay.slot_of = 0x10008
    assert ep.ep_get_layout(cfg, 4, 0x20000, lay, None, None) == ep.EP_ERR_INVALID_ARG
    lay.slot_of = 0x10600
    # num_tokens beyond max_tokens, negative
    assert ep.ep_get_layout(cfg, 17, 0x20000, lay, None, None) == ep.EP_ERR_INVALID_ARG
    assert ep.ep_get_layout(cfg, -1, 0x20000, lay, None, None) == ep.EP_ERR_INVALID_ARG
    assert ep.ep_get_layout(cfg, 4, 0x20004, lay, None, None) == ep.EP_ERR_INVALID_ARG
    # dispatch: recv_w without weights, fp8 without scales
    lay.num_tokens = 4
    assert ep.ep_dispatch(cfg, lay, 0x30000, None, 0x40000, None, 0x50000, None) == ep.EP_ERR_INVALID_ARG
    cfg8 = ep.Config(16, 128, 2, 8, 2, 4, use_fp8_dispatch=True).c()
    assert ep.ep_dispatch(cfg8, lay, 0x30000, None, 0x40000, None, None, None) == ep.EP_ERR_INVALID_ARG
    # host-buffer entry points: chunk count outside 0..64, missing host or
    # staging buffer, misaligned staging buffer; direct mode (0 chunks) on
    # host memory that is not page-locked (a fake address)
    for chunks in (0, 65, -3):
        assert ep.ep_dispatch_from_host(cfg, lay, 0x60000, 0x30000, None, 0x40000, None, None,
                                        chunks, None) == ep.EP_ERR_INVALID_ARG
        assert ep.ep_combine_to_host(cfg, lay, 0x40000, None, 0x30000, 0x60000, chunks,
                                     None) == ep.EP_ERR_INVALID_ARG
    assert ep.ep_dispatch_from_host(cfg, lay, None, 0x30000, None, 0x40000, None, None, 4,
                                    None) == ep.EP_ERR_INVALID_ARG
    assert ep.ep_dispatch_from_host(cfg, lay, 0x60000, 0x30008, None, 0x40000, None, None, 4,
                                    None) == ep.EP_ERR_INVALID_ARG
    assert ep.ep_dispatch_from_host(cfg8, lay, 0x60000, 0x30000, None, 0x40000, None, None, 4,
                                    None) == ep.EP_ERR_INVALID_ARG
    assert ep.ep_combine_to_host(cfg, lay, 0x40000, None, 0x30000, None, 4,
                                 None) == ep.EP_ERR_INVALID_ARG
    assert ep.ep_combine_to_host(cfg, lay, 0x40000, None, None, 0x60000, 4,
                                 None) == ep.EP_ERR_INVALID_ARG
    # layout and dispatch in one call: the checks of both calls
    assert ep.ep_layout_and_dispatch(cfg, 4, None, lay, 0x30000, None, 0x40000, None, None,
                                     None) == ep.EP_ERR_INVALID_ARG          # no routes
    assert ep.ep_layout_and_dispatch(cfg, 4, 0x20000, lay, None, None, 0x40000, None, None,
                                     None) == ep.EP_ERR_INVALID_ARG          # no x
    assert ep.ep_layout_and_dispatch(cfg, 17, 0x20000, lay, 0x30000, None, 0x40000, None,
                                     None, None) == ep.EP_ERR_INVALID_ARG    # > max_tokens
    assert ep.ep_layout_and_dispatch(cfg8, 4, 0x20000, lay, 0x30000, None, 0x40000, None,
                                     None, None) == ep.EP_ERR_INVALID_ARG    # fp8, no scales
    assert ep.ep_layout_and_dispatch(cfg, 4, 0x20000, lay, 0x30000, None, 0x40000, None,
                                     0x50000, None) == ep.EP_ERR_INVALID_ARG  # recv_w, no w


@pytest.mark.skipif(_has_gpu(), reason="uses fake device addresses: host-only check")
def test_layout_timeout_selftest_arguments_checked(ep):
    """ep_selftest_layout_timeout validates its arguments before launching:
    the two-launch layout only, a stall CTA inside the assign grid, a limit in
    [1 us, 1 s]."""
    fake = [0x10000 + 0x100 * i for i in range(10)]
    lay = ep.EpLayout(*fake, None, None, None, 0, 0)
    big = ep.Config(4096, 128, 2, 8, 2, 4).c()       # 8192 pairs: 32 tiles, 32 CTAs
    small = ep.Config(4096, 128, 2, 8, 2, 4).c()
    call = lambda cfg, T, tile, ns: ep.ep_selftest_layout_timeout(cfg, T, 0x20000, lay, tile,
                                                                  ns, None)
    assert call(small, 2048, 0, 10_000) == ep.EP_ERR_INVALID_ARG   # 4096 pairs: one launch
    assert call(big, 0, 0, 10_000) == ep.EP_ERR_INVALID_ARG        # no tokens
    assert call(big, 4096, -1, 10_000) == ep.EP_ERR_INVALID_ARG
    assert call(big, 4096, 32, 10_000) == ep.EP_ERR_INVALID_ARG    # past the grid
    assert call(big, 4096, 0, 999) == ep.EP_ERR_INVALID_ARG
    assert call(big, 4096, 0, 10**9 + 1) == ep.EP_ERR_INVALID_ARG
    assert call(big, 4097, 0, 10_000) == ep.EP_ERR_INVALID_ARG     # > max_tokens


def test_status_strings(ep):
    assert ep.ep_status_str(0) == "EP_OK"
    assert ep.ep_status_str(ep.EP_ERR_TIMEOUT) == "EP_ERR_TIMEOUT"
    assert ep.ep_status_str(ep.EP_ERR_TIMEOUT_PENDING) == "EP_ERR_TIMEOUT_PENDING"
    assert ep.ep_status_str(99) == "EP_ERR_UNKNOWN"
