"""Host-side choices of the benchmark, on CPU: how its end-to-end leg moves
the rows between host and device."""

import pytest

import bench


@pytest.mark.parametrize("requested,device_only,want", [
    ("auto", False, "direct"),
    ("direct", False, "direct"),
    ("chunked", False, "chunked"),
    ("copies", False, "copies"),
    # the combine epilogue and the FP8 input options have device entry points only
    ("auto", True, "copies"),
    ("direct", True, "copies"),
    ("chunked", True, "copies"),
])
def test_e2e_transfer_choice(requested, device_only, want):
    assert bench.e2e_transfer(requested, device_only) == want


def test_e2e_transfer_rejects_unknown_mode():
    with pytest.raises(ValueError):
        bench.e2e_transfer("zero-copy", False)


def test_e2e_transfer_flag_choices_are_all_handled():
    import sys

    argv = sys.argv
    try:
        for mode in ("auto", "direct", "chunked", "copies"):
            sys.argv = ["bench.py", "--e2e-transfer", mode]
            args = bench.parse_args()
            assert bench.e2e_transfer(args.e2e_transfer, False) in ("direct", "chunked",
                                                                    "copies")
    finally:
        sys.argv = argv


def test_path_dtype_follows_the_workload():
    import workloads

    assert bench.path_dtype(workloads.WORKLOADS["prefill"]) == "bf16"
    for name in ("decode", "skew", "sweep16k_fp8"):
        assert bench.path_dtype(workloads.WORKLOADS[name]) == "fp8_e4m3"


def test_cpu_baseline_reports_all_cores_and_one():
    """The CPU baseline times the oracle on every core it may use and on one
    thread, on a bounded sample of the same workload."""
    import workloads

    wl = workloads.WORKLOADS["tiny"]
    inp = workloads.make_inputs(wl, seed=0)
    cb = bench.cpu_baseline(wl, inp, 0.2)
    assert cb["cores"] == bench.host_cores() >= 1
    assert cb["kind"] == "oracle" and cb["unit"] == "tokens/s" and cb["value"] > 0
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0


@pytest.mark.parametrize("requested,device_only,row_bytes,want", [
    ("auto", False, 4096 * 7168 * 2, "chunked"),    # prefill rows: 58.7 MB
    ("auto", False, 128 * 7168 * 2, "direct"),      # decode rows: 1.8 MB
    ("auto", False, 8 << 20, "chunked"),            # exactly two 4 MiB chunks
    ("auto", False, (8 << 20) - 2, "direct"),
    ("copies", False, 128, "copies"),
    ("direct", False, 1 << 30, "direct"),
    ("auto", True, 1 << 30, None),                  # device entry points only
])
def test_pipelined_transfer_choice(requested, device_only, row_bytes, want):
    assert bench.pipelined_transfer(requested, device_only, row_bytes) == want


@pytest.mark.parametrize("requested,row_bytes,want", [
    (0, 4096 * 7168 * 2, 2),        # prefill: two chunks of 29 MB
    (0, 16384 * 7168 * 2, 4),       # 16K tokens: four of 59 MB
    (0, 8 << 20, 2),                # never fewer than two
    (0, 1 << 34, 8),                # never more than eight
    (6, 4096 * 7168 * 2, 6),        # an explicit count stands
])
def test_e2e_chunk_count(requested, row_bytes, want):
    assert bench.e2e_chunk_count(requested, row_bytes) == want


def test_e2e_headline_takes_the_faster_leg():
    seq = {"value": 2.0, "ms_per_step": 1.0, "transfer": "direct"}
    pip = {"value": 3.0, "ms_per_step": 0.5, "transfer": "chunked", "pipelining": "4 in flight",
           "launch": "graph"}
    h = bench.e2e_headline(seq, pip)
    assert (h["value"], h["mode"], h["transfer"], h["launch"]) == (3.0, "pipelined", "chunked",
                                                                   "graph")
    h = bench.e2e_headline(seq, dict(pip, value=1.0))
    assert (h["value"], h["mode"], h["transfer"], h["pipelining"]) == (2.0, "sequential",
                                                                       "direct", None)
    h = bench.e2e_headline(seq, None)      # options with device entry points only
    assert h["mode"] == "sequential" and h["ms_per_step"] == 1.0
