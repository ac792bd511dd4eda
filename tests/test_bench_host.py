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
