"""The instrumented variants of the library still compile (no GPU needed): the
timeline build (-DMHCPB_TRACE, per-stage time stamps read by
mhcpb_debug_trace) and the bounds-checked build (-DMHCPB_CHECKED, see
mhcpb_debug_checked_sites).  Each is built into its own directory, never
over the product library, and exports its debug entry point."""
import ctypes
import os

import pytest

from rms_backward_gb300 import build as B


@pytest.mark.parametrize("define,symbol", [("-DMHCPB_TRACE", "mhcpb_debug_trace"),
                                           ("-DMHCPB_CHECKED", "mhcpb_debug_checked_sites")])
def test_instrumented_build(tmp_path, define, symbol):
    try:
        lib = B.build(extra_flags=[define], out_dir=str(tmp_path))
    except RuntimeError as e:  # pragma: no cover
        if "nvcc not found" in str(e):
            pytest.skip(str(e))
        raise
    assert os.path.dirname(lib) == str(tmp_path) and lib != B.LIB
    handle = ctypes.CDLL(lib)
    assert hasattr(handle, symbol)
    assert hasattr(handle, "mhcpb_execute")


def test_instrumented_build_needs_its_own_directory():
    with pytest.raises(ValueError):
        B.build(extra_flags=["-DMHCPB_CHECKED"])
