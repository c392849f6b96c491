"""The C-ABI library loads on a machine without a GPU and exports every symbol that
include/*.h declares (no compute call is made here)."""
import ctypes
import glob
import os
import re

from paged_kv_varlen_flashattention_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(pa_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_entry_points():
    names = declared_symbols()
    assert {"pa_varlen_fwd", "pa_varlen_check", "pa_last_error", "pa_device_status", "pa_version",
            "pa_kernel_launches"} <= names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(binding.library_path())
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_version_and_empty_error():
    lib = binding.load()
    assert lib.pa_version() >= 100
    assert isinstance(lib.pa_last_error(), bytes)


def test_kernel_timing_record_starts_empty():
    """With nothing launched, the per-kernel timing record reads as zeros, and a null
    output array is an argument error (no CUDA call is made on either path)."""
    assert "pa_kernel_times" in declared_symbols() and "pa_kernel_timing" in declared_symbols()
    assert binding.kernel_times() == {name: (0.0, 0) for name in binding.KERNEL_CLASSES}
    lib = binding.load()
    assert lib.pa_kernel_times(None, None) == 10  # PA_ERR_ARG
    assert b"null" in lib.pa_last_error()
