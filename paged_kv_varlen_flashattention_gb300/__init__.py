"""GB300-native paged-KV varlen flash-attention (forward).

The compute path is the C-ABI library built from ``csrc/`` (hand-written sm_103a
kernels); :mod:`.binding` marshals torch tensors into its descriptors.  Importing
this package does not load the library; the first call does, and raises if the
library is missing.
"""
from .binding import varlen_fwd, last_error, device_status, library_path, kernel_launches, PaError  # noqa: F401

__all__ = ["varlen_fwd", "last_error", "device_status", "library_path", "kernel_launches", "PaError"]
