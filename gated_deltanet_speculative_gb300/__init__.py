"""GB300-native gated-DeltaNet speculative verify path.

The C ABI of include/gdn.h (libgdn.so, hand-written sm_103a kernels) behind a
thin ctypes binding: ``step``, ``window``, ``tree``, ``commit`` and
``get_device_error`` take torch CUDA tensors and enqueue on the current
stream.  ``synth`` draws the seeded synthetic inputs.  Importing the package
does not load the CUDA library; the first call does (and raises if it is
missing).
"""
from . import synth  # noqa: F401
from ._binding import (Dims, GdnError, MAX_WINDOW, commit, get_device_error, load,  # noqa: F401
                       library_path, step, tree, window)
