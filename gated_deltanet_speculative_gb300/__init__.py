"""GB300-native gated-DeltaNet speculative verify path.

The C ABI of include/gdn.h (libgdn.so, hand-written sm_103a kernels) behind a
thin ctypes binding: ``step``, ``window``, ``tree``, ``commit``,
``prefill`` and ``get_device_error`` take torch CUDA tensors and enqueue on the current
stream.  ``synth`` draws the seeded synthetic inputs.  Importing the package
does not load the CUDA library; the first call does (and raises if it is
missing).
"""
from . import synth  # noqa: F401
from ._binding import (Dims, GdnError, MAX_WINDOW, PREFILL_CHUNK, commit, commit_replay,  # noqa: F401
                       get_device_error, library_path, load, prefill, prefill_workspace_size, step, tree,
                       window, window_log)
