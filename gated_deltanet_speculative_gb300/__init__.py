"""GB300-native gated-DeltaNet speculative verify path.

The C ABI of include/gdn.h (libgdn.so, hand-written sm_103a kernels) behind a
thin ctypes binding: ``step``, ``step_ex``, ``window``, ``tree``, ``commit``,
``window_log``, ``commit_replay``, ``tree_log``, ``commit_replay_tree``,
``window_pooled``, ``tree_pooled``, ``commit_swap``,
``prefill``, ``prefill_noalloc`` and ``get_device_error`` take torch CUDA tensors and enqueue on the current
stream; ``prepare`` checks and marshals one such call's arguments once and
returns a callable that enqueues it again.  ``synth`` draws the seeded synthetic inputs.  Importing the package
does not load the CUDA library; the first call does (and raises if it is
missing).
"""
from . import synth  # noqa: F401
from ._binding import (STEP_EARLY_STATE, Dims, GdnError, MAX_WINDOW, PREFILL_CHUNK,  # noqa: F401
                       PREFILL_NOALLOC_SCRATCH_BYTES,
                       commit, commit_replay, commit_replay_tree, commit_swap, debug_wait_timeout, get_device_error,
                       library_path, load, prefill, prepare, PreparedCall,
                       prefill_noalloc, prefill_workspace, prefill_workspace_size, step, step_ex, tree, tree_log, tree_pooled,
                       window, window_log, window_pooled)
