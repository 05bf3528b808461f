"""GB300-native chunked gated-delta-rule forward and backward passes.

The compute path is a C-ABI CUDA library (``include/gdr.h``, built in-tree
into ``_build/libgdr.so``); this package is its thin ctypes binding plus the
seeded synthetic input generator, and ``chunk_gated_delta_rule``, a torch
autograd function over the library's forward and backward entry points.
There is no CPU fallback: every entry point raises if the CUDA library is
missing.
"""
from .api import (GdrError, LaunchTimer, gdr_chunk_fwd, gdr_chunk_fwd_host,  # noqa: F401
                  gdr_chunk_bwd, gdr_bwd_workspace_size,
                  gdr_chunk_fwd_noalloc, gdr_recurrent_fwd,
                  gdr_error_string, gdr_kernel_name, gdr_plan_query, gdr_release_cached,
                  gdr_version,
                  gdr_workspace_size, load_library)

from .autograd import chunk_gated_delta_rule  # noqa: F401,E402

# gdr_chunk_fwd_ex's options (scale, forced plan, workspace, status word) are
# keyword arguments of gdr_chunk_fwd in Python.
gdr_chunk_fwd_ex = gdr_chunk_fwd
