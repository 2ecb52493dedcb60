"""libgdr: the chunked gated-delta-rule forward on one GB300 (sm_103a).

The compute path is the C-ABI shared library built from csrc/ (see include/gdr.h);
`gdr` is its thin ctypes binding.  Importing this package loads nothing: the
library is loaded on the first call, and a missing library raises.
"""
from .gdr import (GdrError, forward, gdr_chunk_output, gdr_forward, gdr_forward_workspace_bytes,  # noqa: F401
                  gdr_get_device_status, gdr_last_variant, gdr_prepare_wy, gdr_prepare_wyp, gdr_scan_h, gdr_scan_output, gdr_status_string,
                  gdr_version, make_problem, problem_for)
