"""GB300-native Mamba-2 SSD (selective state space) forward pass and decode step.

The computation lives in libssd.so (hand-written CUDA for sm_103a, C ABI in
include/ssd.h); this package builds it (``build``), loads it (``_native``) and
offers a thin torch binding (``api``).  ``workloads`` draws seeded synthetic
inputs.  Importing the package does not load the CUDA library; the first call
into ``api`` does, and fails loudly if the library is missing.
"""

def __getattr__(name):
    if name in ("ssd_fwd", "ssd_step", "ssd_chunk_cumsum", "ssd_chunk_state", "ssd_state_passing",
                "ssd_chunk_scan", "workspace_size", "make_desc", "desc_for"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
