"""GB300-native Mamba-2 SSD (selective state space) forward pass and decode step.

The computation lives in libssd.so (hand-written CUDA for sm_103a, C ABI in
include/ssd.h); this package builds it (``build``), loads it (``_native``) and
offers a thin torch binding (``api``) and its autograd form (``autograd``:
the forward pass with the gradient pass behind it).  ``workloads`` draws seeded
synthetic inputs.  Importing the package does not load the CUDA library; the first call
into ``api`` does, and fails loudly if the library is missing.
"""

def __getattr__(name):
    if name in ("ssd_fwd", "ssd_step", "ssd_chunk_cumsum", "ssd_chunk_state", "ssd_state_passing",
                "ssd_chunk_scan", "workspace_size", "make_desc", "desc_for", "ssd_bwd", "s6_fwd"):
        from . import api
        return getattr(api, name)
    if name == "ssd_chunked":
        from . import autograd
        return autograd.ssd_chunked
    raise AttributeError(name)
