"""torch.autograd binding: the chunked SSD forward pass with its gradient pass.

``ssd_chunked(x, dt, A, B, C, D, chunk, h0)`` returns (y, h_final) like ``api.ssd_fwd``;
autograd then differentiates through it with ``api.ssd_bwd`` (the C ABI's gradient
pass).  Both directions run in libssd.so; this module only saves the inputs and maps
the gradients back to them.  The gradient pass needs the output dtype equal to the
input dtype, so the forward pass here always writes y in the input dtype.
"""
from __future__ import annotations

import torch

from . import api


class SSDChunked(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, dt, A, B, C, D, h0, chunk):
        y, h_final = api.ssd_fwd(x, dt, A, B, C, D, chunk, h0)
        ctx.chunk = chunk
        ctx.save_for_backward(x, dt, A, B, C, D, h0)
        return y, h_final

    @staticmethod
    def backward(ctx, dy, dh_final):
        x, dt, A, B, C, D, h0 = ctx.saved_tensors
        dy = torch.zeros_like(x) if dy is None else dy.to(x.dtype).contiguous()
        dh_final = None if dh_final is None else dh_final.to(torch.float32).contiguous()
        g = api.ssd_bwd(x, dt, A, B, C, D, dy, ctx.chunk, h0, dh_final, want_dh0=h0 is not None)
        return g["dx"], g["ddt"], g["dA"], g["dB"], g["dC"], g["dD"], g["dh0"], None


def ssd_chunked(x, dt, A, B, C, D, chunk: int, h0=None):
    """Differentiable chunked SSD forward pass: (y, h_final).  Layouts as in ``api.ssd_fwd``."""
    return SSDChunked.apply(x, dt, A, B, C, D, h0, chunk)
