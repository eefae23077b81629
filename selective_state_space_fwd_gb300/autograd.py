"""The selective scan as a differentiable PyTorch function.

``selective_scan`` runs the library's forward (``scan_fwd``), keeping the
chunk boundary states the backward replays from, and its backward
(``scan_bwd``) when autograd asks for gradients: the recompute scheme of [P1]
s3.4 (only the chunk states are stored between the two passes).  This module
only passes tensors between PyTorch and the C ABI; every step of both passes
runs in the library's kernels.
"""
import torch

from ._binding import scan_bwd, scan_fwd


class _SelectiveScan(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, delta, A, B, C, D, z, valid_len, h0, chunk_len):
        y, states = scan_fwd(x, delta, A, B, C, D, z, valid_len, chunk_len=chunk_len, h0=h0)
        ctx.save_for_backward(x, delta, A, B, C, D, z, valid_len, h0, states)
        ctx.chunk_len = chunk_len
        return y

    @staticmethod
    def backward(ctx, dy):
        x, delta, A, B, C, D, z, valid_len, h0, states = ctx.saved_tensors
        want_dh0 = h0 is not None and ctx.needs_input_grad[8]
        g = scan_bwd(x, delta, A, B, C, D, z, valid_len, chunk_states=states,
                     chunk_len=ctx.chunk_len, dy=dy.contiguous(), h0=h0, want_dh0=want_dh0)
        # B and C share the I/O dtype; their gradients are summed in fp32
        dB = g["dB"].to(B.dtype)
        dC = g["dC"].to(C.dtype)
        return (g["dx"], g["ddelta"], g["dA"], dB, dC, g["dD"], g["dz"], None,
                g["dh0"] if want_dh0 else None, None)


def selective_scan(x, delta, A, B, C, D=None, z=None, valid_len=None, *, h0=None,
                   chunk_len: int = 256):
    """y = the selective scan of the inputs (as ``scan_fwd``), differentiable in
    x, delta, A, B, C, D, z and h0.  ``chunk_len`` (1 .. 512) is the spacing of
    the boundary states kept for the backward: a multiple of 16 lets the
    backward take its tiled kernel."""
    return _SelectiveScan.apply(x, delta, A, B, C, D, z, valid_len, h0, int(chunk_len))
