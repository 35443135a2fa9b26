"""torch.autograd wrapper of the scan: the forward calls mamba_scan_fwd (or
mamba_scan_fwd_ex with an initial state), the backward calls
mamba_scan_bwd.  Argument marshalling only: every computation runs in the
library's kernels, and the backward recomputes the states from the saved
inputs instead of keeping them."""

from __future__ import annotations

from . import _lib


def _torch():
    import torch
    return torch


class _ScanFn:
    """Built lazily so that importing the package does not import torch."""
    cls = None

    @classmethod
    def get(cls):
        if cls.cls is not None:
            return cls.cls
        torch = _torch()

        class ScanFunction(torch.autograd.Function):
            @staticmethod
            def forward(ctx, u, delta, dt_bias, A, B, C, D_skip, z, initial_state, softplus,
                        want_final):
                batch, dim, _ = u.shape
                N = A.shape[1]
                final = torch.empty((batch, dim, N), dtype=torch.float32, device=u.device)
                if initial_state is None:
                    y = _lib.mamba_scan_fwd(u, delta, dt_bias, A, B, C, D_skip, z, softplus,
                                            final_state=final)
                else:
                    y = _lib.mamba_scan_fwd_ex(u, delta, dt_bias, A, B, C, D_skip, z,
                                               softplus=softplus, initial_state=initial_state,
                                               final_state=final)
                ctx.save_for_backward(u, delta, dt_bias, A, B, C, D_skip, z, initial_state)
                ctx.softplus = softplus
                ctx.want_final = want_final
                if want_final:
                    return y, final
                ctx.mark_non_differentiable(final)
                return y, final

            @staticmethod
            @torch.autograd.function.once_differentiable
            def backward(ctx, dy, dfinal):
                u, delta, dt_bias, A, B, C, D_skip, z, h0 = ctx.saved_tensors
                if dy is None:
                    dy = torch.zeros_like(u)
                dy = dy.contiguous()
                dfin = dfinal.contiguous() if (ctx.want_final and dfinal is not None) else None
                g = _lib.mamba_scan_bwd(u, delta, dt_bias, A, B, C, D_skip, z, dy,
                                        softplus=ctx.softplus, initial_state=h0,
                                        d_final_state=dfin,
                                        want_initial_state_grad=h0 is not None)
                need = ctx.needs_input_grad
                pick = lambda i, t, like: (t.to(like.dtype) if need[i] and t is not None else None)
                return (pick(0, g["du"], u), pick(1, g["ddelta"], delta),
                        pick(2, g["ddt_bias"], dt_bias) if dt_bias is not None else None,
                        pick(3, g["dA"], A), pick(4, g["dB"], B), pick(5, g["dC"], C),
                        pick(6, g["dD_skip"], D_skip) if D_skip is not None else None,
                        pick(7, g["dz"], z) if z is not None else None,
                        pick(8, g["d_initial_state"], h0) if h0 is not None else None,
                        None, None)

        cls.cls = ScanFunction
        return ScanFunction


def mamba_scan_fn(u, delta, A, B, C, D_skip=None, z=None, dt_bias=None, softplus: bool = True,
                  initial_state=None, return_final_state: bool = False):
    """Differentiable selective scan (Euler input term).  Shapes and dtypes as
    in mamba_scan_fwd: u, delta, z (batch, dim, L); B, C (batch, N, L); A
    (dim, N) fp32; D_skip, dt_bias (dim,) fp32 or None; initial_state
    (batch, dim, N) fp32 or None.  Returns y, or (y, final_state)."""
    y, final = _ScanFn.get().apply(u, delta, dt_bias, A, B, C, D_skip, z, initial_state,
                                   bool(softplus), bool(return_final_state))
    return (y, final) if return_final_state else y
