"""torch.autograd wrapper of the scan: the forward calls mamba_scan_fwd (or
mamba_scan_fwd_ex with an initial state), the backward calls
mamba_scan_bwd.  Argument marshalling only: every computation runs in the
library's kernels, and the backward recomputes the states from the saved
inputs instead of keeping them.  With keep_checkpoints the forward is
mamba_scan_fwd_train, which also keeps the state every 12 steps (about 2.7
times the bytes of one bf16 input at dstate 16), and the backward
mamba_scan_bwd_ckpt starts from them instead of recomputing them."""

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
                        want_final, keep_checkpoints):
                batch, dim, _ = u.shape
                N = A.shape[1]
                final = torch.empty((batch, dim, N), dtype=torch.float32, device=u.device)
                ckpt = None
                if keep_checkpoints and any(ctx.needs_input_grad):
                    y, ckpt = _lib.mamba_scan_fwd_train(u, delta, dt_bias, A, B, C, D_skip, z,
                                                        softplus=softplus,
                                                        initial_state=initial_state,
                                                        final_state=final)
                elif initial_state is None:
                    y = _lib.mamba_scan_fwd(u, delta, dt_bias, A, B, C, D_skip, z, softplus,
                                            final_state=final)
                else:
                    y = _lib.mamba_scan_fwd_ex(u, delta, dt_bias, A, B, C, D_skip, z,
                                               softplus=softplus, initial_state=initial_state,
                                               final_state=final)
                ctx.save_for_backward(u, delta, dt_bias, A, B, C, D_skip, z, initial_state, ckpt)
                ctx.softplus = softplus
                ctx.want_final = want_final
                if want_final:
                    return y, final
                ctx.mark_non_differentiable(final)
                return y, final

            @staticmethod
            @torch.autograd.function.once_differentiable
            def backward(ctx, dy, dfinal):
                u, delta, dt_bias, A, B, C, D_skip, z, h0, ckpt = ctx.saved_tensors
                if dy is None:
                    dy = torch.zeros_like(u)
                dy = dy.contiguous()
                dfin = dfinal.contiguous() if (ctx.want_final and dfinal is not None) else None
                if ckpt is not None:
                    g = _lib.mamba_scan_bwd_ckpt(u, delta, dt_bias, A, B, C, D_skip, z, dy, ckpt,
                                                 softplus=ctx.softplus, d_final_state=dfin,
                                                 want_initial_state_grad=h0 is not None)
                else:
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
                        None, None, None)

        cls.cls = ScanFunction
        return ScanFunction


def mamba_scan_fn(u, delta, A, B, C, D_skip=None, z=None, dt_bias=None, softplus: bool = True,
                  initial_state=None, return_final_state: bool = False,
                  keep_checkpoints: bool = False):
    """Differentiable selective scan (Euler input term).  Shapes and dtypes as
    in mamba_scan_fwd: u, delta, z (batch, dim, L); B, C (batch, N, L); A
    (dim, N) fp32; D_skip, dt_bias (dim,) fp32 or None; initial_state
    (batch, dim, N) fp32 or None.  keep_checkpoints trades memory for the
    backward's checkpoint pass (see the module docstring).  Returns y, or
    (y, final_state)."""
    y, final = _ScanFn.get().apply(u, delta, dt_bias, A, B, C, D_skip, z, initial_state,
                                   bool(softplus), bool(return_final_state),
                                   bool(keep_checkpoints))
    return (y, final) if return_final_state else y
