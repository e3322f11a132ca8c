"""User-facing API: run the whole ZETA hot path through the C ABI.

``ZetaPlan`` owns the device buffers of one problem size (codes, prefix table,
workspaces, outputs) so that repeated steps allocate nothing.  ``forward`` and
``backward`` enqueue the five library calls on the current stream;
``ZetaAttention`` wraps them as a torch.autograd.Function (selection is not
differentiated).  All arithmetic runs in the library's CUDA kernels.

With ``curves`` = 3 or 6 the plan follows the multi-curve variant (the keys
are indexed along the cyclic shifts, or all orderings, of the three
coordinates and every curve contributes k // curves keys): the codes and
prefix tables gain a leading curve dimension, one sort call covers every
curve, and the union of the windows feeds the same attend kernels.
"""
from __future__ import annotations

import torch

from . import binding as zb


class ZetaPlan:
    def __init__(self, p: zb.zeta_problem_t, device="cuda", backward: bool = True,
                 curves: int = 1, fused: bool = False):
        """fused: select and attend in one call (zeta_select_attend_fwd); one
        curve only."""
        if fused and curves != 1:
            raise ValueError("the fused select + attend call takes one curve")
        self.p = p
        self.curves = curves
        self.fused = fused
        self.axes = zb.curve_axes(p.d_K, curves)
        # Every curve's slices sort as one problem with curves*B batches.
        self.p_sort = zb.problem(p.B * curves, p.H, p.N, p.d_K, p.d_V, p.k, p.C, p.bits,
                                 p.v_dtype, flags=p.flags) if curves > 1 else p
        dev = torch.device(device)
        S = p.B * p.H
        N = p.N
        cdt = zb.code_dtype(p)
        vdt = zb.v_torch_dtype(p)
        T = zb.zeta_prefix_entries(p)
        if T < 0:
            raise zb.ZetaError("zeta_prefix_entries", 1)
        self.T = T
        G = curves * S
        self.q_codes = torch.empty(G * N, dtype=cdt, device=dev)
        self.k_codes = torch.empty(G * N, dtype=cdt, device=dev)
        self.prefix_codes = torch.empty(max(G * T, 1), dtype=cdt, device=dev)[: G * T]
        self.prefix_idx = torch.empty(max(G * T, 1), dtype=torch.int32, device=dev)[: G * T]
        self.sort_ws = torch.empty(max(zb.zeta_sort_workspace_bytes(self.p_sort), 256),
                                   dtype=torch.uint8, device=dev)
        self.idx = torch.empty(S * N * p.k, dtype=torch.int32, device=dev)
        self.out = torch.empty(S * N * p.d_V, dtype=vdt, device=dev)
        self.rowsum = torch.empty(S * N, dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.has_bwd = backward
        if backward:
            self.bwd_ws = torch.empty(max(zb.zeta_bwd_workspace_bytes(p), 256),
                                      dtype=torch.uint8, device=dev)
            self.dq = torch.empty(S * N * p.d_K, dtype=torch.float32, device=dev)
            self.dk = torch.empty(S * N * p.d_K, dtype=torch.float32, device=dev)
            self.dv = torch.empty(S * N * p.d_V, dtype=vdt, device=dev)
            self.dgamma = torch.empty(p.H, dtype=torch.float32, device=dev)

    def forward(self, q, k, v, gamma, stream=None):
        """Encode, sort, select, attend.  Returns (out, rowsum, idx) views."""
        p = self.p
        if self.curves == 1:
            zb.zeta_encode(p, q, self.q_codes, stream)
            zb.zeta_encode(p, k, self.k_codes, stream)
        else:
            zb.zeta_encode_curves(p, q, self.axes, self.q_codes, stream)
            zb.zeta_encode_curves(p, k, self.axes, self.k_codes, stream)
        zb.zeta_sort_chunks(self.p_sort, self.k_codes, self.prefix_codes, self.prefix_idx,
                            self.sort_ws, stream)
        if self.fused:
            zb.zeta_select_attend_fwd(p, q, k, v, gamma, self.q_codes, self.prefix_codes,
                                      self.prefix_idx, self.idx, self.out, self.rowsum,
                                      self.status, stream)
            return self.out, self.rowsum, self.idx
        if self.curves == 1:
            zb.zeta_select_topk(p, self.q_codes, self.prefix_codes, self.prefix_idx, self.idx,
                                stream)
        else:
            zb.zeta_select_topk_curves(p, self.curves, self.q_codes, self.prefix_codes,
                                       self.prefix_idx, self.idx, stream)
        zb.zeta_attend_fwd(p, q, k, v, gamma, self.idx, self.out, self.rowsum, self.status,
                           stream)
        return self.out, self.rowsum, self.idx

    def backward(self, q, k, v, gamma, dout, stream=None):
        """Gradients for the last forward.  Returns (dq, dk, dv, dgamma) views."""
        p = self.p
        zb.zeta_attend_bwd(p, q, k, v, gamma, self.idx, dout, self.dq, self.dk, self.dv,
                           self.dgamma, self.bwd_ws, self.status, stream)
        return self.dq, self.dk, self.dv, self.dgamma


class ZetaAttention(torch.autograd.Function):
    """out = ZETA attention(q, k, v, gamma); q, k [B,H,N,d_K] f32, v [B,H,N,d_V]."""

    @staticmethod
    def forward(ctx, q, k, v, gamma, C: int, k_sel: int, bits: int, curves: int = 1,
                weight: str = "cauchy"):
        B, H, N, d_K = q.shape
        d_V = v.shape[-1]
        vd = "bf16" if v.dtype == torch.bfloat16 else "f32"
        p = zb.problem(B, H, N, d_K, d_V, k_sel, C, bits, vd, weight=weight)
        plan = ZetaPlan(p, q.device, curves=curves)
        q, k, v, gamma = (t.contiguous() for t in (q, k, v, gamma))
        out, _, _ = plan.forward(q, k, v, gamma)
        ctx.plan = plan
        ctx.save_for_backward(q, k, v, gamma)
        return out.view(B, H, N, d_V).clone()

    @staticmethod
    def backward(ctx, dout):
        q, k, v, gamma = ctx.saved_tensors
        dq, dk, dv, dg = ctx.plan.backward(q, k, v, gamma, dout.contiguous().to(v.dtype))
        return (dq.view_as(q).clone(), dk.view_as(k).clone(), dv.view_as(v).clone(),
                dg.clone(), None, None, None, None, None)


def zeta_attention(q, k, v, gamma, C: int, k_sel: int, bits: int = 10, curves: int = 1,
                   weight: str = "cauchy"):
    """weight: 'cauchy' (the method), 'softmax' (of -|q-k|^2/gamma^2) or
    'inv_euclid' (1/|q-k|); see zeta_weight_t in include/zeta.h."""
    return ZetaAttention.apply(q, k, v, gamma, C, k_sel, bits, curves, weight)
