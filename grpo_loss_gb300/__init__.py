"""GB300-native memory-efficient GRPO loss.

The fused lm_head projection, log-softmax and GRPO objective (reverse-KL
estimator plus the exp(q - q.detach()) * A advantage term) over the
flattened token axis, in hand-written sm_103a CUDA kernels behind the C ABI
of include/grpo.h. Importing the package does not load the library; the
first call does, and raises if it has not been built.
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import (GrpoError, Problem, advantages, device_status, loss_bwd, loss_fwd,
                   make_problem, profile_collect, profile_enable, workspace_size)

__all__ = ["GrpoError", "Problem", "advantages", "device_status", "loss_bwd", "loss_fwd",
           "make_problem", "profile_collect", "profile_enable", "workspace_size", "GRPOLoss",
           "grpo_loss"]


class GRPOLoss:
    """Owns the workspaces of one problem shape and runs the library calls.

    ``forward`` returns (loss, kl_mean, logp_pol, logp_ref) as CUDA tensors;
    ``backward`` returns dH_pol (and fills ``self.dW``, float32 [V, d], when
    built with ``compute_dW``). Buffers are allocated once with torch and
    reused across calls.
    """

    def __init__(self, num_seqs: int, seq_len: int, d: int, V: int, group_size: int,
                 beta: float = 0.04, eps: float = 1e-4, std_unbiased: int = 1,
                 chunk_rows: int = 0, dtype=torch.bfloat16, device="cuda",
                 compute_dW: bool = False, token_level: bool = False,
                 logit_multiply: float = 0.0, logit_divide: float = 0.0, softcap: float = 0.0,
                 temperature: float = 0.0, ref_logp_given: bool = False, kl_mode: int = 0,
                 cluster_mode: int = 0):
        self.problem = make_problem(num_seqs, seq_len, d, V, group_size, beta, eps,
                                    std_unbiased, chunk_rows, dtype, compute_dW, token_level,
                                    logit_multiply, logit_divide, softcap, temperature,
                                    ref_logp_given, kl_mode, cluster_mode)
        fwd_b, bwd_b = workspace_size(self.problem)
        dev = torch.device(device)
        self.ws_fwd = torch.empty(fwd_b, dtype=torch.uint8, device=dev)
        self.ws_bwd = torch.empty(bwd_b, dtype=torch.uint8, device=dev)
        N = num_seqs * seq_len
        self.adv = torch.empty(num_seqs, dtype=torch.float32, device=dev)
        self.logp_pol = torch.empty(N, dtype=torch.float32, device=dev)
        self.logp_ref = torch.empty(N, dtype=torch.float32, device=dev)
        self.lse_pol = torch.empty(N, dtype=torch.float32, device=dev)
        self.loss = torch.empty(1, dtype=torch.float32, device=dev)
        self.kl_mean = torch.empty(1, dtype=torch.float32, device=dev)
        self.dtype = dtype
        self.dH = None
        self.dW = (torch.empty(V, d, dtype=torch.float32, device=dev) if compute_dW else None)

    def advantages(self, rewards: torch.Tensor) -> torch.Tensor:
        p = self.problem
        return advantages(rewards, p.group_size, p.eps, p.std_unbiased, self.adv)

    def forward(self, H_pol, H_ref, W, ids, mask, adv, logp_ref=None):
        """With ``ref_logp_given`` pass H_ref=None and the reference log-probs
        as ``logp_ref`` (float32 [N]); they are copied into the engine."""
        if self.problem.ref_logp_given:
            if logp_ref is None:
                raise ValueError("ref_logp_given needs logp_ref")
            self.logp_ref.copy_(logp_ref)
        loss_fwd(self.problem, H_pol, H_ref, W, ids, mask, adv, self.logp_pol, self.logp_ref,
                 self.lse_pol, self.loss, self.kl_mean, self.ws_fwd)
        return self.loss, self.kl_mean, self.logp_pol, self.logp_ref

    def backward(self, H_pol, W, ids, mask, adv, grad_loss: float = 1.0, dH=None):
        if dH is None:
            if self.dH is None:
                self.dH = torch.empty_like(H_pol)
            dH = self.dH
        loss_bwd(self.problem, H_pol, W, ids, mask, adv, self.logp_pol, self.logp_ref,
                 self.lse_pol, grad_loss, dH, self.ws_bwd, dW=self.dW)
        return dH

    def check(self) -> None:
        """Raise if a kernel of the last calls recorded a device error."""
        for ws in (self.ws_fwd, self.ws_bwd):
            st = device_status(ws)
            if st != 0:
                raise GrpoError(st, "device")


class _GRPOLossFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, H_pol, H_ref, W, ids, mask, adv, engine):
        loss, kl_mean, _, _ = engine.forward(H_pol, H_ref, W, ids, mask, adv)
        ctx.engine = engine
        ctx.save_for_backward(H_pol, W, ids, mask, adv)
        return loss.clone().reshape(()), kl_mean.clone().reshape(())

    @staticmethod
    def backward(ctx, g_loss, g_kl):
        H_pol, W, ids, mask, adv = ctx.saved_tensors
        # the upstream gradient is read on the host: one scalar per backward
        dH = ctx.engine.backward(H_pol, W, ids, mask, adv, float(g_loss), dH=torch.empty_like(H_pol))
        dW = ctx.engine.dW.to(W.dtype) if ctx.engine.dW is not None else None
        return dH, None, dW, None, None, None, None


def grpo_loss(H_pol, H_ref, W, ids, mask, adv, engine: GRPOLoss):
    """Autograd entry: returns (loss, kl_mean); backward gives the gradient
    of the loss with respect to H_pol, and with respect to W when the engine
    was built with ``compute_dW`` (the reference model is frozen; kl_mean is a
    metric and carries no gradient)."""
    return _GRPOLossFn.apply(H_pol, H_ref, W, ids, mask, adv, engine)
