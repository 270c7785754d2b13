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
from ._lib import (GrpoError, Problem, advantages, device_status, loss_bwd, loss_bwd_e4m3,
                   loss_fwd, loss_fwd_e4m3, make_problem, profile_collect, profile_enable,
                   quantize_e4m3_rows, workspace_size)

__all__ = ["GrpoError", "Problem", "advantages", "device_status", "loss_bwd", "loss_bwd_e4m3",
           "loss_fwd", "loss_fwd_e4m3", "make_problem", "profile_collect", "profile_enable",
           "quantize_e4m3_rows", "workspace_size", "GRPOLoss", "grpo_loss"]


_CTRL_BYTES = 256  # control block at the start of every workspace (error word, counts)


class GRPOLoss:
    """Owns the workspaces of one problem shape and runs the library calls.

    ``forward`` returns (loss, kl_mean, logp_pol, logp_ref) as CUDA tensors;
    ``backward`` returns dH_pol (and fills ``self.dW``, float32 [V, d], when
    built with ``compute_dW``). Buffers are allocated once with torch and
    reused across calls.

    With ``dtype=torch.float8_e4m3fn`` the engine takes float32 or bf16 H_pol,
    H_ref and W, quantizes them row-wise to e4m3 with the library's quantizer
    and runs the e4m3 problem; dH is then bf16. The backward reuses the
    forward's quantized H_pol and W while those tensors are unchanged (same
    storage and version counter).
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
        # every call clears its workspace's control block (the device error
        # word) first; clear both now, so check() before a backward has run
        # does not read stale bytes from the allocator's cache
        self.ws_fwd[:_CTRL_BYTES].zero_()
        self.ws_bwd[:_CTRL_BYTES].zero_()
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
        self.e4m3 = dtype == torch.float8_e4m3fn
        if self.e4m3:
            u8, f32 = torch.uint8, torch.float32
            self.q_pol = torch.empty(N, d, dtype=u8, device=dev)
            self.s_pol = torch.empty(N, dtype=f32, device=dev)
            self.q_ref = None if ref_logp_given else torch.empty(N, d, dtype=u8, device=dev)
            self.s_ref = None if ref_logp_given else torch.empty(N, dtype=f32, device=dev)
            self.q_W = torch.empty(V, d, dtype=u8, device=dev)
            self.s_W = torch.empty(V, dtype=f32, device=dev)
            self._quantized = None  # (H_pol, W) identities the codes were made from

    @staticmethod
    def _ident(t):
        return (t.data_ptr(), t._version, tuple(t.shape), t.dtype)

    def _quantize(self, H_pol, W):
        quantize_e4m3_rows(H_pol, self.q_pol, self.s_pol)
        quantize_e4m3_rows(W, self.q_W, self.s_W)
        self._quantized = (self._ident(H_pol), self._ident(W))

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
        if self.e4m3:
            self._quantize(H_pol, W)
            if H_ref is not None and self.q_ref is not None:
                quantize_e4m3_rows(H_ref, self.q_ref, self.s_ref)
            loss_fwd_e4m3(self.problem, self.q_pol, self.s_pol, self.q_ref, self.s_ref, self.q_W,
                          self.s_W, ids, mask, adv, self.logp_pol, self.logp_ref, self.lse_pol,
                          self.loss, self.kl_mean, self.ws_fwd)
        else:
            loss_fwd(self.problem, H_pol, H_ref, W, ids, mask, adv, self.logp_pol, self.logp_ref,
                     self.lse_pol, self.loss, self.kl_mean, self.ws_fwd)
        return self.loss, self.kl_mean, self.logp_pol, self.logp_ref

    def backward(self, H_pol, W, ids, mask, adv, grad_loss: float = 1.0, dH=None):
        if dH is None:
            if self.dH is None:
                self.dH = (torch.empty(H_pol.shape, dtype=torch.bfloat16, device=H_pol.device)
                           if self.e4m3 else torch.empty_like(H_pol))
            dH = self.dH
        if self.e4m3:
            if self._quantized != (self._ident(H_pol), self._ident(W)):
                self._quantize(H_pol, W)
            loss_bwd_e4m3(self.problem, self.q_pol, self.s_pol, self.q_W, self.s_W, ids, mask,
                          adv, self.logp_pol, self.logp_ref, self.lse_pol, grad_loss, dH,
                          self.ws_bwd, dW=self.dW)
        else:
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
        eng = ctx.engine
        dH = eng.backward(H_pol, W, ids, mask, adv, float(g_loss),
                          dH=torch.empty(H_pol.shape, dtype=torch.bfloat16, device=H_pol.device)
                          if eng.e4m3 else torch.empty_like(H_pol))
        dH = dH.to(H_pol.dtype)
        dW = ctx.engine.dW.to(W.dtype) if ctx.engine.dW is not None else None
        return dH, None, dW, None, None, None, None


def grpo_loss(H_pol, H_ref, W, ids, mask, adv, engine: GRPOLoss):
    """Autograd entry: returns (loss, kl_mean); backward gives the gradient
    of the loss with respect to H_pol, and with respect to W when the engine
    was built with ``compute_dW`` (the reference model is frozen; kl_mean is a
    metric and carries no gradient)."""
    return _GRPOLossFn.apply(H_pol, H_ref, W, ids, mask, adv, engine)
