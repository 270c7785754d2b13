"""Shared helpers of the GPU parity tests: run the CUDA path through the C
ABI on host inputs, and compare against the float64 oracle."""
from __future__ import annotations

import numpy as np
import torch

from grpo_loss_gb300 import workloads as WL

# Tolerances of the parity bar (relative): advantages, log-probs, loss and
# kl_mean 1e-3; dH 2e-2 in relative L2 norm (bf16 operands, fp32 accumulation).
TOL_REL = 1e-3
TOL_DH_L2 = 2e-2


def torch_dtype(w: WL.Workload):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def oracle_adv(w: WL.Workload, inp) -> np.ndarray:
    from oracle import grpo_oracle as O
    if w.supplied_adv:
        return inp["adv"].double().numpy()
    return O.advantages(inp["rewards"], w.G, w.eps, w.std_unbiased)


def gpu_run(w: WL.Workload, inp, adv32: torch.Tensor, chunk_rows: int = 0, beta=None,
            grad: float = 1.0, H_ref=None, ids=None, mask=None, want_bwd: bool = True,
            check: bool = True, want_dW: bool = False, logp_ref_given=None, **variant):
    """Forward (+ backward) through the library; returns host tensors."""
    import grpo_loss_gb300 as G
    dev = torch.device("cuda")
    eng = G.GRPOLoss(w.B, w.T, w.d, w.V, w.G, beta=w.beta if beta is None else beta,
                     eps=w.eps, std_unbiased=w.std_unbiased, chunk_rows=chunk_rows,
                     dtype=torch_dtype(w), device=dev, compute_dW=want_dW,
                     ref_logp_given=logp_ref_given is not None, **variant)
    Hp = inp["H_pol"].to(dev)
    Hr = (inp["H_ref"] if H_ref is None else H_ref).to(dev)
    Wd = inp["W"].to(dev)
    idd = (inp["ids"] if ids is None else ids).to(dev)
    md = (inp["mask"] if mask is None else mask).to(dev)
    adv = adv32.to(dev)
    if logp_ref_given is not None:
        loss, klm, lp, lr = eng.forward(Hp, None, Wd, idd, md, adv,
                                        logp_ref=logp_ref_given.to(dev))
    else:
        loss, klm, lp, lr = eng.forward(Hp, Hr, Wd, idd, md, adv)
    out = {}
    if want_bwd:
        dH = eng.backward(Hp, Wd, idd, md, adv, grad)
        out["dH"] = dH.float().cpu()
        if want_dW:
            out["dW"] = eng.dW.cpu()
    torch.cuda.synchronize()
    if check:
        eng.check()
    out.update(loss=float(loss.item()), kl_mean=float(klm.item()), logp_pol=lp.cpu().double(),
               logp_ref=lr.cpu().double(), lse_pol=eng.lse_pol.cpu().double(), engine=eng)
    return out


def rel_err(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b) / np.maximum(np.abs(b), 1e-30))) if a.size else 0.0


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def x_and_kl_close(x_gpu, x_or, what: str = "") -> None:
    """x = p - q and KL = exp(x) - x - 1 at sampled valid rows: each within
    1e-3 relative of the oracle's, with absolute floors of 1e-3 of the
    sample's rms x and of its mean KL. The floors keep rows with x near 0
    (where a tiny KL's relative error means nothing) to the size of the
    term the loss carries, beta * mean KL."""
    from oracle import grpo_oracle as O
    x_gpu = np.asarray(x_gpu, np.float64)
    x_or = np.asarray(x_or, np.float64)
    zero = np.zeros_like(x_or)
    kl_gpu, kl_or = O.kl_estimator(zero, x_gpu), O.kl_estimator(zero, x_or)
    ax = 1e-3 * np.sqrt(np.mean(x_or ** 2))
    ak = 1e-3 * np.mean(kl_or)
    dx = np.abs(x_gpu - x_or)
    dk = np.abs(kl_gpu - kl_or)
    assert np.all(dx <= TOL_REL * np.abs(x_or) + ax), \
        "x %s: max |dx| %.3g, floor %.3g" % (what, dx.max(), ax)
    assert np.all(dk <= TOL_REL * np.abs(kl_or) + ak), \
        "KL %s: max |dKL| %.3g, floor %.3g" % (what, dk.max(), ak)
