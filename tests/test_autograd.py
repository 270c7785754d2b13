"""The autograd entry `grpo_loss`: loss.backward() through the library's
kernels gives the oracle's gradients with respect to H_pol and, with an
engine built with compute_dW, W; the upstream gradient scales them; kl_mean
carries no gradient; an e4m3 engine returns gradients in the inputs' dtype."""
import numpy as np
import pytest
import torch

from grpo_loss_gb300 import workloads as WL
from oracle import grpo_oracle as O
from tests.parity_util import TOL_DH_L2, TOL_REL, oracle_adv, rel_l2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("engine_dtype,input_dtype", [
    (torch.bfloat16, torch.bfloat16),
    (torch.float8_e4m3fn, torch.bfloat16),
    (torch.float8_e4m3fn, torch.float32),
], ids=["bf16", "e4m3-from-bf16", "e4m3-from-f32"])
def test_loss_backward_gives_oracle_gradients(engine_dtype, input_dtype):
    import grpo_loss_gb300 as G
    w = WL.SMALL["llama3.1-small"]
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    dev = torch.device("cuda")
    eng = G.GRPOLoss(w.B, w.T, w.d, w.V, w.G, beta=w.beta, eps=w.eps,
                     std_unbiased=w.std_unbiased, dtype=engine_dtype, device=dev,
                     compute_dW=True)
    Hp = inp["H_pol"].to(input_dtype).to(dev).requires_grad_(True)
    Wd = inp["W"].to(input_dtype).to(dev).requires_grad_(True)
    Hr = inp["H_ref"].to(input_dtype).to(dev)
    ids, mask, adv = inp["ids"].to(dev), inp["mask"].to(dev), adv32.to(dev)
    loss, kl = G.grpo_loss(Hp, Hr, Wd, ids, mask, adv, eng)
    assert loss.dim() == 0 and kl.dim() == 0
    (2.5 * loss + 0.0 * kl).backward()
    torch.cuda.synchronize()
    eng.check()
    assert Hp.grad.dtype == input_dtype and Wd.grad.dtype == input_dtype

    src = {k: inp[k].to(input_dtype) for k in ("H_pol", "H_ref", "W")}
    if engine_dtype == torch.float8_e4m3fn:
        ops = {k: O.dequantize_rows(*O.quantize_e4m3_rows(v)) for k, v in src.items()}
    else:
        ops = src
    f = O.forward(ops["H_pol"], ops["H_ref"], ops["W"], inp["ids"], inp["mask"], adv32.double(),
                  w.B, w.T, w.beta)
    g = O.backward(ops["H_pol"], ops["H_ref"], ops["W"], inp["ids"], inp["mask"],
                   adv32.double(), w.B, w.T, w.beta, grad_loss=2.5, want_dW=True)
    assert abs(loss.item() - f["loss"]) <= TOL_REL * abs(f["loss"])
    assert rel_l2(Hp.grad.float().cpu().numpy(), g["dH"]) < TOL_DH_L2
    assert rel_l2(Wd.grad.float().cpu().numpy(), g["dW"]) < TOL_DH_L2
    m = inp["mask"].numpy() > 0
    assert np.all(Hp.grad.float().cpu().numpy()[~m] == 0)


def test_kl_mean_alone_has_no_gradient_path():
    """kl_mean is a metric: a backward from it alone gives zero gradients."""
    import grpo_loss_gb300 as G
    w = WL.TINY
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    dev = torch.device("cuda")
    eng = G.GRPOLoss(w.B, w.T, w.d, w.V, w.G, beta=w.beta, eps=w.eps,
                     std_unbiased=w.std_unbiased, dtype=torch.float32, device=dev)
    Hp = inp["H_pol"].to(dev).requires_grad_(True)
    loss, kl = G.grpo_loss(Hp, inp["H_ref"].to(dev), inp["W"].to(dev), inp["ids"].to(dev),
                           inp["mask"].to(dev), adv32.to(dev), eng)
    kl.backward()
    torch.cuda.synchronize()
    assert Hp.grad is not None and float(Hp.grad.abs().max()) == 0.0
