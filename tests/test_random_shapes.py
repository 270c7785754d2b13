"""GPU parity on seeded random problem shapes, in bf16 and on e4m3 operands.

Each case draws its sizes from a seeded generator: the hidden size d (a
multiple of 16 up to 2400, ragged against the 64- and 128-element K blocks, on both
sides of the column-split threshold of the forward and dZ epilogues), the
vocab V (ragged against the 256-column tiles, so a vocab slice may hold the
ragged last tile alone), the completion length, the group size, padding down
to empty sequences, and the variant (token level, KL mode, logit transforms,
dW). The input generator draws the tensors; the CUDA path runs through the
engine; the oracle evaluates the same problem (on its own quantization of
the operands for e4m3) and everything is compared element by element."""
import numpy as np
import pytest
import torch

from grpo_loss_gb300 import workloads as WL
from oracle import grpo_oracle as O
from tests.parity_util import TOL_DH_L2, TOL_REL, oracle_adv, rel_err, rel_l2

pytestmark = pytest.mark.gpu

SEEDS = list(range(16))


def _case(seed: int):
    g = np.random.default_rng(20260 + seed)
    G = int(g.choice([1, 2, 4]))
    prompts = int(g.integers(1, 3))
    T = int(g.integers(1, 257))
    d = int(16 * g.integers(1, 151))                # 16 .. 2400
    V = int(g.integers(17, 4001))
    lo = int(g.integers(0, T + 1))
    hi = int(g.integers(lo, T + 1))
    rewards = "adv_normal" if G == 1 else "normal"
    w = WL.Workload("random-%d" % seed, prompts=prompts, G=G, T=T, d=d, V=V,
                    mask="pad_uniform", pad_lo=lo, pad_hi=hi, rewards=rewards,
                    seed=3000 + seed)
    variant = {}
    if g.random() < 0.3:
        variant["token_level"] = True
    if g.random() < 0.3:
        variant["kl_mode"] = int(g.integers(1, 4))
    if g.random() < 0.3:
        variant.update(softcap=float(g.choice([2.0, 30.0])), temperature=0.7)
    want_dW = bool(g.random() < 0.4)
    chunk_rows = int(g.choice([0, 128, 256])) if want_dW else 0
    e4m3 = seed % 2 == 1
    return w, variant, want_dW, chunk_rows, e4m3


@pytest.mark.parametrize("seed", SEEDS)
def test_random_shape_matches_oracle(seed):
    import grpo_loss_gb300 as G
    w, variant, want_dW, chunk_rows, e4m3 = _case(seed)
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    dev = torch.device("cuda")
    eng = G.GRPOLoss(w.B, w.T, w.d, w.V, w.G, beta=w.beta, eps=w.eps,
                     std_unbiased=w.std_unbiased, chunk_rows=chunk_rows,
                     dtype=torch.float8_e4m3fn if e4m3 else torch.bfloat16, device=dev,
                     compute_dW=want_dW, **variant)
    Hp, Wd = inp["H_pol"].to(dev), inp["W"].to(dev)
    ids, mask, adv = inp["ids"].to(dev), inp["mask"].to(dev), adv32.to(dev)
    loss, klm, lp, lr = eng.forward(Hp, inp["H_ref"].to(dev), Wd, ids, mask, adv)
    dH = eng.backward(Hp, Wd, ids, mask, adv, 1.0)
    torch.cuda.synchronize()
    eng.check()

    if e4m3:
        ops = {k: O.dequantize_rows(*O.quantize_e4m3_rows(inp[k])) for k in ("H_pol", "H_ref", "W")}
    else:
        ops = {k: inp[k] for k in ("H_pol", "H_ref", "W")}
    xf = None
    if "softcap" in variant:
        xf = {"softcap": variant["softcap"], "temperature": variant["temperature"]}
    kw = dict(token_level=variant.get("token_level", False), xform=xf,
              kl_mode=variant.get("kl_mode", 0))
    f = O.forward(ops["H_pol"], ops["H_ref"], ops["W"], inp["ids"], inp["mask"], adv32.double(),
                  w.B, w.T, w.beta, **kw)
    gr = O.backward(ops["H_pol"], ops["H_ref"], ops["W"], inp["ids"], inp["mask"],
                    adv32.double(), w.B, w.T, w.beta, want_dW=want_dW, **kw)
    m = inp["mask"].numpy() > 0
    desc = (w.B, w.T, w.d, w.V, w.G, variant, want_dW, chunk_rows, e4m3)
    assert rel_err(lp.cpu().double().numpy()[m], f["logp_pol"][m]) < TOL_REL, desc
    assert rel_err(lr.cpu().double().numpy()[m], f["logp_ref"][m]) < TOL_REL, desc
    assert rel_err(eng.lse_pol.cpu().double().numpy()[m], f["lse_pol"][m]) < TOL_REL, desc
    assert abs(loss.item() - f["loss"]) <= TOL_REL * abs(f["loss"]) + 1e-9, (desc, loss.item(), f["loss"])
    assert abs(klm.item() - f["kl_mean"]) <= TOL_REL * abs(f["kl_mean"]) + 1e-9, desc
    d = dH.float().cpu().numpy()
    assert np.all(d[~m] == 0), desc
    if m.any():
        assert rel_l2(d, gr["dH"]) < TOL_DH_L2, (desc, rel_l2(d, gr["dH"]))
    if want_dW and m.any():
        assert rel_l2(eng.dW.cpu().numpy(), gr["dW"]) < TOL_DH_L2, desc
