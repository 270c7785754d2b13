"""GPU parity of the optional variants against the float64 oracle: logit
transforms (scale, softcap, temperature), token-level aggregation and
reference log-probs supplied by the caller, alone and together, for the
forward, dH and dW."""
import numpy as np
import pytest
import torch

from grpo_loss_gb300 import workloads as WL
from oracle import grpo_oracle as O
from tests.parity_util import TOL_DH_L2, TOL_REL, gpu_run, oracle_adv, rel_err, rel_l2

pytestmark = pytest.mark.gpu

XF = {"logit_multiply": 1.5, "logit_divide": 1.2, "softcap": 2.0, "temperature": 0.7}


def _oxf(variant):
    if not any(k in variant for k in XF):
        return None
    return {"multiply": variant.get("logit_multiply", 0.0), "divide": variant.get("logit_divide", 0.0),
            "softcap": variant.get("softcap", 0.0), "temperature": variant.get("temperature", 0.0)}


def _check(w, inp, adv32, res, token_level, xf, given=None, dW=False, kl_mode=0):
    f = O.forward(inp["H_pol"], inp["H_ref"], inp["W"], inp["ids"], inp["mask"], adv32.double(),
                  w.B, w.T, w.beta, token_level=token_level, xform=xf, logp_ref_given=given,
                  kl_mode=kl_mode)
    g = O.backward(inp["H_pol"], inp["H_ref"], inp["W"], inp["ids"], inp["mask"], adv32.double(),
                   w.B, w.T, w.beta, token_level=token_level, xform=xf, logp_ref_given=given,
                   want_dW=dW, kl_mode=kl_mode)
    m = inp["mask"].numpy() > 0
    assert rel_err(res["logp_pol"].numpy()[m], f["logp_pol"][m]) < TOL_REL
    assert rel_err(res["logp_ref"].numpy()[m], f["logp_ref"][m]) < TOL_REL
    assert rel_err(res["lse_pol"].numpy()[m], f["lse_pol"][m]) < TOL_REL
    assert abs(res["loss"] - f["loss"]) <= TOL_REL * abs(f["loss"]), (res["loss"], f["loss"])
    assert abs(res["kl_mean"] - f["kl_mean"]) <= TOL_REL * abs(f["kl_mean"]) + 1e-12
    assert rel_l2(res["dH"].numpy(), g["dH"]) < TOL_DH_L2, rel_l2(res["dH"].numpy(), g["dH"])
    assert np.all(res["dH"].numpy()[~m] == 0)
    if dW:
        assert rel_l2(res["dW"].numpy(), g["dW"]) < TOL_DH_L2


CASES = [
    ("token-level", WL.SMALL["qwen2.5-small"], {"token_level": True}),
    ("token-level-gptoss", WL.SMALL["gpt-oss-small"], {"token_level": True}),
    ("transforms", WL.SMALL["llama3.1-small"], dict(XF)),
    ("softcap-only-tiny", WL.TINY, {"softcap": 1.0}),
    ("temperature-only", WL.SMALL["qwen3-small"], {"temperature": 0.6}),
    ("all", WL.SMALL["gpt-oss-small"], dict(XF, token_level=True)),
    ("kl-no-detach", WL.SMALL["qwen2.5-small"], {"kl_mode": 1}),
    ("kl-times-q", WL.SMALL["qwen2.5-small"], {"kl_mode": 2}),
    ("kl-forward", WL.SMALL["llama3.1-small"], {"kl_mode": 3}),
    ("kl-forward-token-softcap", WL.TINY, {"kl_mode": 3, "token_level": True, "softcap": 1.0}),
    # CTA-pair (cta_group::2) kernels: odd block counts leave a pair partner
    # without a block; d = 2880 pairs 96-row halves of 192-wide column tiles
    ("pairs-llama", WL.SMALL["llama3.1-small"], {"cluster_mode": 1}),
    ("pairs-qwen3-odd-blocks", WL.SMALL["qwen3-small"], {"cluster_mode": 1}),
    ("pairs-tiny-all", WL.TINY, dict(XF, token_level=True, kl_mode=2, cluster_mode=1)),
    ("pairs-d2880", WL.GPTOSS_20B.scaled("gpt-oss-d2880", prompts=1, G=4, T=160, d=2880, V=2056,
                                         pad_lo=80, pad_hi=160), {"cluster_mode": 1}),
]


@pytest.mark.parametrize("name,w,variant", CASES, ids=[c[0] for c in CASES])
def test_variant_matches_oracle(name, w, variant):
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    res = gpu_run(w, inp, adv32, chunk_rows=256, want_dW=True, **variant)
    _check(w, inp, adv32, res, variant.get("token_level", False), _oxf(variant), dW=True,
           kl_mode=variant.get("kl_mode", 0))


@pytest.mark.parametrize("variant", [{}, dict(XF, token_level=True)], ids=["plain", "all"])
def test_given_reference_logprobs(variant):
    """The reference half of the forward is skipped; H_ref is not passed."""
    w = WL.SMALL["qwen2.5-small"]
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    xf = _oxf(variant)
    ids_safe = np.where(inp["mask"].numpy() > 0, inp["ids"].numpy(), 0)
    p, _ = O.token_logprobs(inp["H_ref"], inp["W"], ids_safe, xform=xf)
    given = torch.from_numpy(p).float()          # what a caller would hold: float32
    res = gpu_run(w, inp, adv32, logp_ref_given=given, **variant)
    _check(w, inp, adv32, res, variant.get("token_level", False), xf, given=given.double())
    # the supplied buffer is only read: unchanged, masked rows included
    assert torch.equal(res["logp_ref"].float(), given)
