"""Parity at the full sizes of the five workloads, in the launch
configuration the benchmark times (default chunk plan).

The loss and the KL mean are compared with the float64 oracle's full
forward pass over every token, computed once on the host and stored under
tests/golden/ with a digest of the inputs it used. Per-token quantities are
checked on a seeded, stratified sample of rows one by one (log-probs,
logsumexp, x = p - q, the KL term and the dH row, which depends on that row
alone), and the rest through properties that hold at any size: masked rows
are exactly zero, the loss equals its definition evaluated in float64 from
the per-token outputs, and with the reference equal to the policy the KL is
exactly zero and the loss is -mean(A)."""
import json
import os

import numpy as np
import pytest
import torch

from grpo_loss_gb300 import workloads as WL
from oracle import grpo_oracle as O
from tests.parity_util import (TOL_DH_L2, TOL_REL, gpu_run, oracle_adv, rel_err, rel_l2,
                               x_and_kl_close)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

BIG = [WL.QWEN25_1P5B, WL.LLAMA31_8B_20K, WL.QWEN3_8B_110K, WL.GPTOSS_20B]
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", params=BIG, ids=lambda w: w.name)
def case(request):
    w = request.param
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    res = gpu_run(w, inp, adv32)
    yield w, inp, adv32, res
    del res
    torch.cuda.empty_cache()


def test_sampled_rows_match_oracle(case):
    w, inp, adv32, res = case
    rows = WL.sample_rows(w, inp["mask"], count=2048)
    m = inp["mask"].numpy()[rows] > 0
    vrows = rows[m]
    Wf = O.to_f64(inp["W"])
    q, lse = O.token_logprobs(inp["H_pol"], Wf, inp["ids"], rows=vrows)
    p, _ = O.token_logprobs(inp["H_ref"], Wf, inp["ids"], rows=vrows)
    assert rel_err(res["logp_pol"].numpy()[vrows], q) < TOL_REL
    assert rel_err(res["logp_ref"].numpy()[vrows], p) < TOL_REL
    assert rel_err(res["lse_pol"].numpy()[vrows], lse) < TOL_REL
    x_gpu = res["logp_ref"].numpy()[vrows] - res["logp_pol"].numpy()[vrows]
    x_and_kl_close(x_gpu, p - q, w.name)
    g = O.backward(inp["H_pol"], inp["H_ref"], Wf, inp["ids"], inp["mask"], adv32.double(),
                   w.B, w.T, w.beta, rows=rows)
    dH = res["dH"].numpy()[rows]
    assert rel_l2(dH[m], g["dH"][m]) < TOL_DH_L2
    # each sampled valid row on its own, with room for bf16 rounding of dZ
    for i in np.nonzero(m)[0]:
        assert rel_l2(dH[i], g["dH"][i]) < 3 * TOL_DH_L2, int(rows[i])
    assert np.all(dH[~m] == 0)


def test_loss_and_kl_match_the_full_oracle_forward(case):
    """loss and kl_mean within 1e-3 relative of the oracle's full float64
    forward over every token (tests/golden/make_fullsize_golden.py), on the
    same inputs: the stored digest must equal this run's."""
    w, inp, adv32, res = case
    with open(os.path.join(GOLDEN, "fullsize_%s.json" % w.name)) as fh:
        rec = json.load(fh)
    assert WL.input_digest(inp) == rec["input_digest"], \
        "inputs differ from the ones the stored oracle values were computed on"
    assert adv32.tolist() == rec["adv_float32"]
    m = inp["mask"].numpy() > 0
    assert int(m.sum()) == rec["n_valid"]
    assert abs(res["loss"] - rec["loss"]) <= TOL_REL * abs(rec["loss"]), (res["loss"], rec["loss"])
    assert abs(res["kl_mean"] - rec["kl_mean"]) <= TOL_REL * abs(rec["kl_mean"]), \
        (res["kl_mean"], rec["kl_mean"])
    # sums over every valid token: a per-token bias would show here
    q = res["logp_pol"].numpy()[m].astype(np.float64)
    p = res["logp_ref"].numpy()[m].astype(np.float64)
    assert abs(q.sum() - rec["sum_logp_pol"]) <= 1e-5 * abs(rec["sum_logp_pol"])
    assert abs(p.sum() - rec["sum_logp_ref"]) <= 1e-5 * abs(rec["sum_logp_ref"])
    assert abs(np.sum((p - q) ** 2) - rec["sum_x_sq"]) <= TOL_REL * rec["sum_x_sq"]


def test_masked_rows_are_zero_everywhere(case):
    w, inp, adv32, res = case
    masked = inp["mask"].numpy() == 0
    assert np.all(res["logp_pol"].numpy()[masked] == 0)
    assert np.all(res["logp_ref"].numpy()[masked] == 0)
    assert bool(torch.all(res["dH"][torch.from_numpy(masked)] == 0))
    assert np.all(np.isfinite(res["logp_pol"].numpy())) and bool(torch.isfinite(res["dH"]).all())


def test_loss_is_its_definition_over_the_outputs(case):
    """loss = sum_n w_n (-A_b + beta (exp(x) - x - 1)) and kl_mean = masked
    mean of KL, evaluated in float64 on the host from the per-token outputs."""
    w, inp, adv32, res = case
    wts, cnt = O.sequence_weights(inp["mask"], w.B, w.T)
    kl = O.kl_estimator(res["logp_pol"].numpy(), res["logp_ref"].numpy())
    A = np.repeat(adv32.double().numpy(), w.T)
    m = inp["mask"].numpy() > 0
    loss = float(np.sum(np.where(m, wts * (-A + w.beta * kl), 0.0)))
    assert abs(res["loss"] - loss) <= 1e-5 * abs(loss) + 1e-9
    assert abs(res["kl_mean"] - kl[m].mean()) <= 1e-5 * abs(kl[m].mean())
    assert res["kl_mean"] > 0


def test_reference_equal_policy_full_size(case):
    w, inp, adv32, _ = case
    res = gpu_run(w, inp, adv32, H_ref=inp["H_pol"], want_bwd=False)
    cnt = inp["mask"].reshape(w.B, w.T).sum(1) > 0
    expect = -adv32.double()[cnt].sum().item() / w.B
    assert res["kl_mean"] == 0.0
    assert abs(res["loss"] - expect) <= 1e-6 * max(1.0, abs(expect))


@pytest.mark.parametrize("variant", [{"softcap": 30.0, "temperature": 0.7, "token_level": True},
                                     {"kl_mode": 3}, {"cluster_mode": 1}],
                         ids=["softcap-temp-token", "forward-kl", "cta-pairs"])
def test_variant_sampled_rows_full_size(variant):
    """A variant at the full Llama-shaped size: sampled rows against the oracle."""
    w = WL.LLAMA31_8B_20K
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    res = gpu_run(w, inp, adv32, **variant)
    xf = None
    if "softcap" in variant:
        xf = {"softcap": variant["softcap"], "temperature": variant["temperature"]}
    rows = WL.sample_rows(w, inp["mask"], count=48)
    Wf = O.to_f64(inp["W"])
    q, lse = O.token_logprobs(inp["H_pol"], Wf, inp["ids"], rows=rows, xform=xf)
    p, _ = O.token_logprobs(inp["H_ref"], Wf, inp["ids"], rows=rows, xform=xf)
    assert rel_err(res["logp_pol"].numpy()[rows], q) < TOL_REL
    assert rel_err(res["logp_ref"].numpy()[rows], p) < TOL_REL
    x_and_kl_close(res["logp_ref"].numpy()[rows] - res["logp_pol"].numpy()[rows], p - q,
                   str(variant))
    g = O.backward(inp["H_pol"], inp["H_ref"], Wf, inp["ids"], inp["mask"], adv32.double(),
                   w.B, w.T, w.beta, rows=rows, token_level=variant.get("token_level", False),
                   xform=xf, kl_mode=variant.get("kl_mode", 0))
    assert rel_l2(res["dH"].numpy()[rows], g["dH"]) < TOL_DH_L2
    del res
    torch.cuda.empty_cache()


def test_wide_vocab_softcap_head():
    """A Gemma-3-shaped head (the pages list Gemma among the supported models,
    and Gemma applies logit softcapping): V = 262144, d = 5376, softcap 30,
    sampled rows against the oracle."""
    w = WL.Workload("gemma3-shaped-head", prompts=1, G=4, T=512, d=5376, V=262144,
                    mask="pad_uniform", pad_lo=384, pad_hi=512, rewards="normal", seed=1010)
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    res = gpu_run(w, inp, adv32, softcap=30.0)
    xf = {"softcap": 30.0}
    rows = WL.sample_rows(w, inp["mask"], count=40)
    m = inp["mask"].numpy()[rows] > 0
    vrows = rows[m]
    Wf = O.to_f64(inp["W"])
    q, lse = O.token_logprobs(inp["H_pol"], Wf, inp["ids"], rows=vrows, xform=xf)
    p, _ = O.token_logprobs(inp["H_ref"], Wf, inp["ids"], rows=vrows, xform=xf)
    assert rel_err(res["logp_pol"].numpy()[vrows], q) < TOL_REL
    assert rel_err(res["logp_ref"].numpy()[vrows], p) < TOL_REL
    assert rel_err(res["lse_pol"].numpy()[vrows], lse) < TOL_REL
    g = O.backward(inp["H_pol"], inp["H_ref"], Wf, inp["ids"], inp["mask"], adv32.double(),
                   w.B, w.T, w.beta, rows=rows, xform=xf)
    assert rel_l2(res["dH"].numpy()[rows][m], g["dH"][m]) < TOL_DH_L2
    assert np.all(res["dH"].numpy()[rows][~m] == 0)
    del res
    torch.cuda.empty_cache()


def _mem_available_gb() -> float:
    try:
        with open("/proc/meminfo") as fh:
            for line in fh:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) / 1e6
    except OSError:
        pass
    return 0.0


def test_operands_past_2_31_elements_sampled_rows():
    """524288 tokens on the Llama-8B head: H holds 2^31 elements (8.6 GB of
    bf16 bytes), so any 32-bit element or byte offset would wrap. Sampled
    rows, including the last valid row of the last sequence, against the
    oracle; the loss against its definition over the per-token outputs."""
    if _mem_available_gb() < 96:
        pytest.skip("needs about 30 GB of host memory for the inputs")
    w = WL.LLAMA31_8B_20K.scaled("llama3.1-head-512k", prompts=8, G=8, T=8192,
                                 mask="pad_uniform", pad_lo=6144, pad_hi=8192, seed=1020)
    assert w.N * w.d == 1 << 31
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    res = gpu_run(w, inp, adv32)
    rows = WL.sample_rows(w, inp["mask"], count=48)
    m = inp["mask"].numpy()
    last_valid = int(np.nonzero(m)[0][-1])
    rows = np.unique(np.concatenate([rows, [last_valid]]))
    valid = m[rows] > 0
    Wf = O.to_f64(inp["W"])
    q, lse = O.token_logprobs(inp["H_pol"], Wf, inp["ids"], rows=rows[valid])
    p, _ = O.token_logprobs(inp["H_ref"], Wf, inp["ids"], rows=rows[valid])
    assert rel_err(res["logp_pol"].numpy()[rows[valid]], q) < TOL_REL
    assert rel_err(res["logp_ref"].numpy()[rows[valid]], p) < TOL_REL
    assert rel_err(res["lse_pol"].numpy()[rows[valid]], lse) < TOL_REL
    g = O.backward(inp["H_pol"], inp["H_ref"], Wf, inp["ids"], inp["mask"], adv32.double(),
                   w.B, w.T, w.beta, rows=rows)
    dH = res["dH"].numpy()[rows]
    assert rel_l2(dH[valid], g["dH"][valid]) < TOL_DH_L2
    assert np.all(dH[~valid] == 0)
    wts, _ = O.sequence_weights(inp["mask"], w.B, w.T)
    kl = O.kl_estimator(res["logp_pol"].numpy(), res["logp_ref"].numpy())
    A = np.repeat(adv32.double().numpy(), w.T)
    mm = m > 0
    loss = float(np.sum(np.where(mm, wts * (-A + w.beta * kl), 0.0)))
    assert abs(res["loss"] - loss) <= 1e-5 * abs(loss) + 1e-9
    del res
    torch.cuda.empty_cache()


def test_dW_full_size_qwen_head():
    """dW (the lm_head gradient) at the full Qwen2.5-1.5B-shaped head
    (16384 tokens, 11998 valid; d = 1536, V = 151936), in the benchmark's
    default chunk plan, against the oracle's full float64 dW; dH on every row."""
    w = WL.QWEN25_1P5B
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    res = gpu_run(w, inp, adv32, want_dW=True)
    g = O.backward(inp["H_pol"], inp["H_ref"], inp["W"], inp["ids"], inp["mask"], adv32.double(),
                   w.B, w.T, w.beta, want_dW=True)
    assert rel_l2(res["dW"].numpy(), g["dW"]) < TOL_DH_L2
    assert rel_l2(res["dH"].numpy(), g["dH"]) < TOL_DH_L2
    m = inp["mask"].numpy() > 0
    assert np.all(res["dH"].numpy()[~m] == 0)
    del res
    torch.cuda.empty_cache()
