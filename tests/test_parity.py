"""GPU parity of the CUDA path against the float64 oracle on the same seeded
inputs, through the C ABI: oracle-sized workloads (every element compared)
and edge cases. The oracle is given the exact input values; advantages fed
to the loss are the oracle's, rounded to float32, on both sides."""
import numpy as np
import pytest
import torch

from grpo_loss_gb300 import workloads as WL
from oracle import grpo_oracle as O
from tests.parity_util import TOL_DH_L2, TOL_REL, gpu_run, oracle_adv, rel_err, rel_l2

pytestmark = pytest.mark.gpu

CASES = [WL.TINY] + list(WL.SMALL.values())


def _oracle(w, inp, adv32, beta=None, grad=1.0, H_ref=None, ids=None, mask=None):
    b = w.beta if beta is None else beta
    Hr = inp["H_ref"] if H_ref is None else H_ref
    ids = inp["ids"] if ids is None else ids
    mask = inp["mask"] if mask is None else mask
    f = O.forward(inp["H_pol"], Hr, inp["W"], ids, mask, adv32.double(), w.B, w.T, b)
    g = O.backward(inp["H_pol"], Hr, inp["W"], ids, mask, adv32.double(), w.B, w.T, b,
                   grad_loss=grad)
    return f, g


def _compare(w, res, f, g, mask):
    m = mask.numpy() > 0
    assert rel_err(res["logp_pol"].numpy()[m], f["logp_pol"][m]) < TOL_REL
    assert rel_err(res["logp_ref"].numpy()[m], f["logp_ref"][m]) < TOL_REL
    assert rel_err(res["lse_pol"].numpy()[m], f["lse_pol"][m]) < TOL_REL
    assert np.all(res["logp_pol"].numpy()[~m] == 0) and np.all(res["logp_ref"].numpy()[~m] == 0)
    assert abs(res["loss"] - f["loss"]) <= TOL_REL * abs(f["loss"]), (res["loss"], f["loss"])
    assert abs(res["kl_mean"] - f["kl_mean"]) <= TOL_REL * abs(f["kl_mean"]) + 1e-12
    dH = res["dH"].numpy()
    assert rel_l2(dH, g["dH"]) < TOL_DH_L2, rel_l2(dH, g["dH"])
    assert np.all(dH[~m] == 0)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_advantages_match_oracle(w):
    import grpo_loss_gb300 as G
    if w.supplied_adv:
        pytest.skip("advantages supplied directly")
    inp = WL.make_inputs(w)
    r = inp["rewards"].cuda()
    adv = torch.empty_like(r)
    G.advantages(r, w.G, w.eps, w.std_unbiased, adv)
    ref = O.advantages(inp["rewards"], w.G, w.eps, w.std_unbiased)
    got = adv.cpu().double().numpy()
    assert np.all(np.abs(got - ref) <= TOL_REL * np.abs(ref) + 1e-6)
    assert np.all(np.abs(got.reshape(-1, w.G).sum(1)) < 1e-5)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_forward_backward_match_oracle(w):
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    res = gpu_run(w, inp, adv32)
    f, g = _oracle(w, inp, adv32)
    _compare(w, res, f, g, inp["mask"])


@pytest.mark.parametrize("w,chunk_rows", [(WL.TINY, 0), (WL.SMALL["qwen2.5-small"], 256),
                                          (WL.SMALL["gpt-oss-small"], 0),
                                          (WL.SMALL["qwen3-small"], 128)],
                         ids=["tiny", "qwen2.5-small-chunk256", "gpt-oss-small",
                              "qwen3-small-chunk128"])
def test_dW_matches_oracle(w, chunk_rows):
    """dW = sum over chunks of dZ^T H_pol, with several chunks accumulating."""
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    res = gpu_run(w, inp, adv32, chunk_rows=chunk_rows, want_dW=True)
    g = O.backward(inp["H_pol"], inp["H_ref"], inp["W"], inp["ids"], inp["mask"],
                   adv32.double(), w.B, w.T, w.beta, want_dW=True)
    assert rel_l2(res["dW"].numpy(), g["dW"]) < TOL_DH_L2, rel_l2(res["dW"].numpy(), g["dW"])
    assert rel_l2(res["dH"].numpy(), g["dH"]) < TOL_DH_L2


def test_dW_ragged_and_rejected_without_flag():
    import grpo_loss_gb300 as G
    w = WL.Workload("ragged-dw", prompts=1, G=3, T=50, d=200, V=1001, mask="pad_uniform",
                    pad_lo=25, pad_hi=50, rewards="normal", seed=78)
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    res = gpu_run(w, inp, adv32, chunk_rows=128, want_dW=True)
    g = O.backward(inp["H_pol"], inp["H_ref"], inp["W"], inp["ids"], inp["mask"],
                   adv32.double(), w.B, w.T, w.beta, want_dW=True)
    assert rel_l2(res["dW"].numpy(), g["dW"]) < TOL_DH_L2
    # dW pointer without compute_dW (and the reverse) is an argument error
    eng = res["engine"]
    with pytest.raises(G.GrpoError) as e:
        G.loss_bwd(eng.problem, inp["H_pol"].cuda(), inp["W"].cuda(), inp["ids"].cuda(),
                   inp["mask"].cuda(), adv32.cuda(), eng.logp_pol, eng.logp_ref, eng.lse_pol,
                   1.0, torch.empty(w.N, w.d, dtype=torch.bfloat16, device="cuda"), eng.ws_bwd,
                   dW=None)
    assert e.value.status == 1


def test_small_chunks_give_identical_gradients_and_runs_are_deterministic():
    w = WL.SMALL["qwen2.5-small"]
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    a = gpu_run(w, inp, adv32, chunk_rows=128)
    b = gpu_run(w, inp, adv32, chunk_rows=384)
    c = gpu_run(w, inp, adv32)
    assert torch.equal(a["dH"], b["dH"]) and torch.equal(a["dH"], c["dH"])
    assert a["loss"] == c["loss"] and torch.equal(a["logp_pol"], c["logp_pol"])


def test_reference_equal_policy():
    """KL vanishes and the loss is -mean(A) (pages: exp(q - q.detach()) is 1)."""
    w = WL.SMALL["gpt-oss-small"]
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    res = gpu_run(w, inp, adv32, H_ref=inp["H_pol"])
    m = inp["mask"].reshape(w.B, w.T).sum(1) > 0
    expect = -adv32.double()[m].sum().item() / w.B
    assert res["kl_mean"] == 0.0
    assert abs(res["loss"] - expect) <= 1e-6 * max(1.0, abs(expect))
    assert torch.equal(res["logp_pol"], res["logp_ref"])


def test_beta_zero_and_negative_grad_scale():
    w = WL.SMALL["llama3.1-small"]
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    res = gpu_run(w, inp, adv32, beta=0.0, grad=-2.5)
    f, g = _oracle(w, inp, adv32, beta=0.0, grad=-2.5)
    assert abs(res["loss"] - f["loss"]) <= 1e-6
    assert rel_l2(res["dH"].numpy(), g["dH"]) < TOL_DH_L2


@pytest.mark.parametrize("shape", [(3, 50, 200, 1001, 3), (2, 130, 64, 300, 2), (1, 129, 8, 17, 1)],
                         ids=["d200-V1001", "N260-V300", "d8-V17"])
def test_ragged_sizes(shape):
    """K tail (d not a multiple of 64), vocab not a multiple of 8 or 256, N not
    a multiple of 128, tiny d and V."""
    B, T, d, V, G = shape
    w = WL.Workload("ragged", prompts=B // G, G=G, T=T, d=d, V=V, mask="pad_uniform",
                    pad_lo=T // 2, pad_hi=T, rewards="normal", std_unbiased=1 if G > 1 else 0,
                    seed=77)
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    res = gpu_run(w, inp, adv32, chunk_rows=128)
    f, g = _oracle(w, inp, adv32)
    _compare(w, res, f, g, inp["mask"])


def test_masked_rows_and_empty_sequences():
    w = WL.SMALL["qwen3-small"].scaled("qwen3-masked", prompts=4, G=2, T=300)
    inp = WL.make_inputs(w)
    mask = inp["mask"].clone().reshape(w.B, w.T)
    mask[1] = 0                        # a sequence with no valid token
    mask[2, 100:260] = 0               # a hole spanning a whole 128-row block
    mask = mask.reshape(-1)
    ids = inp["ids"].clone()
    ids[mask == 0] = -100              # ignore labels at masked rows are accepted
    adv32 = torch.from_numpy(np.random.default_rng(3).standard_normal(w.B)).float()
    res = gpu_run(w, inp, adv32, ids=ids, mask=mask, chunk_rows=256)
    inp2 = dict(inp, ids=ids, mask=mask)
    f, g = _oracle(w, inp2, adv32)
    _compare(w, res, f, g, mask)


def test_all_masked_problem():
    w = WL.SMALL["llama3.1-small"]
    inp = WL.make_inputs(w)
    mask = torch.zeros_like(inp["mask"])
    adv32 = torch.ones(w.B)
    res = gpu_run(w, inp, adv32, mask=mask)
    assert res["loss"] == 0.0 and res["kl_mean"] == 0.0
    assert torch.all(res["dH"] == 0) and torch.all(res["logp_pol"] == 0)


def test_bad_token_is_reported_on_device():
    import grpo_loss_gb300 as G
    w = WL.TINY
    inp = WL.make_inputs(w)
    ids = inp["ids"].clone()
    ids[5] = w.V                       # a valid row (mask 1) with id == V
    adv32 = torch.zeros(w.B)
    res = gpu_run(w, inp, adv32, ids=ids, want_bwd=False, check=False)
    assert G.device_status(res["engine"].ws_fwd) == 6
    assert G.device_status(res["engine"].ws_fwd) == 0      # read clears it


def test_short_workspace_and_bad_problem_rejected():
    import ctypes
    import grpo_loss_gb300 as G
    from grpo_loss_gb300 import _lib as L
    w = WL.TINY
    p = G.make_problem(w.B, w.T, w.d, w.V, w.G, dtype=torch.float32)
    fb, bb = G.workspace_size(p)
    assert fb > 0 and bb > 0
    x = torch.zeros(w.N * w.d, device="cuda")
    small = torch.empty(fb - 256, dtype=torch.uint8, device="cuda")
    f32 = torch.zeros(w.N, device="cuda")
    with pytest.raises(G.GrpoError) as e:
        G.loss_fwd(p, x, x, torch.zeros(w.V * w.d, device="cuda"),
                   torch.zeros(w.N, dtype=torch.int32, device="cuda"),
                   torch.ones(w.N, dtype=torch.uint8, device="cuda"),
                   torch.zeros(w.B, device="cuda"), f32, f32.clone(), f32.clone(),
                   torch.zeros(1, device="cuda"), None, small)
    assert e.value.status == 3
