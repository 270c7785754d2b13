"""Pins of the float64 oracle against facts fixed outside the oracle itself:
hand-worked closed forms, library routines on special cases, invariants the
pages state, a literal autograd of the objective, finite differences, and
the pages' printed memory figures. CPU only."""
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import grpo_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- advantages

def test_advantages_hand_worked_group():
    # rewards 0,1,2,3: mean 1.5; squared deviations 2.25+0.25+0.25+2.25 = 5
    A = O.advantages([0.0, 1.0, 2.0, 3.0], 4, eps=1e-4, std_unbiased=1)
    std = np.sqrt(5.0 / 3.0)            # ddof 1: 5 / 3
    assert np.allclose(A, np.array([-1.5, -0.5, 0.5, 1.5]) / (std + 1e-4), rtol=1e-15)
    A0 = O.advantages([0.0, 1.0, 2.0, 3.0], 4, eps=1e-4, std_unbiased=0)
    assert np.allclose(A0, np.array([-1.5, -0.5, 0.5, 1.5]) / (np.sqrt(1.25) + 1e-4), rtol=1e-15)


def test_advantages_pair_and_constant_groups():
    # group {0, 2}: mean 1, ddof-1 std sqrt(2); group {5, 5}: all equal -> 0
    A = O.advantages([0.0, 2.0], 2, eps=0.0, std_unbiased=1)
    s = 1.0 / np.sqrt(2.0)
    assert np.allclose(A, [-s, s], rtol=1e-15, atol=0)
    assert np.all(O.advantages([5.0, 5.0, 0.0, 2.0], 2, eps=1e-4, std_unbiased=1)[:2] == 0.0)


def test_advantages_match_torch_std_and_sum_to_zero():
    g = torch.Generator().manual_seed(3)
    r = torch.randn(12, 8, generator=g, dtype=torch.float64)
    for unbiased in (True, False):
        ref = (r - r.mean(1, keepdim=True)) / (r.std(1, keepdim=True, unbiased=unbiased) + 1e-4)
        A = O.advantages(r.reshape(-1), 8, eps=1e-4, std_unbiased=int(unbiased))
        assert np.allclose(A, ref.reshape(-1).numpy(), rtol=1e-13, atol=1e-14)
        assert np.all(np.abs(A.reshape(12, 8).sum(1)) < 1e-12)


def test_advantages_reject_bad_groups():
    with pytest.raises(ValueError):
        O.advantages([1.0, 2.0, 3.0], 2, 1e-4, 1)
    with pytest.raises(ValueError):
        O.advantages([1.0, 2.0], 1, 1e-4, 1)
    assert np.all(O.advantages([1.0, 2.0], 1, 1e-4, 0) == 0.0)


# ------------------------------------------------------------------ log-probs

def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return scale * torch.randn(*shape, generator=g, dtype=torch.float64)


def test_logprobs_match_torch_log_softmax_and_scipy_logsumexp():
    H, W = _rand((300, 24), 1), _rand((700, 24), 2, 0.5)
    ids = torch.randint(0, 700, (300,), generator=torch.Generator().manual_seed(4))
    logp, lse = O.token_logprobs(H, W, ids, row_block=64)
    Z = H @ W.T
    ref = torch.log_softmax(Z, dim=1)[torch.arange(300), ids]
    assert np.allclose(logp, ref.numpy(), rtol=1e-13, atol=1e-12)
    assert np.allclose(lse, scipy.special.logsumexp(Z.numpy(), axis=1), rtol=1e-14)
    # |z| < 30: the naive log(sum(exp(z))) is exact enough to compare against
    assert float(Z.abs().max()) < 30
    assert np.allclose(lse, np.log(np.exp(Z.numpy()).sum(1)), rtol=1e-13)


def test_softmax_of_logprobs_sums_to_one():
    H, W = _rand((1, 16), 5), _rand((257, 16), 6)
    V = 257
    logp, _ = O.token_logprobs(H.repeat(V, 1), W, np.arange(V))  # one row, every id
    assert abs(np.exp(logp).sum() - 1.0) < 1e-13


def test_logprobs_equal_logits_closed_form():
    # every vocab row identical -> all logits equal to c = h.w -> lse = c + log V
    V, d = 1000, 4
    W = np.tile(np.array([[300.0, -2.0, 1.0, 0.5]]), (V, 1))
    H = np.array([[4.0, 1.0, 0.0, 2.0]])
    c = 4 * 300.0 - 2.0 + 0 + 1.0
    logp, lse = O.token_logprobs(H, W, [17])
    assert abs(lse[0] - (c + np.log(V))) < 1e-10
    assert abs(logp[0] + np.log(V)) < 1e-12


# ------------------------------------------------------------------------- KL

def test_kl_estimator_properties():
    x = np.array([-3.0, -1e-3, 0.0, 1e-6, 0.07, 2.0])
    kl = O.kl_estimator(np.zeros_like(x), x)       # p - q = x
    literal = np.exp(x) - x - 1.0
    assert kl[2] == 0.0
    assert np.all(kl >= 0)
    # moderate x: equals the literal exp(x) - x - 1
    assert np.allclose(kl[[0, 4, 5]], literal[[0, 4, 5]], rtol=1e-12)
    # small x: the series x^2/2 + x^3/6 + x^4/24
    s = x[[1, 3]]
    assert np.allclose(kl[[1, 3]], s ** 2 / 2 + s ** 3 / 6 + s ** 4 / 24, rtol=1e-9)


# --------------------------------------------------------------- small problem

def _problem(B=8, T=6, G=4, d=12, V=40, seed=11, scale=0.4, ref_noise=0.3):
    g = torch.Generator().manual_seed(seed)
    N = B * T
    Hp = torch.randn(N, d, generator=g, dtype=torch.float64)
    Hr = Hp + ref_noise * torch.randn(N, d, generator=g, dtype=torch.float64)
    W = scale * torch.randn(V, d, generator=g, dtype=torch.float64)
    ids = torch.randint(0, V, (N,), generator=g)
    mask = torch.ones(B, T, dtype=torch.uint8)
    mask[1, T // 2:] = 0
    mask[3, 1:] = 0
    mask[B - 2, :] = 0                  # a sequence with no valid token
    mask = mask.reshape(-1)
    rewards = torch.randn(B, generator=g, dtype=torch.float64)
    A = O.advantages(rewards, G, 1e-4, 1)
    return dict(Hp=Hp, Hr=Hr, W=W, ids=ids, mask=mask, A=A, B=B, T=T, beta=0.04)


def test_loss_at_reference_equal_policy_is_minus_mean_advantage():
    P = _problem()
    f = O.forward(P["Hp"], P["Hp"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"], P["beta"])
    cnt = P["mask"].reshape(P["B"], P["T"]).sum(1).numpy()
    expected = -np.sum(P["A"][cnt > 0]) / P["B"]
    assert np.all(f["kl"] == 0.0) and f["kl_mean"] == 0.0
    assert abs(f["loss"] - expected) < 1e-15
    # and the KL part of the gradient vanishes: with A = 0 the gradient is 0
    b = O.backward(P["Hp"], P["Hp"], P["W"], P["ids"], P["mask"], np.zeros(P["B"]), P["B"], P["T"],
                   P["beta"], want_dW=True)
    assert np.abs(b["dH"]).max() < 1e-15 and np.abs(b["dW"]).max() < 1e-15


def test_beta_zero_loss_and_gradient_reduce_to_weighted_cross_entropy():
    P = _problem()
    f = O.forward(P["Hp"], P["Hr"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"], 0.0)
    cnt = P["mask"].reshape(P["B"], P["T"]).sum(1).numpy()
    assert abs(f["loss"] + np.sum(P["A"][cnt > 0]) / P["B"]) < 1e-15
    # gradient = grad of sum_n w_n A_b CE(z_n, y_n) (library cross entropy)
    H = P["Hp"].clone().requires_grad_(True)
    W = P["W"].clone().requires_grad_(True)
    ce = torch.nn.functional.cross_entropy(H @ W.T, P["ids"], reduction="none")
    w = torch.from_numpy(O.sequence_weights(P["mask"], P["B"], P["T"])[0])
    At = torch.from_numpy(np.repeat(P["A"], P["T"]))
    (w * At * ce).sum().backward()
    b = O.backward(P["Hp"], P["Hr"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"], 0.0,
                   want_dW=True)
    assert np.allclose(b["dH"], H.grad.numpy(), rtol=1e-11, atol=1e-15)
    assert np.allclose(b["dW"], W.grad.numpy(), rtol=1e-11, atol=1e-15)


def _literal_torch_loss(P, H, W, grad_scale=1.0):
    """The objective written as the pages state it, under torch autograd:
    exp(q - q.detach()) * A - beta * (exp(p - q) - (p - q) - 1), p from the
    frozen reference (no gradient), masked mean per sequence, mean over B."""
    B, T = P["B"], P["T"]
    q = torch.log_softmax(H @ W.T, dim=1)[torch.arange(B * T), P["ids"]]
    with torch.no_grad():
        p = torch.log_softmax(P["Hr"] @ W.detach().T, dim=1)[torch.arange(B * T), P["ids"]]
    A = torch.from_numpy(np.repeat(P["A"], T))
    m = P["mask"].double()
    obj = torch.exp(q - q.detach()) * A - P["beta"] * (torch.exp(p - q) - (p - q) - 1)
    per_seq = (obj * m).reshape(B, T).sum(1) / m.reshape(B, T).sum(1).clamp(min=1)
    return -grad_scale * per_seq.mean()


def test_literal_autograd_matches_closed_form_forward_and_backward():
    P = _problem()
    H = P["Hp"].clone().requires_grad_(True)
    W = P["W"].clone().requires_grad_(True)
    L = _literal_torch_loss(P, H, W)
    L.backward()
    f = O.forward(P["Hp"], P["Hr"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"], P["beta"])
    assert abs(f["loss"] - L.item()) < 1e-14
    for g in (1.0, -2.5):
        b = O.backward(P["Hp"], P["Hr"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"],
                       P["beta"], grad_loss=g, want_dW=True)
        assert np.allclose(b["dH"], g * H.grad.numpy(), rtol=1e-10, atol=1e-16)
        assert np.allclose(b["dW"], g * W.grad.numpy(), rtol=1e-10, atol=1e-16)


def test_finite_differences_of_surrogate():
    """exp(q - sg(q)) has value 1 for every H, so the reported loss cannot be
    differentiated numerically; the surrogate sum_n w_n (-A_b q_n + beta KL_n)
    has the same gradient and can."""
    P = _problem(B=4, T=4, G=2, d=8, V=32, seed=21, scale=0.8)
    w, _ = O.sequence_weights(P["mask"], P["B"], P["T"])
    At = np.repeat(P["A"], P["T"])
    m = P["mask"].numpy() > 0
    Hp, Hr, W = P["Hp"].numpy(), P["Hr"].numpy(), P["W"].numpy()
    ids = P["ids"].numpy()

    def Ls(Hp_, Wp_):
        q, _ = O.token_logprobs(Hp_, Wp_, ids)
        p, _ = O.token_logprobs(Hr, W, ids)          # frozen reference lm_head
        kl = O.kl_estimator(q, p)
        return float(np.sum(np.where(m, w * (-At * q + P["beta"] * kl), 0.0)))

    b = O.backward(Hp, Hr, W, ids, P["mask"], P["A"], P["B"], P["T"], P["beta"], want_dW=True)
    h = 1e-6
    rng = np.random.default_rng(0)
    for (i, j) in [tuple(rng.integers(0, s) for s in Hp.shape) for _ in range(12)]:
        Hplus, Hminus = Hp.copy(), Hp.copy()
        Hplus[i, j] += h
        Hminus[i, j] -= h
        fd = (Ls(Hplus, W) - Ls(Hminus, W)) / (2 * h)
        assert abs(fd - b["dH"][i, j]) <= 1e-7 * max(1.0, abs(b["dH"][i, j])) + 1e-9
    for (i, j) in [tuple(rng.integers(0, s) for s in W.shape) for _ in range(12)]:
        Wplus, Wminus = W.copy(), W.copy()
        Wplus[i, j] += h
        Wminus[i, j] -= h
        fd = (Ls(Hp, Wplus) - Ls(Hp, Wminus)) / (2 * h)
        assert abs(fd - b["dW"][i, j]) <= 1e-7 * max(1.0, abs(b["dW"][i, j])) + 1e-9


def test_row_structure_and_row_subsets():
    P = _problem()
    b = O.backward(P["Hp"], P["Hr"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"],
                   P["beta"], want_dZ=True)
    assert np.all(np.abs(b["dZ"].sum(1)) < 1e-15)              # softmax - onehot sums to 0
    masked = P["mask"].numpy() == 0
    assert np.all(b["dZ"][masked] == 0) and np.all(b["dH"][masked] == 0)
    rows = np.array([0, 5, 9, 10, 33, 47])
    bs = O.backward(P["Hp"], P["Hr"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"],
                    P["beta"], rows=rows, row_block=4)
    assert np.array_equal(bs["dH"], b["dH"][rows]) or np.allclose(bs["dH"], b["dH"][rows], rtol=1e-14, atol=1e-18)


def test_masked_rows_may_carry_out_of_range_ids():
    P = _problem()
    ids = P["ids"].clone()
    ids[P["mask"] == 0] = -100                  # a typical ignore label
    f = O.forward(P["Hp"], P["Hr"], P["W"], ids, P["mask"], P["A"], P["B"], P["T"], P["beta"])
    f0 = O.forward(P["Hp"], P["Hr"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"], P["beta"])
    assert f["loss"] == f0["loss"]


# -------------------------------------------------------------- memory model

def test_memory_model_against_printed_figures():
    with open(os.path.join(GOLDEN, "memory_figures.txt")) as fh:
        rows = [l.split("|") for l in fh if l.strip() and not l.startswith("#")]
    assert len(rows) == 4
    for name, r, v, mult, bpe, printed, tol, _cite in rows:
        val = O.logit_memory_gib(int(r), int(v), int(mult), int(bpe))
        assert abs(val - float(printed)) <= float(tol), (name.strip(), val, printed)
    assert abs(O.hidden_state_memory_gib(8, 64000, 4096) - 1.953125) < 1e-12


# ------------------------------------------------------ optional variants

XF = {"multiply": 1.5, "divide": 1.2, "softcap": 3.0, "temperature": 0.7}


def test_scale_and_temperature_equal_scaled_weights():
    H, W = _rand((40, 10), 31), _rand((90, 10), 32, 0.7)
    ids = np.arange(40) % 90
    for xf, factor in [({"multiply": 2.0}, 2.0), ({"divide": 4.0}, 0.25),
                       ({"temperature": 2.0}, 0.5), ({"multiply": 3.0, "divide": 2.0,
                                                      "temperature": 0.5}, 3.0)]:
        a, la = O.token_logprobs(H, W, ids, xform=xf)
        b, lb = O.token_logprobs(H, factor * W, ids)
        assert np.allclose(a, b, rtol=1e-13, atol=1e-13) and np.allclose(la, lb, rtol=1e-13)


def test_softcap_bounds_and_large_cap_limit():
    H, W = _rand((30, 8), 33, 3.0), _rand((50, 8), 34, 2.0)
    Z, g = O.transform_logits((H @ W.T).numpy(), {"softcap": 5.0})
    assert np.all(np.abs(Z) < 5.0) and np.all((g > 0) & (g <= 1.0))
    ids = np.arange(30)
    a, _ = O.token_logprobs(H, W, ids, xform={"softcap": 1e7})
    b, _ = O.token_logprobs(H, W, ids)
    assert np.allclose(a, b, rtol=1e-9, atol=1e-9)


def test_transform_matches_torch_literal_log_softmax():
    H, W = _rand((60, 12), 35), _rand((80, 12), 36, 0.6)
    ids = torch.randint(0, 80, (60,), generator=torch.Generator().manual_seed(7))
    z = (H @ W.T) * XF["multiply"] / XF["divide"]
    z = XF["softcap"] * torch.tanh(z / XF["softcap"]) / XF["temperature"]
    ref = torch.log_softmax(z, dim=1)[torch.arange(60), ids]
    a, _ = O.token_logprobs(H, W, ids, xform=XF)
    assert np.allclose(a, ref.numpy(), rtol=1e-13, atol=1e-12)


def _literal_torch_loss_v(P, H, W, token_level=False, xform=None):
    B, T = P["B"], P["T"]

    def f(z):
        if not xform:
            return z
        z = z * xform["multiply"] / xform["divide"]
        z = xform["softcap"] * torch.tanh(z / xform["softcap"])
        return z / xform["temperature"]

    q = torch.log_softmax(f(H @ W.T), dim=1)[torch.arange(B * T), P["ids"]]
    with torch.no_grad():
        p = torch.log_softmax(f(P["Hr"] @ W.detach().T), dim=1)[torch.arange(B * T), P["ids"]]
    A = torch.from_numpy(np.repeat(P["A"], T))
    m = P["mask"].double()
    obj = torch.exp(q - q.detach()) * A - P["beta"] * (torch.exp(p - q) - (p - q) - 1)
    if token_level:
        return -(obj * m).sum() / m.sum().clamp(min=1)
    per_seq = (obj * m).reshape(B, T).sum(1) / m.reshape(B, T).sum(1).clamp(min=1)
    return -per_seq.mean()


@pytest.mark.parametrize("token_level,xform", [(True, None), (False, XF), (True, XF)],
                         ids=["token-level", "transforms", "both"])
def test_variants_match_literal_autograd(token_level, xform):
    P = _problem()
    H = P["Hp"].clone().requires_grad_(True)
    W = P["W"].clone().requires_grad_(True)
    L = _literal_torch_loss_v(P, H, W, token_level, xform)
    L.backward()
    f = O.forward(P["Hp"], P["Hr"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"],
                  P["beta"], token_level=token_level, xform=xform)
    assert abs(f["loss"] - L.item()) < 1e-14
    b = O.backward(P["Hp"], P["Hr"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"],
                   P["beta"], want_dW=True, token_level=token_level, xform=xform)
    assert np.allclose(b["dH"], H.grad.numpy(), rtol=1e-10, atol=1e-16)
    assert np.allclose(b["dW"], W.grad.numpy(), rtol=1e-10, atol=1e-16)


def test_finite_differences_with_softcap_and_token_level():
    P = _problem(B=4, T=4, G=2, d=8, V=32, seed=22, scale=1.2)
    xf = {"softcap": 2.0, "temperature": 0.8}
    w, _ = O.sequence_weights(P["mask"], P["B"], P["T"], token_level=True)
    At = np.repeat(P["A"], P["T"])
    m = P["mask"].numpy() > 0
    Hp, Hr, W = P["Hp"].numpy(), P["Hr"].numpy(), P["W"].numpy()
    ids = P["ids"].numpy()

    def Ls(Hp_):
        q, _ = O.token_logprobs(Hp_, W, ids, xform=xf)
        p, _ = O.token_logprobs(Hr, W, ids, xform=xf)
        return float(np.sum(np.where(m, w * (-At * q + P["beta"] * O.kl_estimator(q, p)), 0.0)))

    b = O.backward(Hp, Hr, W, ids, P["mask"], P["A"], P["B"], P["T"], P["beta"],
                   token_level=True, xform=xf)
    h = 1e-6
    rng = np.random.default_rng(1)
    for (i, j) in [tuple(rng.integers(0, s) for s in Hp.shape) for _ in range(12)]:
        Hplus, Hminus = Hp.copy(), Hp.copy()
        Hplus[i, j] += h
        Hminus[i, j] -= h
        fd = (Ls(Hplus) - Ls(Hminus)) / (2 * h)
        assert abs(fd - b["dH"][i, j]) <= 1e-7 * max(1.0, abs(b["dH"][i, j])) + 1e-9


def test_token_level_reference_equal_policy():
    P = _problem()
    f = O.forward(P["Hp"], P["Hp"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"],
                  P["beta"], token_level=True)
    m = P["mask"].numpy().reshape(P["B"], P["T"]).astype(float)
    expected = -np.sum(m.sum(1) * P["A"]) / m.sum()
    assert abs(f["loss"] - expected) < 1e-15 and f["kl_mean"] == 0.0


def test_given_reference_logprobs_equal_computed_ones():
    P = _problem()
    f = O.forward(P["Hp"], P["Hr"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"], P["beta"])
    g = O.forward(P["Hp"], None, P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"], P["beta"],
                  logp_ref_given=f["logp_ref"])
    assert g["loss"] == f["loss"] and np.array_equal(g["kl"], f["kl"])
    b1 = O.backward(P["Hp"], P["Hr"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"], P["beta"])
    b2 = O.backward(P["Hp"], None, P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"], P["beta"],
                    logp_ref_given=f["logp_ref"])
    assert np.allclose(b1["dH"], b2["dH"], rtol=1e-14, atol=1e-18)


# ------------------------------------------------------------ KL variants

def _literal_kl_mode_loss(P, H, W, kl_mode):
    B, T = P["B"], P["T"]
    q = torch.log_softmax(H @ W.T, dim=1)[torch.arange(B * T), P["ids"]]
    with torch.no_grad():
        p = torch.log_softmax(P["Hr"] @ W.detach().T, dim=1)[torch.arange(B * T), P["ids"]]
    A = torch.from_numpy(np.repeat(P["A"], T))
    m = P["mask"].double()
    if kl_mode == 1:
        adv_term = torch.exp(q - q) * A                  # the detach removed
    else:
        adv_term = torch.exp(q - q.detach()) * A
    k3 = torch.exp(p - q) - (p - q) - 1
    if kl_mode in (0, 1):
        kl = k3
    elif kl_mode == 2:
        kl = torch.exp(q) * k3                           # the extra Q factor
    else:
        r = torch.exp(p - q)                             # forward KL, samples from Q
        kl = r * torch.log(r) - (r - 1)
    obj = adv_term - P["beta"] * kl
    per_seq = (obj * m).reshape(B, T).sum(1) / m.reshape(B, T).sum(1).clamp(min=1)
    return -per_seq.mean()


@pytest.mark.parametrize("kl_mode", [0, 1, 2, 3])
def test_kl_modes_match_literal_autograd(kl_mode):
    P = _problem()
    H = P["Hp"].clone().requires_grad_(True)
    W = P["W"].clone().requires_grad_(True)
    L = _literal_kl_mode_loss(P, H, W, kl_mode)
    L.backward()
    f = O.forward(P["Hp"], P["Hr"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"],
                  P["beta"], kl_mode=kl_mode)
    assert abs(f["loss"] - L.item()) < 1e-13
    b = O.backward(P["Hp"], P["Hr"], P["W"], P["ids"], P["mask"], P["A"], P["B"], P["T"],
                   P["beta"], want_dW=True, kl_mode=kl_mode)
    assert np.allclose(b["dH"], H.grad.numpy(), rtol=1e-10, atol=1e-16)
    assert np.allclose(b["dW"], W.grad.numpy(), rtol=1e-10, atol=1e-16)


def test_kl_mode_estimators_vanish_at_equal_policies_and_are_nonnegative():
    x = np.linspace(-3, 3, 61)
    q = -np.abs(x) - 2.0
    for mode in (0, 2, 3):
        k = O.kl_estimator(q, q + x, mode)
        assert np.all(k >= -1e-15)
        assert O.kl_estimator(q[:1], q[:1], mode)[0] == 0.0
    # mode 3 small x: x^2/2 + x^3/3 + ...
    s = np.array([1e-3, -2e-3])
    assert np.allclose(O.kl_estimator(np.zeros(2), s, 3), s ** 2 / 2 + s ** 3 / 3, rtol=1e-5)


# ------------------------------------------------------------------ FP8 E4M3

def _torch_e4m3_codes(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch_float8_on_all_codes():
    c = np.arange(256, dtype=np.uint8)
    d = O.e4m3_decode(c)
    t = torch.from_numpy(c).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(d), np.isnan(t))
    assert np.isnan(d).sum() == 2                      # 0x7F and 0xFF only
    ok = ~np.isnan(d)
    assert np.array_equal(d[ok], t[ok])
    assert d[0x7E] == 448.0 and d[0x01] == 2.0 ** -9 and d[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_torch_cast_including_exact_ties():
    g = np.random.default_rng(11)
    mags = np.exp2(g.uniform(-12, np.log2(448.0), 20000))
    x = (mags * g.choice([-1.0, 1.0], mags.size)).astype(np.float32)
    # exact midpoints between neighbouring codes (ties go to the even code)
    vals = O.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (vals[:-1] + vals[1:]) / 2)  # exact in f32
    x = np.concatenate([x, mids, -mids, np.float32([0.0, -0.0, 1e-30, -1e-30, 448.0, -448.0])])
    assert np.array_equal(O.e4m3_encode(x), _torch_e4m3_codes(x))


def test_e4m3_encode_saturates_roundtrips_and_flags_nan():
    x = np.float32([1000.0, -1e6, 449.0, 463.9, np.nan])
    assert list(O.e4m3_encode(x)) == [0x7E, 0xFE, 0x7E, 0x7E, 0x7F]
    c = np.array([k for k in range(256) if k not in (0x7F, 0xFF)], dtype=np.uint8)
    again = O.e4m3_encode(O.e4m3_decode(c).astype(np.float32))
    assert np.array_equal(O.e4m3_decode(again), O.e4m3_decode(c))
    assert np.array_equal(again[c != 0x80], c[c != 0x80])


def test_quantize_rows_hand_worked_row_and_zero_row():
    # amax 4: scale 4/448 = 1/112, inv 112; scaled row 112, -224, 56, 448
    # = 1.75 * 2^6, -1.75 * 2^7, 1.75 * 2^5, 1.75 * 2^8: exponent fields 13, 14,
    # 12, 15 with mantissa 6
    q, s = O.quantize_e4m3_rows(np.float32([[1.0, -2.0, 0.5, 4.0], [0.0, 0.0, 0.0, 0.0]]))
    assert list(q[0]) == [0x6E, 0xF6, 0x66, 0x7E]
    assert s[0] == np.float32(4.0) / np.float32(448.0)
    assert list(q[1]) == [0, 0, 0, 0] and s[1] == 1.0
    assert np.allclose(O.dequantize_rows(q[:1], s[:1]), [[1.0, -2.0, 0.5, 4.0]], rtol=1e-6)


def test_quantize_rows_error_bound_and_dequantize_matches_torch():
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(64, 300, generator=g) * torch.exp2(torch.randint(-20, 20, (64, 1), generator=g)))
    x = x.to(torch.bfloat16)
    q, s = O.quantize_e4m3_rows(x)
    xf = x.double().numpy()
    deq = O.dequantize_rows(q, s)
    assert np.all(np.abs(O.e4m3_decode(q)).max(axis=1) == 448.0)
    # normal codes: half a unit of 3 mantissa bits, 2^-4 relative (plus the
    # float32 roundings of inv, scale and the product); subnormal codes: half
    # their spacing 2^-9, in units of the row scale
    y = np.abs(xf) * (448.0 / np.abs(xf).max(axis=1, keepdims=True))
    bound = np.where(y >= 2.0 ** -6, np.abs(xf) * (2.0 ** -4 + 1e-6),
                     2.0 ** -10 * s.astype(np.float64)[:, None] * (1 + 1e-6) + np.abs(xf) * 1e-6)
    assert np.all(np.abs(deq - xf) <= bound)
    t = torch.from_numpy(q).view(torch.float8_e4m3fn).double() * torch.from_numpy(s).double()[:, None]
    assert np.array_equal(deq, t.numpy())
