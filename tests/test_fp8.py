"""GPU parity of the e4m3 (FP8) operand path against the float64 oracle.

* The row quantizer is compared byte for byte (codes) and bit for bit
  (scales) with the oracle's quantizer, including rows of zeros, negative
  zeros, values that round into the subnormals or to zero, and exact ties.
* The loss runs on e4m3 operands made two ways. (a) The GPU quantizes the
  seeded float32/bf16 workloads with its own kernel; the oracle quantizes the
  same host tensors with its own codec and evaluates the loss on the
  dequantized operands. (b) The input generator draws random codes and row
  scales, handed to both sides as they are.
Forward outputs, dH (the gradient with respect to the dequantized H_pol) and
dW (with respect to the dequantized W) are held to the same tolerances as
the bf16 path.
"""
import numpy as np
import pytest
import torch

from grpo_loss_gb300 import workloads as WL
from oracle import grpo_oracle as O
from tests.parity_util import TOL_DH_L2, TOL_REL, oracle_adv, rel_err, rel_l2, x_and_kl_close

pytestmark = pytest.mark.gpu

F8 = torch.float8_e4m3fn


def _gpu_quantize(x):
    import grpo_loss_gb300 as G
    q, s = G.quantize_e4m3_rows(x.cuda())
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def _special_rows(cols: int) -> torch.Tensor:
    """Rows that exercise the edges of the codec (float32)."""
    vals = O.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2          # exact ties once scaled by 448 / 448
    rows = []
    z = np.zeros(cols, np.float32)
    rows.append(z.copy())                                       # zeros: scale 1, codes 0
    r = z.copy()
    r[::2] = -0.0
    r[1] = 1.0
    rows.append(r)                                              # negative zeros kept
    r = np.full(cols, 1e-6, np.float32)
    r[0] = 448.0
    r[1::3] = -1e-7                                             # round to (negative) zero
    r[2::5] = 0.75 * 2.0 ** -9                                  # rounds to the smallest subnormal
    r[3::7] = 2.5 * 2.0 ** -9                                   # subnormal tie: to code 2
    rows.append(r.astype(np.float32))
    r = np.resize(np.concatenate([mids, -mids]), cols).astype(np.float32)
    r[0] = 448.0                                                # amax 448: inv = 1, ties stay ties
    rows.append(r)
    g = np.random.default_rng(3)
    rows.append((g.standard_normal(cols) * np.exp2(g.uniform(-30, 30, cols))).astype(np.float32))
    return torch.from_numpy(np.stack(rows))


@pytest.mark.parametrize("rows,cols,dtype", [(37, 4096, torch.bfloat16), (300, 2880, torch.float32),
                                             (5, 16, torch.bfloat16), (1, 8192, torch.float32)])
def test_quantizer_matches_oracle_bit_for_bit(rows, cols, dtype):
    g = torch.Generator().manual_seed(rows * 31 + cols)
    x = torch.randn(rows, cols, generator=g) * torch.exp2(torch.randint(-24, 24, (rows, 1), generator=g))
    x = x.to(dtype)
    q, s = _gpu_quantize(x)
    qo, so = O.quantize_e4m3_rows(x)
    assert np.array_equal(q, qo)
    assert np.array_equal(s.view(np.uint32), so.view(np.uint32))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantizer_edge_rows(dtype):
    x = _special_rows(512).to(dtype)
    q, s = _gpu_quantize(x)
    qo, so = O.quantize_e4m3_rows(x)
    assert np.array_equal(q, qo), np.argwhere(q != qo)[:8]
    assert np.array_equal(s.view(np.uint32), so.view(np.uint32))
    assert s[0] == 1.0 and not q[0].any()


def test_quantizer_rejects_bad_arguments():
    import grpo_loss_gb300 as G
    with pytest.raises(G.GrpoError) as e:
        G.quantize_e4m3_rows(torch.zeros(4, 24, device="cuda"))   # cols % 16 != 0
    assert e.value.status == 2
    with pytest.raises(ValueError):
        G.quantize_e4m3_rows(torch.zeros(4, 32, dtype=torch.float16, device="cuda"))


# ------------------------------------------------------------------ the loss

def _oracle_operands(inp, ref: bool = True):
    """The oracle's own quantization of the workload's float tensors."""
    out = {}
    names = ("H_pol", "H_ref", "W") if ref else ("H_pol", "W")
    for k in names:
        q, s = O.quantize_e4m3_rows(inp[k])
        out[k] = O.dequantize_rows(q, s)
    return out


def _check(w, inp, ops, adv32, res, dW=False, xf=None, token_level=False, given=None,
           kl_mode=0):
    Hr = ops.get("H_ref")
    f = O.forward(ops["H_pol"], Hr, ops["W"], inp["ids"], inp["mask"], adv32.double(), w.B, w.T,
                  w.beta, token_level=token_level, xform=xf, logp_ref_given=given,
                  kl_mode=kl_mode)
    g = O.backward(ops["H_pol"], Hr, ops["W"], inp["ids"], inp["mask"], adv32.double(), w.B, w.T,
                   w.beta, token_level=token_level, xform=xf, logp_ref_given=given,
                   want_dW=dW, kl_mode=kl_mode)
    m = inp["mask"].numpy() > 0
    assert rel_err(res["logp_pol"][m], f["logp_pol"][m]) < TOL_REL
    assert rel_err(res["logp_ref"][m], f["logp_ref"][m]) < TOL_REL
    assert rel_err(res["lse_pol"][m], f["lse_pol"][m]) < TOL_REL
    assert abs(res["loss"] - f["loss"]) <= TOL_REL * abs(f["loss"]), (res["loss"], f["loss"])
    assert abs(res["kl_mean"] - f["kl_mean"]) <= TOL_REL * abs(f["kl_mean"]) + 1e-12
    assert rel_l2(res["dH"], g["dH"]) < TOL_DH_L2, rel_l2(res["dH"], g["dH"])
    assert np.all(res["dH"][~m] == 0)
    if dW:
        assert rel_l2(res["dW"], g["dW"]) < TOL_DH_L2, rel_l2(res["dW"], g["dW"])


def _engine_run(w, inp, adv32, want_dW=False, chunk_rows=0, given=None, **variant):
    import grpo_loss_gb300 as G
    dev = torch.device("cuda")
    eng = G.GRPOLoss(w.B, w.T, w.d, w.V, w.G, beta=w.beta, eps=w.eps,
                     std_unbiased=w.std_unbiased, chunk_rows=chunk_rows, dtype=F8, device=dev,
                     compute_dW=want_dW, ref_logp_given=given is not None, **variant)
    Hp, Wd = inp["H_pol"].to(dev), inp["W"].to(dev)
    ids, mask, adv = inp["ids"].to(dev), inp["mask"].to(dev), adv32.to(dev)
    if given is not None:
        loss, klm, lp, lr = eng.forward(Hp, None, Wd, ids, mask, adv, logp_ref=given.to(dev))
    else:
        loss, klm, lp, lr = eng.forward(Hp, inp["H_ref"].to(dev), Wd, ids, mask, adv)
    dH = eng.backward(Hp, Wd, ids, mask, adv, 1.0)
    torch.cuda.synchronize()
    eng.check()
    assert dH.dtype == torch.bfloat16
    out = {"loss": float(loss.item()), "kl_mean": float(klm.item()),
           "logp_pol": lp.cpu().double().numpy(), "logp_ref": lr.cpu().double().numpy(),
           "lse_pol": eng.lse_pol.cpu().double().numpy(), "dH": dH.float().cpu().numpy()}
    if want_dW:
        out["dW"] = eng.dW.cpu().numpy()
    return out


XF = {"logit_multiply": 1.5, "logit_divide": 1.2, "softcap": 2.0, "temperature": 0.7}

CASES = [
    ("llama-dW", WL.SMALL["llama3.1-small"], dict(want_dW=True)),
    ("qwen2.5-chunks", WL.SMALL["qwen2.5-small"], dict(chunk_rows=256, want_dW=True)),
    # d = 192: the second 128-element K block is half past the row (zero fill)
    ("gptoss-d192-ktail", WL.SMALL["gpt-oss-small"], {}),
    ("tiny-f32-transforms-token", WL.TINY, dict(XF, token_level=True)),
    ("qwen3-kl-forward", WL.SMALL["qwen3-small"], {"kl_mode": 3}),
    ("llama-pairs", WL.SMALL["llama3.1-small"], dict(cluster_mode=1, want_dW=True)),
]


@pytest.mark.parametrize("name,w,variant", CASES, ids=[c[0] for c in CASES])
def test_e4m3_loss_matches_oracle(name, w, variant):
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    variant = dict(variant)
    want_dW = variant.pop("want_dW", False)
    chunk_rows = variant.pop("chunk_rows", 0)
    res = _engine_run(w, inp, adv32, want_dW=want_dW, chunk_rows=chunk_rows, **variant)
    xf = None
    if any(k in variant for k in XF):
        xf = {"multiply": variant.get("logit_multiply", 0.0),
              "divide": variant.get("logit_divide", 0.0),
              "softcap": variant.get("softcap", 0.0),
              "temperature": variant.get("temperature", 0.0)}
    _check(w, inp, _oracle_operands(inp), adv32, res, dW=want_dW, xf=xf,
           token_level=variant.get("token_level", False), kl_mode=variant.get("kl_mode", 0))


def test_e4m3_with_reference_logprobs_given():
    w = WL.SMALL["qwen2.5-small"]
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    ops = _oracle_operands(inp)
    given = O.token_logprobs(ops["H_ref"], ops["W"], inp["ids"])[0]
    given = np.where(inp["mask"].numpy() > 0, given, 0.0)
    res = _engine_run(w, inp, adv32, given=torch.from_numpy(given).float())
    ops.pop("H_ref")
    _check(w, inp, ops, adv32, res, given=torch.from_numpy(given).float().double().numpy())


def test_e4m3_random_codes_and_scales_through_the_c_abi():
    """Every code pattern (subnormals included) with arbitrary row scales,
    given to the library's e4m3 entry points and to the oracle unchanged."""
    import grpo_loss_gb300 as G
    w = WL.SMALL["llama3.1-small"]
    inp = WL.make_inputs(w)
    ops = WL.random_e4m3_operands(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    dev = torch.device("cuda")
    p = G.make_problem(w.B, w.T, w.d, w.V, w.G, beta=w.beta, eps=w.eps,
                       std_unbiased=w.std_unbiased, dtype=F8, compute_dW=True)
    fb, bb = G.workspace_size(p)
    wsf = torch.empty(fb, dtype=torch.uint8, device=dev)
    wsb = torch.empty(bb, dtype=torch.uint8, device=dev)
    d = {k: v.to(dev) for k, v in ops.items()}
    ids, mask, adv = inp["ids"].to(dev), inp["mask"].to(dev), adv32.to(dev)
    N = w.N
    lp, lr, lse = (torch.empty(N, device=dev) for _ in range(3))
    loss, klm = torch.empty(1, device=dev), torch.empty(1, device=dev)
    G.loss_fwd_e4m3(p, d["q_pol"], d["s_pol"], d["q_ref"], d["s_ref"], d["q_W"], d["s_W"], ids,
                    mask, adv, lp, lr, lse, loss, klm, wsf)
    dH = torch.empty(N, w.d, dtype=torch.bfloat16, device=dev)
    dW = torch.empty(w.V, w.d, dtype=torch.float32, device=dev)
    G.loss_bwd_e4m3(p, d["q_pol"], d["s_pol"], d["q_W"], d["s_W"], ids, mask, adv, lp, lr, lse,
                    1.0, dH, wsb, dW=dW)
    torch.cuda.synchronize()
    assert G.device_status(wsf) == 0 and G.device_status(wsb) == 0
    res = {"loss": float(loss.item()), "kl_mean": float(klm.item()),
           "logp_pol": lp.cpu().double().numpy(), "logp_ref": lr.cpu().double().numpy(),
           "lse_pol": lse.cpu().double().numpy(), "dH": dH.float().cpu().numpy(),
           "dW": dW.cpu().numpy()}
    oops = {"H_pol": O.dequantize_rows(ops["q_pol"], ops["s_pol"]),
            "H_ref": O.dequantize_rows(ops["q_ref"], ops["s_ref"]),
            "W": O.dequantize_rows(ops["q_W"], ops["s_W"])}
    _check(w, inp, oops, adv32, res, dW=True)


def test_e4m3_problems_need_the_e4m3_entry_points():
    import grpo_loss_gb300 as G
    w = WL.TINY
    dev = torch.device("cuda")
    p8 = G.make_problem(w.B, w.T, w.d, w.V, w.G, dtype=F8)
    pb = G.make_problem(w.B, w.T, w.d, w.V, w.G, dtype=torch.bfloat16)
    fb, _ = G.workspace_size(p8)
    ws = torch.empty(max(fb, G.workspace_size(pb)[0]), dtype=torch.uint8, device=dev)
    N = w.N
    H = torch.zeros(N, w.d, dtype=torch.bfloat16, device=dev)
    Wt = torch.zeros(w.V, w.d, dtype=torch.bfloat16, device=dev)
    ids = torch.zeros(N, dtype=torch.int32, device=dev)
    mask = torch.ones(N, dtype=torch.uint8, device=dev)
    adv = torch.zeros(w.B, device=dev)
    outs = [torch.empty(N, device=dev) for _ in range(3)] + [torch.empty(1, device=dev)] * 2
    with pytest.raises(G.GrpoError) as e:
        G.loss_fwd(p8, H, H, Wt, ids, mask, adv, *outs, ws)
    assert e.value.status == 1
    q = torch.zeros(N, w.d, dtype=torch.uint8, device=dev)
    qW = torch.zeros(w.V, w.d, dtype=torch.uint8, device=dev)
    s, sW = torch.ones(N, device=dev), torch.ones(w.V, device=dev)
    with pytest.raises(G.GrpoError) as e:
        G.loss_fwd_e4m3(pb, q, s, q, s, qW, sW, ids, mask, adv, *outs, ws)
    assert e.value.status == 1
    # d % 16 != 0 is refused for e4m3 problems
    with pytest.raises(G.GrpoError) as e:
        G.workspace_size(G.make_problem(2, 8, 40, 64, 2, dtype=F8))
    assert e.value.status == 2


# ------------------------------------------------------------- full size

class _SampledRows:
    """Dequantized rows of a large operand, held for a sample of rows only;
    indexing with sampled row numbers returns them (the oracle's per-row
    functions read only the rows they are asked for)."""

    def __init__(self, rows, data):
        self.pos = {int(r): i for i, r in enumerate(rows)}
        self.data = data

    def __getitem__(self, idx):
        idx = np.asarray(idx).reshape(-1)
        return self.data[[self.pos[int(i)] for i in idx]]


@pytest.mark.slow
def test_e4m3_full_size_llama_sampled_rows():
    """The Llama-3.1-8B-shaped 20K x 8 head with e4m3 operands quantized on the
    GPU, in the benchmark's launch configuration: sampled rows against the
    oracle's own quantization, the GPU's codes of those rows against the
    oracle's byte for byte, and the loss against its definition over the
    per-token outputs."""
    import grpo_loss_gb300 as G
    w = WL.LLAMA31_8B_20K
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    res = _engine_run(w, inp, adv32)
    rows = WL.sample_rows(w, inp["mask"], count=64)
    # codes of the sampled rows, quantized on the GPU, byte for byte
    qg, sg = G.quantize_e4m3_rows(inp["H_pol"][torch.from_numpy(rows)].cuda())
    qo, so = O.quantize_e4m3_rows(inp["H_pol"][torch.from_numpy(rows)])
    assert np.array_equal(qg.cpu().numpy(), qo) and np.array_equal(sg.cpu().numpy(), so)
    Hp = _SampledRows(rows, O.dequantize_rows(qo, so))
    Hr = _SampledRows(rows, O.dequantize_rows(*O.quantize_e4m3_rows(inp["H_ref"][torch.from_numpy(rows)])))
    Wf = np.empty((w.V, w.d))
    for r0 in range(0, w.V, 8192):
        Wf[r0:r0 + 8192] = O.dequantize_rows(*O.quantize_e4m3_rows(inp["W"][r0:r0 + 8192]))
    q, lse = O.token_logprobs(Hp, Wf, inp["ids"], rows=rows)
    p, _ = O.token_logprobs(Hr, Wf, inp["ids"], rows=rows)
    assert rel_err(res["logp_pol"][rows], q) < TOL_REL
    assert rel_err(res["logp_ref"][rows], p) < TOL_REL
    assert rel_err(res["lse_pol"][rows], lse) < TOL_REL
    x_and_kl_close(res["logp_ref"][rows] - res["logp_pol"][rows], p - q, "e4m3")
    g = O.backward(Hp, Hr, Wf, inp["ids"], inp["mask"], adv32.double(), w.B, w.T, w.beta,
                   rows=rows)
    assert rel_l2(res["dH"][rows], g["dH"]) < TOL_DH_L2
    for i in range(rows.size):
        assert rel_l2(res["dH"][rows[i]], g["dH"][i]) < 3 * TOL_DH_L2, int(rows[i])
    wts, _ = O.sequence_weights(inp["mask"], w.B, w.T)
    kl = O.kl_estimator(res["logp_pol"], res["logp_ref"])
    A = np.repeat(adv32.double().numpy(), w.T)
    m = inp["mask"].numpy() > 0
    loss = float(np.sum(np.where(m, wts * (-A + w.beta * kl), 0.0)))
    assert abs(res["loss"] - loss) <= 1e-5 * abs(loss) + 1e-9
    torch.cuda.empty_cache()


def test_e4m3_bad_token_is_reported():
    """A valid row whose id is V, on a vocab whose last tile is ragged (V =
    3000), so the id falls inside the last chunk's column window: the device
    reports GRPO_ERR_BAD_TOKEN and reads no scale past the end of s_W."""
    import grpo_loss_gb300 as G
    w = WL.SMALL["qwen2.5-small"]
    assert w.V % 256 != 0 and (w.V % 256) % 32 != 0
    inp = WL.make_inputs(w)
    assert int(inp["mask"][3]) == 1
    ids = inp["ids"].clone()
    ids[3] = w.V
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    dev = torch.device("cuda")
    eng = G.GRPOLoss(w.B, w.T, w.d, w.V, w.G, beta=w.beta, eps=w.eps,
                     std_unbiased=w.std_unbiased, dtype=F8, device=dev)
    eng.forward(inp["H_pol"].to(dev), inp["H_ref"].to(dev), inp["W"].to(dev), ids.to(dev),
                inp["mask"].to(dev), adv32.to(dev))
    torch.cuda.synchronize()
    assert G.device_status(eng.ws_fwd) == 6
