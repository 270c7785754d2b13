"""The forward + backward step captured in a CUDA graph and replayed.

Every library call is stream-ordered with no host synchronisation, so a
training step can be captured once and replayed. The first call on a device
sets kernel attributes and must come before capture; the test makes one eager
call first, then captures, replays on new inputs copied into the captured
buffers, and compares with eager results bit for bit."""
import pytest
import torch

from grpo_loss_gb300 import workloads as WL

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float8_e4m3fn], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("w", [WL.SMALL["qwen2.5-small"], WL.SMALL["gpt-oss-small"]],
                         ids=lambda w: w.name)
def test_step_replays_from_a_cuda_graph(w, dtype):
    """With e4m3 operands the captured step also holds the row quantization of
    H_pol, H_ref and W."""
    import grpo_loss_gb300 as G
    dev = torch.device("cuda")
    eng = G.GRPOLoss(w.B, w.T, w.d, w.V, w.G, beta=w.beta, eps=w.eps, dtype=dtype,
                     chunk_rows=256, compute_dW=True)
    a = {k: v.to(dev) for k, v in WL.make_inputs(w).items() if v is not None}
    b = {k: v.to(dev) for k, v in WL.make_inputs(w.scaled(w.name, seed=w.seed + 9)).items()
         if v is not None}
    static = {k: v.clone() for k, v in a.items()}
    dH = torch.empty(a["H_pol"].shape, dtype=torch.bfloat16, device=dev)

    def step(d):
        adv = eng.advantages(d["rewards"])
        eng.forward(d["H_pol"], d["H_ref"], d["W"], d["ids"], d["mask"], adv)
        eng.backward(d["H_pol"], d["W"], d["ids"], d["mask"], adv, 1.0, dH=dH)

    def snapshot():
        return (eng.loss.clone(), eng.kl_mean.clone(), eng.logp_pol.clone(), dH.clone(),
                eng.dW.clone())

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(static)                                   # first call: sets kernel attributes
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(static)
    results = []
    for src in (a, b):
        for k in static:
            static[k].copy_(src[k])
        graph.replay()
        torch.cuda.synchronize()
        got = snapshot()
        step(src)                                      # eager, same buffers
        torch.cuda.synchronize()
        eng.check()
        want = snapshot()
        for x, y in zip(got, want):
            assert torch.equal(x, y)
        results.append(got[0].item())
    assert results[0] != results[1]                    # the replay saw the new inputs
