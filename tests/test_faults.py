"""Device-side failure detection, exercised without faulting the GPU.

A testing hook makes one CTA of the forward GEMM withhold a shared-memory
stage, so its bounded MMA wait runs out (a barrier that nothing arrives on).
The kernel must record GRPO_ERR_TIMEOUT, leave through its orderly abort
path (drain its copies, free tensor memory) within the short wait limit,
and leave the context usable: the next clean call returns correct results.
"""
import time

import numpy as np
import pytest
import torch

from grpo_loss_gb300 import _lib as L
from grpo_loss_gb300 import workloads as WL
from oracle import grpo_oracle as O
from tests.parity_util import TOL_REL, gpu_run, oracle_adv, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cluster_mode", [0, 1], ids=["single", "pairs"])
def test_pipeline_wait_timeout_is_reported_and_context_survives(cluster_mode):
    import grpo_loss_gb300 as G
    w = WL.SMALL["llama3.1-small"]
    inp = WL.make_inputs(w)
    adv32 = torch.from_numpy(oracle_adv(w, inp)).float()
    lib = L.lib()
    assert lib.grpo_test_pipeline_stall(1, 200) == 0
    try:
        t0 = time.time()
        res = gpu_run(w, inp, adv32, want_bwd=False, check=False, cluster_mode=cluster_mode)
        status = G.device_status(res["engine"].ws_fwd)
        elapsed = time.time() - t0
    finally:
        assert lib.grpo_test_pipeline_stall(0, 0) == 0
    assert status == 5, status                     # GRPO_ERR_TIMEOUT
    assert elapsed < 30.0
    assert G.device_status(res["engine"].ws_fwd) == 0   # read clears the word
    # the context is intact: a clean call matches the oracle
    ok = gpu_run(w, inp, adv32, want_bwd=False, cluster_mode=cluster_mode)
    f = O.forward(inp["H_pol"], inp["H_ref"], inp["W"], inp["ids"], inp["mask"], adv32.double(),
                  w.B, w.T, w.beta)
    m = inp["mask"].numpy() > 0
    assert rel_err(ok["logp_pol"].numpy()[m], f["logp_pol"][m]) < TOL_REL
    assert abs(ok["loss"] - f["loss"]) <= TOL_REL * abs(f["loss"])
    torch.cuda.synchronize()
