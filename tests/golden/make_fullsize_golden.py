"""Write the float64 oracle's full forward pass over the four large workloads
to tests/golden/fullsize_<workload>.json.

Every token's logits are formed in float64 (the oracle's token_logprobs, in
256-row blocks), so this takes about an hour of host time for all four; it
is run once, and the GPU tests compare against the stored values. The file
also records input_digest of the inputs it used: the generator gives the
same bytes on every host, and a test that finds another digest reports that
the inputs differ instead of a parity failure.

Only the oracle and the seeded input generator are used here.

    python tests/golden/make_fullsize_golden.py [workload ...]
"""
from __future__ import annotations

import json
import os
import platform
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from grpo_loss_gb300 import workloads as WL  # noqa: E402
from oracle import grpo_oracle as O  # noqa: E402

LARGE = [WL.QWEN25_1P5B, WL.LLAMA31_8B_20K, WL.QWEN3_8B_110K, WL.GPTOSS_20B]


def golden_path(name: str) -> str:
    return os.path.join(HERE, "fullsize_%s.json" % name)


def compute(w: WL.Workload) -> dict:
    t0 = time.time()
    inp = WL.make_inputs(w)
    digest = WL.input_digest(inp)
    if w.supplied_adv:
        adv = inp["adv"].numpy().astype(np.float64)
    else:
        # the GPU tests pass the oracle's advantages rounded to float32 to both sides
        adv = O.advantages(inp["rewards"], w.G, w.eps, w.std_unbiased).astype(np.float32)
        adv = adv.astype(np.float64)
    out = O.forward(inp["H_pol"], inp["H_ref"], inp["W"], inp["ids"], inp["mask"], adv,
                    w.B, w.T, w.beta)
    m = inp["mask"].numpy() > 0
    x = out["logp_ref"] - out["logp_pol"]
    return {
        "workload": w.name,
        "input_digest": digest,
        "n_valid": int(m.sum()),
        "loss": out["loss"],
        "kl_mean": out["kl_mean"],
        "sum_logp_pol": float(out["logp_pol"][m].sum()),
        "sum_logp_ref": float(out["logp_ref"][m].sum()),
        "sum_x_sq": float(np.sum(x[m] ** 2)),
        "adv_float32": [float(a) for a in adv],
        "host_seconds": round(time.time() - t0, 1),
        "host": platform.machine(),
    }


def main(names) -> None:
    todo = [w for w in LARGE if not names or w.name in names]
    for w in todo:
        print("oracle forward on %s (N = %d, d = %d, V = %d) ..." % (w.name, w.N, w.d, w.V),
              flush=True)
        rec = compute(w)
        with open(golden_path(w.name), "w") as fh:
            json.dump(rec, fh, indent=1)
            fh.write("\n")
        print("  loss %.17g  kl_mean %.17g  (%s s)" % (rec["loss"], rec["kl_mean"],
                                                    rec["host_seconds"]), flush=True)


if __name__ == "__main__":
    main(sys.argv[1:])
