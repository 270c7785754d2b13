"""The workspace-free forward entry point, grpo_loss_fwd_noalloc.

It exists for callers that cannot allocate device memory: hosts without an
allocator of their own (for them cudaMalloc synchronises the device) and
code that must stay within a memory budget fixed before training starts.
Those callers cannot pass a workspace, so the library keeps this entry
point's scratch in a static device array.

The test calls it through the C ABI and checks it against the regular
grpo_loss_fwd (which takes a caller-owned workspace). It makes two calls in
a row on different problem shapes, so the second reuses the scratch the
first left behind. It also checks that an oversized problem is rejected
before any launch, and that a device-detected error marks the loss NaN.
This file is named so that it is collected after every other test file.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from grpo_loss_gb300 import _lib as L
from grpo_loss_gb300 import workloads as WL

pytestmark = pytest.mark.gpu

TOL_REL = 1e-3


def _noalloc_fn():
    fn = L.lib().grpo_loss_fwd_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(L.Problem)] + [ctypes.c_void_p] * 11 + [ctypes.c_void_p]
    return fn


def _device_inputs(w):
    inp = WL.make_inputs(w)
    dev = torch.device("cuda")
    d = {k: v.to(dev) for k, v in inp.items() if v is not None}
    g = torch.Generator().manual_seed(w.seed)
    d["adv"] = torch.randn(w.B, generator=g).to(dev)
    return d


def _outputs(w):
    dev = torch.device("cuda")
    return {"logp_pol": torch.empty(w.N, device=dev), "logp_ref": torch.empty(w.N, device=dev),
            "lse_pol": torch.empty(w.N, device=dev), "loss": torch.empty(1, device=dev),
            "kl_mean": torch.empty(1, device=dev)}


def _problem(w):
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    return L.make_problem(w.B, w.T, w.d, w.V, w.G, beta=w.beta, eps=w.eps,
                          std_unbiased=w.std_unbiased, dtype=dt)


def _call_noalloc(fn, p, x, o):
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return fn(ctypes.byref(p), ptr(x["H_pol"]), ptr(x["H_ref"]), ptr(x["W"]), ptr(x["ids"]),
              ptr(x["mask"]), ptr(x["adv"]), ptr(o["logp_pol"]), ptr(o["logp_ref"]),
              ptr(o["lse_pol"]), ptr(o["loss"]), ptr(o["kl_mean"]),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _call_regular(p, x, o):
    fwd_bytes, _ = L.workspace_size(p)
    ws = torch.empty(fwd_bytes, dtype=torch.uint8, device="cuda")
    L.loss_fwd(p, x["H_pol"], x["H_ref"], x["W"], x["ids"], x["mask"], x["adv"],
               o["logp_pol"], o["logp_ref"], o["lse_pol"], o["loss"], o["kl_mean"], ws)
    torch.cuda.synchronize()
    assert L.device_status(ws) == 0
    return o


def _assert_close(w, x, got, ref):
    m = x["mask"].bool()
    for k in ("logp_pol", "logp_ref", "lse_pol"):
        a, b = got[k][m].double(), ref[k][m].double()
        assert torch.all((a - b).abs() <= TOL_REL * b.abs()), k
        assert torch.all(got[k][~m] == ref[k][~m]) if k != "lse_pol" else True
    for k in ("loss", "kl_mean"):
        a, b = got[k].item(), ref[k].item()
        assert abs(a - b) <= TOL_REL * abs(b), (k, a, b)


def test_noalloc_matches_regular_forward_on_two_calls_in_a_row():
    fn = _noalloc_fn()
    wa = WL.SMALL["qwen2.5-small"]
    wb = WL.SMALL["llama3.1-small"]
    xa, xb = _device_inputs(wa), _device_inputs(wb)
    pa, pb = _problem(wa), _problem(wb)
    oa, ob = _outputs(wa), _outputs(wb)
    assert _call_noalloc(fn, pa, xa, oa) == 0
    assert _call_noalloc(fn, pb, xb, ob) == 0          # reuses the same scratch
    torch.cuda.synchronize()
    ra = _call_regular(pa, xa, _outputs(wa))
    rb = _call_regular(pb, xb, _outputs(wb))
    _assert_close(wa, xa, oa, ra)
    _assert_close(wb, xb, ob, rb)
    # and once more on the first shape, after the second left its contents
    oa2 = _outputs(wa)
    assert _call_noalloc(fn, pa, xa, oa2) == 0
    torch.cuda.synchronize()
    _assert_close(wa, xa, oa2, ra)


def test_noalloc_rejects_problems_beyond_its_scratch():
    fn = _noalloc_fn()
    # 64 sequences of 32K tokens on the Llama-8B head: far beyond 32 MiB of scratch
    p = L.make_problem(64, 32768, 4096, 128256, 8)
    fwd_bytes, _ = L.workspace_size(p)
    assert fwd_bytes > (32 << 20)
    z = torch.zeros(1, device="cuda")
    args = [ctypes.byref(p)] + [ctypes.c_void_p(z.data_ptr())] * 11 + [None]
    assert fn(*args) == 3                                 # GRPO_ERR_WORKSPACE, nothing launched


def test_noalloc_marks_device_errors_in_the_loss():
    fn = _noalloc_fn()
    w = WL.SMALL["llama3.1-small"]
    x = _device_inputs(w)
    x["ids"] = x["ids"].clone()
    x["ids"][3] = w.V                                     # valid row, id out of range
    o = _outputs(w)
    assert _call_noalloc(fn, _problem(w), x, o) == 0
    torch.cuda.synchronize()
    assert math.isnan(o["loss"].item())
    # the next clean call clears the error word again
    x2 = _device_inputs(w)
    o2 = _outputs(w)
    assert _call_noalloc(fn, _problem(w), x2, o2) == 0
    torch.cuda.synchronize()
    assert np.isfinite(o2["loss"].item())
