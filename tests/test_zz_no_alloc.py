"""The workspace-free forward entry point, grpo_loss_fwd_noalloc.

It exists for callers that cannot allocate device memory: hosts without an
allocator of their own (for them cudaMalloc synchronises the device) and
code that must stay within a memory budget fixed before training starts.
Those callers cannot pass a workspace, so the library keeps this entry
point's scratch in a static device array.

The tests call it through the C ABI and check it against the regular
grpo_loss_fwd (which takes a caller-owned workspace). Both run the same
kernels on the same plan, so every output must be bit-identical: on two
calls in a row with different shapes (the second reuses what the first left
in the array), on float32 inputs (whose bf16 copies live in the array), and
at the largest problem that fits the array. One token more is rejected
before any launch, and a device-detected error makes the loss and the KL
mean NaN. This file is named so that it is collected after every other
test file.
"""
import ctypes
import math

import pytest
import torch

from grpo_loss_gb300 import _lib as L
from grpo_loss_gb300 import workloads as WL

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20            # GRPO_NOALLOC_SCRATCH_BYTES in include/grpo.h
GRPO_ERR_WORKSPACE = 3


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


def _outputs(N):
    dev = torch.device("cuda")
    return {"logp_pol": torch.empty(N, device=dev), "logp_ref": torch.empty(N, device=dev),
            "lse_pol": torch.empty(N, device=dev), "loss": torch.empty(1, device=dev),
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


def _assert_identical(x, got, ref):
    """Bit-identical outputs; lse_pol is specified at valid rows only."""
    m = x["mask"].bool()
    for k in ("logp_pol", "logp_ref", "loss", "kl_mean"):
        assert torch.equal(got[k], ref[k]), k
    assert torch.equal(got["lse_pol"][m], ref["lse_pol"][m])
    assert math.isfinite(got["loss"].item()) and math.isfinite(got["kl_mean"].item())


def test_noalloc_matches_regular_forward_on_two_calls_in_a_row():
    fn = _noalloc_fn()
    wa = WL.SMALL["qwen2.5-small"]
    wb = WL.SMALL["llama3.1-small"]
    xa, xb = _device_inputs(wa), _device_inputs(wb)
    pa, pb = _problem(wa), _problem(wb)
    oa, ob = _outputs(wa.N), _outputs(wb.N)
    assert _call_noalloc(fn, pa, xa, oa) == 0
    assert _call_noalloc(fn, pb, xb, ob) == 0          # reuses the same scratch
    torch.cuda.synchronize()
    ra = _call_regular(pa, xa, _outputs(wa.N))
    rb = _call_regular(pb, xb, _outputs(wb.N))
    _assert_identical(xa, oa, ra)
    _assert_identical(xb, ob, rb)
    # and once more on the first shape, after the second left its contents
    oa2 = _outputs(wa.N)
    assert _call_noalloc(fn, pa, xa, oa2) == 0
    torch.cuda.synchronize()
    _assert_identical(xa, oa2, ra)


def test_noalloc_float32_inputs_keep_their_bf16_copies_in_the_array():
    fn = _noalloc_fn()
    w = WL.TINY
    x = _device_inputs(w)
    p = _problem(w)
    fwd_bytes, _ = L.workspace_size(p)
    assert fwd_bytes > 2 * (2 * w.N * w.d + w.V * w.d)   # the bf16 copies are in the need
    o1, o2 = _outputs(w.N), _outputs(w.N)
    assert _call_noalloc(fn, p, x, o1) == 0
    assert _call_noalloc(fn, p, x, o2) == 0
    torch.cuda.synchronize()
    ref = _call_regular(p, x, _outputs(w.N))
    _assert_identical(x, o1, ref)
    _assert_identical(x, o2, ref)


def _boundary_problem(T):
    return L.make_problem(8, T, 128, 1000, 4)


def test_noalloc_runs_the_largest_problem_that_fits_and_rejects_one_more():
    """The need comes from grpo_workspace_size on this device: the longest
    sequences whose need fits the array run (bit-identical to the regular
    forward); the next length is rejected before any launch."""
    fn = _noalloc_fn()
    need = lambda T: L.workspace_size(_boundary_problem(T))[0]  # noqa: E731
    lo, hi = 1, 1 << 20
    assert need(lo) <= SCRATCH_BYTES < need(hi)
    while hi - lo > 1:                                  # need grows with T
        mid = (lo + hi) // 2
        if need(mid) <= SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    T_fit, T_over = lo, hi
    assert need(T_fit) <= SCRATCH_BYTES < need(T_over)
    assert need(T_fit) > SCRATCH_BYTES - (1 << 16)      # just under: within 64 KB

    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(11)
    p = _boundary_problem(T_fit)
    N, d, V = p.N, p.d, p.V
    x = {"H_pol": torch.randn(N, d, generator=g, device=dev).bfloat16(),
         "W": (0.05 * torch.randn(V, d, generator=g, device=dev)).bfloat16(),
         "ids": torch.randint(0, V, (N,), generator=g, device=dev, dtype=torch.int32),
         "mask": (torch.rand(N, generator=g, device=dev) < 0.9).to(torch.uint8),
         "adv": torch.randn(8, generator=g, device=dev)}
    x["H_ref"] = (x["H_pol"].float() + 0.05 * torch.randn(N, d, generator=g, device=dev)).bfloat16()
    o = _outputs(N)
    assert _call_noalloc(fn, p, x, o) == 0
    torch.cuda.synchronize()
    _assert_identical(x, o, _call_regular(p, x, _outputs(N)))

    p_over = _boundary_problem(T_over)
    z = torch.zeros(1, device=dev)
    args = [ctypes.byref(p_over)] + [ctypes.c_void_p(z.data_ptr())] * 11 + [None]
    assert fn(*args) == GRPO_ERR_WORKSPACE             # nothing launched: no pointer is read


def test_noalloc_rejects_problems_far_beyond_its_scratch():
    fn = _noalloc_fn()
    # 64 sequences of 32K tokens on the Llama-8B head: far beyond 32 MiB of scratch
    p = L.make_problem(64, 32768, 4096, 128256, 8)
    fwd_bytes, _ = L.workspace_size(p)
    assert fwd_bytes > SCRATCH_BYTES
    z = torch.zeros(1, device="cuda")
    args = [ctypes.byref(p)] + [ctypes.c_void_p(z.data_ptr())] * 11 + [None]
    assert fn(*args) == GRPO_ERR_WORKSPACE


def test_noalloc_marks_device_errors_in_the_loss_and_kl_mean():
    fn = _noalloc_fn()
    w = WL.SMALL["llama3.1-small"]
    x = _device_inputs(w)
    x["ids"] = x["ids"].clone()
    x["ids"][3] = w.V                                     # valid row, id out of range
    o = _outputs(w.N)
    assert _call_noalloc(fn, _problem(w), x, o) == 0
    torch.cuda.synchronize()
    assert math.isnan(o["loss"].item()) and math.isnan(o["kl_mean"].item())
    # the next clean call clears the error word again
    x2 = _device_inputs(w)
    o2 = _outputs(w.N)
    assert _call_noalloc(fn, _problem(w), x2, o2) == 0
    torch.cuda.synchronize()
    _assert_identical(x2, o2, _call_regular(_problem(w), x2, _outputs(w.N)))
