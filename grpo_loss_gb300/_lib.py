"""ctypes binding of the C ABI declared in include/grpo.h.

Argument marshalling only: every step of the loss runs in the library's CUDA
kernels. There is no CPU fallback; if the shared library has not been built
the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

# The in-tree build; GRPO_GB300_LIB may name another build of the same library.
LIB_PATH = os.environ.get("GRPO_GB300_LIB") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "libgrpo_gb300.so")

GRPO_OK = 0
STATUS_NAMES = {0: "GRPO_OK", 1: "GRPO_ERR_INVALID_ARG", 2: "GRPO_ERR_UNSUPPORTED",
                3: "GRPO_ERR_WORKSPACE", 4: "GRPO_ERR_CUDA", 5: "GRPO_ERR_TIMEOUT",
                6: "GRPO_ERR_BAD_TOKEN"}
GRPO_F32, GRPO_BF16, GRPO_E4M3 = 0, 1, 2


class GrpoError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (%s)" % (where, STATUS_NAMES.get(status, status),
                                                  status_string(status)))


class Problem(ctypes.Structure):
    """Mirror of ``grpo_problem``."""
    _fields_ = [("N", ctypes.c_int64), ("d", ctypes.c_int64), ("V", ctypes.c_int64),
                ("num_seqs", ctypes.c_int32), ("seq_len", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("beta", ctypes.c_float),
                ("eps", ctypes.c_float), ("std_unbiased", ctypes.c_int32),
                ("chunk_rows", ctypes.c_int64), ("compute_dW", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("token_level", ctypes.c_int32),
                ("logit_multiply", ctypes.c_float), ("logit_divide", ctypes.c_float),
                ("softcap", ctypes.c_float), ("temperature", ctypes.c_float),
                ("ref_logp_given", ctypes.c_int32), ("kl_mode", ctypes.c_int32),
                ("cluster_mode", ctypes.c_int32)]


def make_problem(num_seqs: int, seq_len: int, d: int, V: int, group_size: int,
                 beta: float = 0.04, eps: float = 1e-4, std_unbiased: int = 1,
                 chunk_rows: int = 0, dtype=torch.bfloat16, compute_dW: int = 0,
                 token_level: bool = False, logit_multiply: float = 0.0,
                 logit_divide: float = 0.0, softcap: float = 0.0, temperature: float = 0.0,
                 ref_logp_given: bool = False, kl_mode: int = 0,
                 cluster_mode: int = 0) -> Problem:
    return Problem(N=num_seqs * seq_len, d=d, V=V, num_seqs=num_seqs, seq_len=seq_len,
                   group_size=group_size, beta=beta, eps=eps, std_unbiased=std_unbiased,
                   chunk_rows=chunk_rows, compute_dW=1 if compute_dW else 0,
                   dtype=dtype_code(dtype),
                   token_level=1 if token_level else 0, logit_multiply=logit_multiply,
                   logit_divide=logit_divide, softcap=softcap, temperature=temperature,
                   ref_logp_given=1 if ref_logp_given else 0, kl_mode=kl_mode,
                   cluster_mode=cluster_mode)


def dtype_code(dtype) -> int:
    """grpo_dtype of a torch dtype: float32, bfloat16, or float8_e4m3fn for an
    e4m3 problem (operands as codes with row scales)."""
    if dtype == torch.float32:
        return GRPO_F32
    if dtype == torch.float8_e4m3fn:
        return GRPO_E4M3
    if dtype == torch.bfloat16:
        return GRPO_BF16
    raise ValueError("unsupported dtype %s" % (dtype,))


_lib = None
_lock = threading.Lock()

_VP = ctypes.c_void_p
_SIGNATURES = {
    "grpo_workspace_size": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.POINTER(ctypes.c_size_t),
                                           ctypes.POINTER(ctypes.c_size_t)]),
    "grpo_chunk_plan": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.POINTER(ctypes.c_int64),
                                       ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_size_t)]),
    "grpo_advantages": (ctypes.c_int, [_VP, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                       ctypes.c_int32, _VP, _VP]),
    "grpo_loss_fwd": (ctypes.c_int, [ctypes.POINTER(Problem)] + [_VP] * 11 +
                      [_VP, ctypes.c_size_t, _VP]),
    "grpo_loss_bwd": (ctypes.c_int, [ctypes.POINTER(Problem)] + [_VP] * 8 +
                      [ctypes.c_float, _VP, _VP, _VP, ctypes.c_size_t, _VP]),
    "grpo_loss_fwd_e4m3": (ctypes.c_int, [ctypes.POINTER(Problem)] + [_VP] * 14 +
                           [_VP, ctypes.c_size_t, _VP]),
    "grpo_loss_bwd_e4m3": (ctypes.c_int, [ctypes.POINTER(Problem)] + [_VP] * 10 +
                           [ctypes.c_float, _VP, _VP, _VP, ctypes.c_size_t, _VP]),
    "grpo_quantize_e4m3_rows": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                               _VP, _VP, _VP]),
    "grpo_get_device_status": (ctypes.c_int, [_VP, _VP]),
    "grpo_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "grpo_profile_enable": (ctypes.c_int, [ctypes.c_int32]),
    "grpo_profile_collect": (ctypes.c_int, [ctypes.POINTER(ctypes.c_double),
                                            ctypes.POINTER(ctypes.c_int64), ctypes.c_int32]),
    "grpo_profile_kind_count": (ctypes.c_int32, []),
    "grpo_test_pipeline_stall": (ctypes.c_int, [ctypes.c_int32, ctypes.c_uint32]),
    "grpo_profile_kind_name": (ctypes.c_char_p, [ctypes.c_int32]),
}


def lib() -> ctypes.CDLL:
    """Load the in-tree shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        "libgrpo_gb300.so is missing: build it with "
                        "`python -m grpo_loss_gb300.build` (needs nvcc); there is no CPU fallback")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in _SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().grpo_status_string(status).decode()


def _check(status: int, where: str) -> None:
    if status != GRPO_OK:
        raise GrpoError(status, where)


def _ptr(t: Optional[torch.Tensor], name: str, dtype=None, numel: Optional[int] = None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if numel is not None and t.numel() != numel:
        raise ValueError("%s must have %d elements, got %d" % (name, numel, t.numel()))
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def workspace_size(problem: Problem):
    f, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib().grpo_workspace_size(ctypes.byref(problem), ctypes.byref(f), ctypes.byref(b)),
           "grpo_workspace_size")
    return f.value, b.value


def chunk_plan(problem: Problem):
    """(chunk_rows, n_chunks, dz_chunk_bytes) of the backward's chunk plan."""
    r, n, b = ctypes.c_int64(0), ctypes.c_int32(0), ctypes.c_size_t(0)
    _check(lib().grpo_chunk_plan(ctypes.byref(problem), ctypes.byref(r), ctypes.byref(n),
                                 ctypes.byref(b)), "grpo_chunk_plan")
    return r.value, n.value, b.value


def advantages(rewards: torch.Tensor, group_size: int, eps: float, std_unbiased: int,
               adv: torch.Tensor, stream=None) -> torch.Tensor:
    B = rewards.numel()
    _check(lib().grpo_advantages(_ptr(rewards, "rewards", torch.float32), B, group_size, eps,
                                 std_unbiased, _ptr(adv, "adv", torch.float32, B), _stream(stream)),
           "grpo_advantages")
    return adv


def loss_fwd(problem: Problem, H_pol, H_ref, W, ids, mask, adv, logp_pol, logp_ref, lse_pol,
             loss, kl_mean, workspace: torch.Tensor, stream=None) -> None:
    N = problem.N
    _check(lib().grpo_loss_fwd(
        ctypes.byref(problem), _ptr(H_pol, "H_pol"),
        None if H_ref is None else _ptr(H_ref, "H_ref"), _ptr(W, "W"),
        _ptr(ids, "ids", torch.int32, N), _ptr(mask, "mask", torch.uint8, N),
        _ptr(adv, "adv", torch.float32, problem.num_seqs),
        _ptr(logp_pol, "logp_pol", torch.float32, N), _ptr(logp_ref, "logp_ref", torch.float32, N),
        _ptr(lse_pol, "lse_pol", torch.float32, N), _ptr(loss, "loss", torch.float32, 1),
        _ptr(kl_mean, "kl_mean", torch.float32, 1), _ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)), "grpo_loss_fwd")


def loss_bwd(problem: Problem, H_pol, W, ids, mask, adv, logp_pol, logp_ref, lse_pol,
             grad_loss: float, dH, workspace: torch.Tensor, stream=None, dW=None) -> None:
    N = problem.N
    _check(lib().grpo_loss_bwd(
        ctypes.byref(problem), _ptr(H_pol, "H_pol"), _ptr(W, "W"),
        _ptr(ids, "ids", torch.int32, N), _ptr(mask, "mask", torch.uint8, N),
        _ptr(adv, "adv", torch.float32, problem.num_seqs),
        _ptr(logp_pol, "logp_pol", torch.float32, N), _ptr(logp_ref, "logp_ref", torch.float32, N),
        _ptr(lse_pol, "lse_pol", torch.float32, N), float(grad_loss), _ptr(dH, "dH"),
        _ptr(dW, "dW", torch.float32, problem.V * problem.d),
        _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)), "grpo_loss_bwd")


def _codes(t, name: str, numel: int):
    """Pointer to e4m3 codes held as uint8 or float8_e4m3fn."""
    if t is None:
        return None
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise ValueError("%s must hold e4m3 codes (uint8 or float8_e4m3fn), got %s" % (name, t.dtype))
    return _ptr(t, name, None, numel)


def quantize_e4m3_rows(x: torch.Tensor, q=None, scale=None, stream=None):
    """Row-wise e4m3 codes (uint8 [rows, cols]) and scales (float32 [rows]) of
    a float32 or bf16 CUDA matrix; see grpo_quantize_e4m3_rows."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D")
    rows, cols = x.shape
    if x.dtype == torch.float32:
        code = GRPO_F32
    elif x.dtype == torch.bfloat16:
        code = GRPO_BF16
    else:
        raise ValueError("x must be float32 or bfloat16")
    if q is None:
        q = torch.empty(rows, cols, dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check(lib().grpo_quantize_e4m3_rows(_ptr(x, "x"), code, rows, cols,
                                         _codes(q, "q", rows * cols),
                                         _ptr(scale, "scale", torch.float32, rows),
                                         _stream(stream)), "grpo_quantize_e4m3_rows")
    return q, scale


def loss_fwd_e4m3(problem: Problem, H_pol, s_pol, H_ref, s_ref, W, s_W, ids, mask, adv,
                  logp_pol, logp_ref, lse_pol, loss, kl_mean, workspace: torch.Tensor,
                  stream=None) -> None:
    N, Nd, Vd = problem.N, problem.N * problem.d, problem.V * problem.d
    _check(lib().grpo_loss_fwd_e4m3(
        ctypes.byref(problem), _codes(H_pol, "H_pol", Nd), _ptr(s_pol, "s_pol", torch.float32, N),
        _codes(H_ref, "H_ref", Nd), _ptr(s_ref, "s_ref", torch.float32, N),
        _codes(W, "W", Vd), _ptr(s_W, "s_W", torch.float32, problem.V),
        _ptr(ids, "ids", torch.int32, N), _ptr(mask, "mask", torch.uint8, N),
        _ptr(adv, "adv", torch.float32, problem.num_seqs),
        _ptr(logp_pol, "logp_pol", torch.float32, N), _ptr(logp_ref, "logp_ref", torch.float32, N),
        _ptr(lse_pol, "lse_pol", torch.float32, N), _ptr(loss, "loss", torch.float32, 1),
        _ptr(kl_mean, "kl_mean", torch.float32, 1), _ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)), "grpo_loss_fwd_e4m3")


def loss_bwd_e4m3(problem: Problem, H_pol, s_pol, W, s_W, ids, mask, adv, logp_pol, logp_ref,
                  lse_pol, grad_loss: float, dH, workspace: torch.Tensor, stream=None,
                  dW=None) -> None:
    N, Nd, Vd = problem.N, problem.N * problem.d, problem.V * problem.d
    _check(lib().grpo_loss_bwd_e4m3(
        ctypes.byref(problem), _codes(H_pol, "H_pol", Nd), _ptr(s_pol, "s_pol", torch.float32, N),
        _codes(W, "W", Vd), _ptr(s_W, "s_W", torch.float32, problem.V),
        _ptr(ids, "ids", torch.int32, N), _ptr(mask, "mask", torch.uint8, N),
        _ptr(adv, "adv", torch.float32, problem.num_seqs),
        _ptr(logp_pol, "logp_pol", torch.float32, N), _ptr(logp_ref, "logp_ref", torch.float32, N),
        _ptr(lse_pol, "lse_pol", torch.float32, N), float(grad_loss),
        _ptr(dH, "dH", torch.bfloat16, Nd),
        _ptr(dW, "dW", torch.float32, Vd),
        _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)), "grpo_loss_bwd_e4m3")


def device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise and return (and clear) the workspace's device error status."""
    return lib().grpo_get_device_status(_ptr(workspace, "workspace"), _stream(stream))


def profile_enable(on: bool) -> None:
    _check(lib().grpo_profile_enable(1 if on else 0), "grpo_profile_enable")


def profile_collect():
    """{kernel name: (milliseconds, launches)} since the last collect."""
    n = lib().grpo_profile_kind_count()
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    _check(lib().grpo_profile_collect(ms, cnt, n), "grpo_profile_collect")
    return {lib().grpo_profile_kind_name(k).decode(): (ms[k], cnt[k]) for k in range(n)}
