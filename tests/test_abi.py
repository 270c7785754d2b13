"""The C-ABI library: it loads, exports every function include/grpo.h
declares, and rejects malformed problems on the host before touching the
GPU. No kernel is launched here."""
import ctypes
import os
import re

import pytest

from grpo_loss_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(grpo_[a-z_0-9]+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.LIB_PATH):
        pytest.skip("library not built (python -m grpo_loss_gb300.build)")
    return L.lib()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("grpo_advantages", "grpo_loss_fwd", "grpo_loss_bwd",
                     "grpo_workspace_size", "grpo_get_device_status", "grpo_status_string"):
        assert required in names


def test_library_exports_every_declared_function(lib):
    handle = ctypes.CDLL(L.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(handle, name), name


def test_status_strings(lib):
    for code in range(7):
        assert len(L.status_string(code)) > 1
    assert L.status_string(99) == "unknown status"


def _problem(**kw):
    base = dict(num_seqs=8, seq_len=64, d=256, V=1024, group_size=4)
    base.update(kw)
    p = L.make_problem(**base)
    return p


@pytest.mark.parametrize("field,value,expected", [
    ("N", 7, 1),                 # N != num_seqs * seq_len
    ("group_size", 3, 1),        # does not divide num_seqs
    ("group_size", 0, 1),
    ("num_seqs", 0, 1),
    ("d", 4, 1),                 # d < 8
    ("d", 260, 2),               # d % 8 != 0: rows not 16-byte aligned for TMA
    ("V", 0, 1),
    ("chunk_rows", -1, 1),
    ("compute_dW", 2, 1),
    ("dtype", 7, 1),
    ("cluster_mode", -1, 1),
    ("cluster_mode", 2, 2),      # the removed multicast tiling
])
def test_workspace_size_rejects_bad_problems_on_host(lib, field, value, expected):
    p = _problem()
    setattr(p, field, value)
    f, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.grpo_workspace_size(ctypes.byref(p), ctypes.byref(f), ctypes.byref(b)) == expected


def test_chunk_plan_rejects_bad_problems_on_host(lib):
    p = _problem(group_size=3)
    r, n, b = ctypes.c_int64(0), ctypes.c_int32(0), ctypes.c_size_t(0)
    assert lib.grpo_chunk_plan(ctypes.byref(p), ctypes.byref(r), ctypes.byref(n),
                               ctypes.byref(b)) == 1
    assert lib.grpo_chunk_plan(None, None, None, None) == 1
    p = _problem(chunk_rows=-5)
    assert lib.grpo_chunk_plan(ctypes.byref(p), None, None, None) == 1


def test_null_problem_and_pointers_rejected(lib):
    assert lib.grpo_workspace_size(None, None, None) == 1
    assert lib.grpo_advantages(None, 8, 4, 1e-4, 1, None, None) == 1
    # unbiased std needs two members per group
    buf = ctypes.c_void_p(16)
    assert lib.grpo_advantages(buf, 4, 1, 1e-4, 1, buf, None) == 1
    p = _problem()
    args = [ctypes.byref(p)] + [None] * 11 + [None, 0, None]
    assert lib.grpo_loss_fwd(*args) == 1
    args = [ctypes.byref(p)] + [None] * 8 + [1.0, None, None, None, 0, None]
    assert lib.grpo_loss_bwd(*args) == 1
    assert lib.grpo_get_device_status(None, None) == 1


def test_profile_kinds(lib):
    n = lib.grpo_profile_kind_count()
    names = [lib.grpo_profile_kind_name(k).decode() for k in range(n)]
    assert "fwd_gemm_lse" in names and "bwd_dh_gemm" in names and "bwd_dz_gemm" in names
    assert lib.grpo_profile_kind_name(n).decode() == "unknown"


def test_problem_struct_layout_matches_the_header(tmp_path):
    """The ctypes mirror of grpo_problem has the C header's field offsets and
    size (compiled with the host C compiler against include/grpo.h)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    fields = [name for name, _ in L.Problem._fields_]
    src = ["#include <stddef.h>", "#include <stdio.h>", '#include "grpo.h"', "int main(void) {",
           '  printf("size %zu\\n", sizeof(grpo_problem));']
    for f in fields:
        src.append('  printf("%s %%zu\\n", offsetof(grpo_problem, %s));' % (f, f))
    src += ["  return 0;", "}"]
    c = tmp_path / "layout.c"
    c.write_text("\n".join(src))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I" + os.path.join(ROOT, "include"), str(c), "-o", str(exe)],
                   check=True)
    out = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True,
                                                       text=True, check=True).stdout.splitlines())
    assert int(out["size"]) == ctypes.sizeof(L.Problem)
    for f in fields:
        assert int(out[f]) == getattr(L.Problem, f).offset, f


def test_e4m3_calls_reject_bad_arguments_on_host(lib):
    """The e4m3 entry points and the quantizer check their arguments before
    any CUDA call (no GPU needed)."""
    import torch
    f, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    # e4m3 rows are d bytes: d must be a multiple of 16 (8 suffices for bf16)
    p8 = L.make_problem(8, 64, 264, 1024, 4, dtype=torch.float8_e4m3fn)
    assert p8.dtype == L.GRPO_E4M3
    assert lib.grpo_workspace_size(ctypes.byref(p8), ctypes.byref(f), ctypes.byref(b)) == 2
    fake = ctypes.c_void_p(256)                      # aligned, never dereferenced
    # a bf16 problem through the e4m3 forward, an e4m3 problem through the bf16 calls
    pb = _problem()
    args = [ctypes.byref(pb)] + [fake] * 14 + [fake, 1 << 20, None]
    assert lib.grpo_loss_fwd_e4m3(*args) == 1
    p8ok = L.make_problem(8, 64, 256, 1024, 4, dtype=torch.float8_e4m3fn)
    args = [ctypes.byref(p8ok)] + [fake] * 11 + [fake, 1 << 20, None]
    assert lib.grpo_loss_fwd(*args) == 1
    args = [ctypes.byref(p8ok)] + [fake] * 8 + [1.0, fake, None, fake, 1 << 20, None]
    assert lib.grpo_loss_bwd(*args) == 1
    # missing scales
    args = [ctypes.byref(p8ok), fake, None, fake, fake, fake, fake] + [fake] * 8 + [fake, 1 << 20,
                                                                               None]
    assert lib.grpo_loss_fwd_e4m3(*args) == 1
    args = [ctypes.byref(p8ok), fake, fake, fake, None] + [fake] * 6 + [1.0, fake, None, fake,
                                                                     1 << 20, None]
    assert lib.grpo_loss_bwd_e4m3(*args) == 1
    # s_W must be 16-byte aligned (it is read with 16-byte loads)
    odd = ctypes.c_void_p(260)
    args = [ctypes.byref(p8ok), fake, fake, fake, fake, fake, odd] + [fake] * 8 + [fake, 1 << 20,
                                                                              None]
    assert lib.grpo_loss_fwd_e4m3(*args) == 2
    # the quantizer
    q = lib.grpo_quantize_e4m3_rows
    assert q(None, L.GRPO_BF16, 4, 32, fake, fake, None) == 1
    assert q(fake, L.GRPO_E4M3, 4, 32, fake, fake, None) == 1
    assert q(fake, L.GRPO_BF16, -1, 32, fake, fake, None) == 1
    assert q(fake, L.GRPO_BF16, 4, 0, fake, fake, None) == 1
    assert q(fake, L.GRPO_BF16, 4, 24, fake, fake, None) == 2
    assert q(odd, L.GRPO_F32, 4, 32, fake, fake, None) == 2


def test_plain_c_host_links_and_calls_the_library(tmp_path):
    """A C program with no Python and no CUDA runtime calls links
    libgrpo_gb300.so through include/grpo.h alone and gets host-side statuses
    back (no GPU needed: every call below is rejected before any launch)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    if not os.path.exists(L.LIB_PATH):
        pytest.skip("library not built (python -m grpo_loss_gb300.build)")
    src = r'''
#include <stdio.h>
#include "grpo.h"
int main(void) {
  grpo_problem p = {0};
  p.num_seqs = 8; p.seq_len = 64; p.N = 8 * 64; p.d = 256; p.V = 1024; p.group_size = 3;
  p.beta = 0.04f; p.eps = 1e-4f; p.std_unbiased = 1; p.dtype = GRPO_BF16;
  size_t f = 0, b = 0;
  printf("%d\n", (int)grpo_workspace_size(&p, &f, &b));          /* group does not divide */
  p.group_size = 4; p.dtype = GRPO_E4M3; p.d = 264;
  printf("%d\n", (int)grpo_workspace_size(&p, &f, &b));          /* e4m3 needs d % 16 */
  printf("%d\n", (int)grpo_advantages(NULL, 8, 4, 1e-4f, 1, NULL, NULL));
  printf("%d\n", (int)grpo_quantize_e4m3_rows(NULL, GRPO_BF16, 4, 32, NULL, NULL, NULL));
  printf("%s\n", grpo_status_string(GRPO_ERR_UNSUPPORTED));
  return 0;
}
'''
    c = tmp_path / "host.c"
    c.write_text(src)
    exe = tmp_path / "host"
    libdir = os.path.dirname(L.LIB_PATH)
    subprocess.run([cc, "-std=c11", "-Wall", "-I" + os.path.join(ROOT, "include"), str(c),
                    "-L" + libdir, "-l:libgrpo_gb300.so", "-Wl,-rpath," + libdir, "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    assert out[:4] == ["1", "2", "1", "1"]
    assert out[4] == "unsupported problem layout"
