"""The backward's chunk scheduler against the pages' memory model.

The Unsloth long-context page (flattened sequence chunking, Equations 1-3)
counts the logits of one chunk as rows x vocab / multiplier elements; the
Unsloth GRPO blog's figures for the Llama 3.1 8B head at 20K context with
8 generations are 78.3 GB of float32 logits for the batch and 9.8 GB for one
generation (tests/golden/memory_figures.txt). The oracle's logit_memory_gib
restates that model and is pinned to those figures in test_oracle.py. Here
the library's chunk plan (grpo_chunk_plan, which needs the device's SM
count) is checked against it: the dZ chunk it sizes is that model's bf16
chunk, it stays within the default budget, it fills whole waves of dH tiles,
and one generation's chunk is half the pages' float32 figure."""
import math
import os

import pytest
import torch

from grpo_loss_gb300 import _lib as L
from grpo_loss_gb300 import workloads as WL
from oracle import grpo_oracle as O

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
BUDGET = 4 << 30                    # GRPO_DEFAULT_DZ_BUDGET_BYTES


def _figures():
    out = {}
    with open(os.path.join(GOLDEN, "memory_figures.txt")) as fh:
        for line in fh:
            if line.strip() and not line.startswith("#"):
                f = [x.strip() for x in line.split("|")]
                out[f[0]] = float(f[5])
    return out


def _problem(w, chunk_rows=0):
    return L.make_problem(w.B, w.T, w.d, w.V, w.G, chunk_rows=chunk_rows)


def _dh_tiles(d):
    # dH column tiles: the widest multiple of 64 up to 256 that divides d
    for bn in range(256, 63, -64):
        if d % bn == 0:
            return d // bn
    return math.ceil(d / 256)


@pytest.mark.parametrize("w", [WL.QWEN25_1P5B, WL.LLAMA31_8B_20K, WL.QWEN3_8B_110K,
                               WL.GPTOSS_20B], ids=lambda w: w.name)
def test_default_chunk_fits_the_budget_in_whole_waves(w):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows, n_chunks, dz = L.chunk_plan(_problem(w))
    ldv = (w.V + 7) // 8 * 8
    blocks = math.ceil(w.N / 128)
    assert rows % 128 == 0 and n_chunks == math.ceil(blocks / (rows // 128))
    # the dZ chunk is the pages' chunk of logits at two bytes each (ldv columns)
    assert dz == round(O.logit_memory_gib(rows, ldv, 1, 2) * 1024 ** 3)
    assert dz <= BUDGET
    m0 = sms // math.gcd(sms, _dh_tiles(w.d))
    max_fit = BUDGET // (128 * ldv * 2)              # blocks whose dZ fits the budget
    if rows // 128 < blocks:
        if max_fit >= m0:
            # the largest multiple of m0 blocks that fits: whole waves of dH
            # tiles on the device's SMs
            assert (rows // 128) % m0 == 0
            assert O.logit_memory_gib(rows + 128 * m0, ldv, 1, 2) * 1024 ** 3 > BUDGET
            assert (rows // 128) * _dh_tiles(w.d) % sms == 0
        else:
            # fewer than m0 blocks fit (gpt-oss: 15 dH tiles, m0 = 152): the
            # count from 3/4 of max_fit up whose dH tiles fill their last wave
            # best, ties to the larger
            def eff(b):
                waves = b * _dh_tiles(w.d) / sms
                return waves / math.ceil(waves)
            cands = [b for b in range(max_fit, 0, -1) if 4 * b >= 3 * max_fit]
            best = max(cands, key=lambda b: (round(eff(b), 9), b))
            assert rows // 128 == best
            assert eff(best) >= eff(max_fit)


def test_explicit_chunk_rows_give_the_pages_chunk_size():
    w = WL.LLAMA31_8B_20K
    figs = _figures()
    # the pages' memory model: 8 generations of 20480 tokens, float32 logits
    assert abs(O.logit_memory_gib(w.N, w.V, 1, 4) - figs["llama_logits_total"]) < 0.05
    # one generation per chunk (multiplier 8): 20480 rows, whose float32
    # logits are the pages' 9.8 GB; the library's bf16 dZ chunk is half that
    rows, n_chunks, dz = L.chunk_plan(_problem(w, chunk_rows=w.T))
    assert rows == w.T and n_chunks == w.G
    assert dz * 2 == round(O.logit_memory_gib(w.T, w.V, 1, 4) * 1024 ** 3)
    assert abs(2 * dz / 1024 ** 3 - figs["llama_logits_per_generation"]) < 0.05
    # the pages' default multiplier max(4, ctx // 4096) = 5 for 20K context
    mult = max(4, w.T // 4096)
    rows, n_chunks, dz = L.chunk_plan(_problem(w, chunk_rows=w.N // mult))
    assert rows == w.N // mult and n_chunks == mult
    assert dz == round(O.logit_memory_gib(w.N, w.V, mult, 2) * 1024 ** 3)
    # a chunk that is not a multiple of 128 rows is rounded up to one
    rows, _, _ = L.chunk_plan(_problem(w, chunk_rows=1000))
    assert rows == 1024


def test_backward_workspace_holds_the_chunk():
    w = WL.LLAMA31_8B_20K
    _, bwd = L.workspace_size(_problem(w))
    _, _, dz = L.chunk_plan(_problem(w))
    assert dz < bwd < dz + 2 * w.d * ((w.V + 7) // 8 * 8) + (64 << 20)
