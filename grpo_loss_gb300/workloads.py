"""Seeded synthetic inputs for the GRPO loss path.

This module only draws random numbers. It holds none of the loss arithmetic,
so both the float64 oracle and the CUDA path can be fed from it without
sharing any of the method's code.

The five named workloads stand in for the models and settings that the
Unsloth long-context GRPO pages discuss (Llama 3.1 8B at 20K context with 8
generations, Qwen3-8B at 110K, gpt-oss-20b, a Qwen2.5-1.5B head, and a tiny
correctness case). No model weights or datasets are used: hidden states and
the lm_head weight are Gaussian, token ids are uniform or Zipf-distributed,
and rewards are drawn per generation.

Every generator runs on the host with ``torch.Generator('cpu')`` seeded from
the workload, so a given workload always yields the same tensors.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and value recipe of one synthetic GRPO loss problem.

    Rows are laid out sequence-major: row ``n = b * T + t`` for sequence
    ``b`` (``B = prompts * G`` sequences, the ``G`` generations of a prompt
    contiguous) and completion position ``t``.
    """

    name: str
    prompts: int
    G: int
    T: int
    d: int
    V: int
    dtype: str = "bf16"          # "f32" or "bf16": dtype of H and W
    ref: str = "noise"           # "noise": H_ref = H_pol + 0.05 N(0,1); "independent"
    mask: str = "full"           # "full", "tiny", "pad_uniform", "tail_frac"
    pad_lo: int = 0              # pad_uniform: valid length ~ U{pad_lo..pad_hi}
    pad_hi: int = 0
    tail_frac: float = 0.0       # tail_frac: the last round(frac*T) tokens are padding
    rewards: str = "normal"      # "normal", "choice", "adv_normal" (advantages supplied)
    reward_values: Tuple[float, ...] = ()
    ids: str = "uniform"         # "uniform" or "zipf"
    zipf_s: float = 1.1
    w_std: float = 0.02
    beta: float = 0.04
    eps: float = 1e-4
    std_unbiased: int = 1
    seed: int = 1000

    @property
    def B(self) -> int:
        return self.prompts * self.G

    @property
    def N(self) -> int:
        return self.B * self.T

    @property
    def supplied_adv(self) -> bool:
        return self.rewards == "adv_normal"

    def scaled(self, name: str, **kw) -> "Workload":
        """A smaller copy with the same value recipe (for oracle-sized parity)."""
        return dataclasses.replace(self, name=name, **kw)


TINY = Workload("tiny", prompts=2, G=4, T=64, d=256, V=1024, dtype="f32",
                ref="independent", mask="tiny", rewards="normal", w_std=0.02,
                seed=1000)
QWEN25_1P5B = Workload("qwen2.5-1.5b-head", prompts=4, G=8, T=512, d=1536,
                       V=151936, mask="pad_uniform", pad_lo=256, pad_hi=512,
                       rewards="choice", reward_values=(0.0, 1.0, 2.0, 3.0),
                       seed=1001)
LLAMA31_8B_20K = Workload("llama3.1-8b-head-20kx8", prompts=1, G=8, T=20480,
                          d=4096, V=128256, mask="full", rewards="normal",
                          seed=1002)
QWEN3_8B_110K = Workload("qwen3-8b-head-110k", prompts=1, G=1, T=110000,
                         d=4096, V=151936, mask="tail_frac", tail_frac=0.1,
                         rewards="adv_normal", seed=1003)
GPTOSS_20B = Workload("gpt-oss-20b-head", prompts=2, G=4, T=32768, d=2880,
                      V=201088, mask="pad_uniform", pad_lo=16384, pad_hi=32768,
                      rewards="choice", reward_values=(-3.0, 0.0, 3.0),
                      ids="zipf", seed=1004)

FULL = {w.name: w for w in (TINY, QWEN25_1P5B, LLAMA31_8B_20K, QWEN3_8B_110K, GPTOSS_20B)}

# Oracle-sized copies of the four large workloads: same value recipe, mask
# structure and id distribution, sizes that still span several 128-row
# blocks, several 256-column vocab tiles and a ragged tail of each.
SMALL = {
    "qwen2.5-small": QWEN25_1P5B.scaled("qwen2.5-small", prompts=2, G=4, T=200,
                                        d=320, V=3000, pad_lo=100, pad_hi=200),
    "llama3.1-small": LLAMA31_8B_20K.scaled("llama3.1-small", prompts=1, G=8,
                                            T=160, d=512, V=2304),
    "qwen3-small": QWEN3_8B_110K.scaled("qwen3-small", T=1100, d=384, V=1560),
    "gpt-oss-small": GPTOSS_20B.scaled("gpt-oss-small", prompts=2, G=4, T=192,
                                       d=192, V=4104, pad_lo=96, pad_hi=192),
}


def _zipf_ids(gen: torch.Generator, n: int, V: int, s: float) -> torch.Tensor:
    """Ranks k = 1..V with pmf proportional to k^-s, sampled by inverse CDF
    from a float64 cumulative table; rank k maps to token id k - 1."""
    k = np.arange(1, V + 1, dtype=np.float64)
    cdf = np.cumsum(k ** (-s))
    cdf /= cdf[-1]
    u = torch.rand(n, generator=gen, dtype=torch.float64).numpy()
    ids = np.searchsorted(cdf, u, side="right")
    return torch.from_numpy(np.minimum(ids, V - 1).astype(np.int32))


def make_inputs(w: Workload) -> Dict[str, Optional[torch.Tensor]]:
    """Draw the host tensors of workload ``w``.

    Returns H_pol, H_ref ([N, d], dtype of ``w``), W ([V, d]), ids (int32
    [N]), mask (uint8 [N]) and either rewards (float32 [B]) or adv (float32
    [B], when advantages are supplied directly). Draw order is fixed.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    N, d, V, B, T = w.N, w.d, w.V, w.B, w.T

    H_pol = torch.randn(N, d, generator=gen, dtype=torch.float32).to(tdt)
    if w.ref == "independent":
        H_ref = torch.randn(N, d, generator=gen, dtype=torch.float32).to(tdt)
    else:
        noise = torch.randn(N, d, generator=gen, dtype=torch.float32)
        H_ref = (H_pol.float() + 0.05 * noise).to(tdt)
        del noise
    W = (w.w_std * torch.randn(V, d, generator=gen, dtype=torch.float32)).to(tdt)

    if w.ids == "zipf":
        ids = _zipf_ids(gen, N, V, w.zipf_s)
    else:
        ids = torch.randint(0, V, (N,), generator=gen, dtype=torch.int64).to(torch.int32)

    mask = torch.ones(B, T, dtype=torch.uint8)
    if w.mask == "tiny":
        # last 8 tokens of the generations with odd in-group index
        for b in range(B):
            if (b % w.G) % 2 == 1:
                mask[b, T - 8:] = 0
    elif w.mask == "pad_uniform":
        lengths = torch.randint(w.pad_lo, w.pad_hi + 1, (B,), generator=gen)
        pos = torch.arange(T)[None, :]
        mask = (pos < lengths[:, None]).to(torch.uint8)
    elif w.mask == "tail_frac":
        mask[:, T - int(round(w.tail_frac * T)):] = 0
    mask = mask.reshape(N).contiguous()

    rewards = adv = None
    if w.rewards == "normal":
        rewards = torch.randn(B, generator=gen, dtype=torch.float32)
    elif w.rewards == "choice":
        vals = torch.tensor(w.reward_values, dtype=torch.float32)
        rewards = vals[torch.randint(0, len(w.reward_values), (B,), generator=gen)]
    elif w.rewards == "adv_normal":
        adv = torch.randn(B, generator=gen, dtype=torch.float32)
    else:
        raise ValueError(w.rewards)

    return {"H_pol": H_pol, "H_ref": H_ref, "W": W, "ids": ids, "mask": mask,
            "rewards": rewards, "adv": adv}


def sample_rows(w: Workload, mask: torch.Tensor, count: int, seed: int = 7) -> np.ndarray:
    """A seeded, stratified sample of row indices for row-wise parity checks:
    every sequence's first and last valid row, rows on either side of 128-row
    block boundaries, and uniform random rows (valid and masked)."""
    m = mask.numpy().reshape(w.B, w.T)
    rows = set()
    for b in range(w.B):
        valid = np.nonzero(m[b])[0]
        if valid.size:
            rows.add(b * w.T + int(valid[0]))
            rows.add(b * w.T + int(valid[-1]))
            if valid[-1] + 1 < w.T:
                rows.add(b * w.T + int(valid[-1]) + 1)
    rng = np.random.default_rng(seed)
    nblk = (w.N + 127) // 128
    for blk in rng.choice(nblk, size=min(nblk, max(1, count // 8)), replace=False):
        for r in (blk * 128 - 1, blk * 128, blk * 128 + 127):
            if 0 <= r < w.N:
                rows.add(int(r))
    while len(rows) < count and len(rows) < w.N:
        rows.add(int(rng.integers(0, w.N)))
    return np.array(sorted(rows), dtype=np.int64)


def random_e4m3_operands(w: Workload, seed: int = 0) -> Dict[str, torch.Tensor]:
    """E4M3 codes and float32 row scales drawn directly (no quantization):
    codes uniform over the 254 non-NaN bytes (every sign, exponent and
    mantissa pattern, subnormals included), scales 2^U(-1, 1) times a base
    that puts the logits near unit scale. Keys q_pol, s_pol, q_ref, s_ref,
    q_W, s_W (host tensors)."""
    gen = torch.Generator().manual_seed(w.seed * 7919 + seed)
    pool = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8)
    # E[decode(code)^2] over that pool is about 1.0e4; z = s_h s_w sum_k q_h q_w
    # has a standard deviation near s_h s_w sqrt(d) 1.0e4, so s ~ (sqrt(d) 1.0e4)^-1/2
    base = float((np.sqrt(w.d) * 1.0e4) ** -0.5)

    def codes(rows):
        return pool[torch.randint(0, pool.numel(), (rows, w.d), generator=gen)]

    def scales(rows):
        return (base * torch.exp2(torch.rand(rows, generator=gen) * 2 - 1)).float()

    return {"q_pol": codes(w.N), "s_pol": scales(w.N), "q_ref": codes(w.N), "s_ref": scales(w.N),
            "q_W": codes(w.V), "s_W": scales(w.V)}
