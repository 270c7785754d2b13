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

The draws come from a counter-based generator (SplitMix64's output
function applied to a per-tensor key plus the element counter), turned into
uniforms by exact integer arithmetic and into normals by the Box-Muller
transform in float64, then rounded to float32 and, for bf16 workloads, to
bf16 by round-to-nearest-even on the bits. Every step but the three
float64 library functions of Box-Muller (log, cos, sin) is exact, and those
differ between hosts by an ulp at most, far below the float32 and bf16
roundings that follow. So a workload yields the same bytes on every host
(x86 or Arm, any thread count), which lets values computed once from these
inputs on one machine be checked on another; ``input_digest`` fingerprints
them. torch's own CPU generator does not give that: its normal sampler
takes a different vectorised path on different CPUs.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import hashlib
import os
from typing import Callable, Dict, Optional, Tuple

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


_M64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15      # SplitMix64's counter increment (the golden ratio in 64 bits)
_PAIRS_PER_TASK = 1 << 20        # Box-Muller pairs generated per thread task


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64's output function (Steele, Lea and Flood, "Fast splittable
    pseudorandom number generators", OOPSLA 2014) on a uint64 array; the
    products wrap modulo 2^64."""
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


class Stream:
    """Counter-based stream of 64-bit words for one tensor of one workload:
    word j is mix64(key + (j + 1) * gamma) modulo 2^64, as in SplitMix64
    started at ``key``; the key is derived from the seed and the tensor's
    name. Any range of words can be drawn independently of the others."""

    def __init__(self, seed: int, tag: str):
        digest = hashlib.sha256(("%d:%s" % (seed, tag)).encode()).digest()
        self.key = int.from_bytes(digest[:8], "little")

    def words(self, j0: int, n: int) -> np.ndarray:
        j = np.arange(j0 + 1, j0 + 1 + n, dtype=np.uint64)
        with np.errstate(over="ignore"):
            return _mix64(np.uint64(self.key) + j * np.uint64(_GAMMA))

    def below(self, n: int, bound: int) -> np.ndarray:
        """n integers uniform on [0, bound) (bound < 2^32): the high 32 bits of
        each word times bound, shifted down by 32 (exact in uint64)."""
        assert 0 < bound < (1 << 32)
        return ((self.words(0, n) >> np.uint64(32)) * np.uint64(bound)) >> np.uint64(32)

    def unit(self, n: int) -> np.ndarray:
        """n float64 uniforms on [0, 1): the top 53 bits of each word, times 2^-53."""
        return (self.words(0, n) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53

    def normal_pairs(self, j0: int, npairs: int) -> np.ndarray:
        """2 * npairs standard normals (float64) from words j0 .. j0 + npairs - 1
        by Box-Muller: u1 = (high 32 bits + 1/2) 2^-32 in (0, 1), u2 = (low 32
        bits) 2^-32, r = sqrt(-2 ln u1); the pair is (r cos 2 pi u2, r sin 2 pi u2)."""
        w = self.words(j0, npairs)
        u1 = ((w >> np.uint64(32)).astype(np.float64) + 0.5) * 2.0 ** -32
        u2 = (w & np.uint64(0xFFFFFFFF)).astype(np.float64) * 2.0 ** -32
        r = np.sqrt(-2.0 * np.log(u1))
        t = (2.0 * np.pi) * u2
        out = np.empty(2 * npairs)
        out[0::2] = r * np.cos(t)
        out[1::2] = r * np.sin(t)
        return out


def _bf16_bits(x32: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of float32 values, rounded to nearest even (finite inputs)."""
    b = x32.view(np.uint32)
    return ((b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
            ).astype(np.uint16)


def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _normal_tensor(stream: Stream, n: int, make: Callable[[int, np.ndarray], np.ndarray],
                   out: np.ndarray) -> None:
    """Fill out[0:n] with make(e0, normals) over tasks of consecutive elements
    e0 .. e0 + len(normals) - 1, in parallel; element 2j and 2j + 1 come from
    word j."""
    npairs = (n + 1) // 2

    def task(p0: int) -> None:
        p1 = min(npairs, p0 + _PAIRS_PER_TASK)
        z = stream.normal_pairs(p0, p1 - p0)
        e0 = 2 * p0
        e1 = min(n, 2 * p1)
        out[e0:e1] = make(e0, z[:e1 - e0])

    with cf.ThreadPoolExecutor(max_workers=_threads()) as ex:
        list(ex.map(task, range(0, npairs, _PAIRS_PER_TASK)))


def _gaussian(seed: int, tag: str, shape, std: float, dtype: str,
              base: Optional[np.ndarray] = None) -> np.ndarray:
    """std * N(0, 1) (plus ``base``, a float32 array or bf16 bit patterns of the
    same shape, when given), formed in float64, rounded to float32 and, for
    dtype "bf16", to bf16. Returns float32 values or uint16 bf16 bits."""
    n = int(np.prod(shape))
    st = Stream(seed, tag)
    bflat = None if base is None else base.reshape(-1)
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)

    def make(e0: int, z: np.ndarray) -> np.ndarray:
        x = std * z
        if bflat is not None:
            seg = bflat[e0:e0 + z.size]
            x = x + (_bf16_to_f64(seg) if dtype == "bf16" else seg.astype(np.float64))
        x32 = x.astype(np.float32)
        return _bf16_bits(x32) if dtype == "bf16" else x32

    _normal_tensor(st, n, make, out)
    return out.reshape(shape)


def _to_torch(a: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)


def _zipf_ids(seed: int, n: int, V: int, s: float) -> np.ndarray:
    """Ranks k = 1..V with pmf proportional to k^-s, sampled by inverse CDF
    from a float64 cumulative table; rank k maps to token id k - 1."""
    k = np.arange(1, V + 1, dtype=np.float64)
    cdf = np.cumsum(k ** (-s))
    cdf /= cdf[-1]
    u = Stream(seed, "ids").unit(n)
    ids = np.searchsorted(cdf, u, side="right")
    return np.minimum(ids, V - 1).astype(np.int32)


def make_mask(w: Workload) -> np.ndarray:
    """The uint8 [N] mask of workload ``w`` (its own stream: cheap to draw alone)."""
    B, T = w.B, w.T
    mask = np.ones((B, T), dtype=np.uint8)
    if w.mask == "tiny":
        # last 8 tokens of the generations with odd in-group index
        for b in range(B):
            if (b % w.G) % 2 == 1:
                mask[b, T - 8:] = 0
    elif w.mask == "pad_uniform":
        lengths = w.pad_lo + Stream(w.seed, "lengths").below(B, w.pad_hi - w.pad_lo + 1)
        mask = (np.arange(T)[None, :] < lengths.astype(np.int64)[:, None]).astype(np.uint8)
    elif w.mask == "tail_frac":
        mask[:, T - int(round(w.tail_frac * T)):] = 0
    return np.ascontiguousarray(mask.reshape(w.N))


def make_rewards(w: Workload):
    """(rewards, adv) of workload ``w``, float32 [B] each, one of them None:
    rewards per generation, or advantages supplied directly."""
    B = w.B
    rewards = adv = None
    if w.rewards == "normal":
        rewards = Stream(w.seed, "rewards").normal_pairs(0, (B + 1) // 2)[:B].astype(np.float32)
    elif w.rewards == "choice":
        vals = np.array(w.reward_values, dtype=np.float32)
        rewards = vals[Stream(w.seed, "rewards").below(B, len(w.reward_values)).astype(np.int64)]
    elif w.rewards == "adv_normal":
        adv = Stream(w.seed, "adv").normal_pairs(0, (B + 1) // 2)[:B].astype(np.float32)
    else:
        raise ValueError(w.rewards)
    return rewards, adv


def make_inputs(w: Workload) -> Dict[str, Optional[torch.Tensor]]:
    """Draw the host tensors of workload ``w``.

    Returns H_pol, H_ref ([N, d], dtype of ``w``), W ([V, d]), ids (int32
    [N]), mask (uint8 [N]) and either rewards (float32 [B]) or adv (float32
    [B], when advantages are supplied directly). Each tensor has its own
    stream, so the tensors do not depend on one another's sizes.
    """
    N, d, V, B, T = w.N, w.d, w.V, w.B, w.T
    dt = "f32" if w.dtype == "f32" else "bf16"

    H_pol = _gaussian(w.seed, "H_pol", (N, d), 1.0, dt)
    if w.ref == "independent":
        H_ref = _gaussian(w.seed, "H_ref", (N, d), 1.0, dt)
    else:
        H_ref = _gaussian(w.seed, "H_ref", (N, d), 0.05, dt, base=H_pol)
    W = _gaussian(w.seed, "W", (V, d), w.w_std, dt)

    if w.ids == "zipf":
        ids = _zipf_ids(w.seed, N, V, w.zipf_s)
    else:
        ids = Stream(w.seed, "ids").below(N, V).astype(np.int32)

    mask = make_mask(w)
    rewards, adv = make_rewards(w)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a))  # noqa: E731
    return {"H_pol": _to_torch(H_pol, dt), "H_ref": _to_torch(H_ref, dt), "W": _to_torch(W, dt),
            "ids": t(ids), "mask": t(mask), "rewards": t(rewards), "adv": t(adv)}


def input_digest(inp: Dict[str, Optional[torch.Tensor]]) -> str:
    """sha256 over the names, dtypes, shapes and bytes of a workload's host
    tensors, in a fixed order: a fingerprint that tells whether two machines
    drew the same inputs."""
    h = hashlib.sha256()
    for k in ("H_pol", "H_ref", "W", "ids", "mask", "rewards", "adv"):
        v = inp.get(k)
        if v is None:
            continue
        t = v.contiguous()
        raw = t.view(torch.int16) if t.dtype == torch.bfloat16 else t
        h.update(("%s|%s|%s|" % (k, t.dtype, tuple(t.shape))).encode())
        h.update(raw.numpy().tobytes())
    return h.hexdigest()


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
