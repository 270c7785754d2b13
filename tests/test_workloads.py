"""The seeded input generator: its counter-based words match SplitMix64's
published definition, its conversions are exact, its draws have the stated
distributions, and a workload's bytes depend on nothing but the workload
(not the thread count, not the order of the draws)."""
import numpy as np
import pytest
import torch

from grpo_loss_gb300 import workloads as WL


def _splitmix64_reference(state: int, n: int):
    """SplitMix64 as published (Steele, Lea and Flood, OOPSLA 2014), on Python
    ints: state += gamma; z = state; two xor-shift-multiply rounds; a final
    xor-shift."""
    m = (1 << 64) - 1
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & m
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
        out.append(z ^ (z >> 31))
    return out


def test_words_follow_splitmix64():
    s = WL.Stream(0, "any")
    s.key = 1234567
    # the first outputs of SplitMix64 seeded with 1234567, as printed by its
    # reference implementation
    assert s.words(0, 5).tolist() == [6457827717110365317, 3203168211198807973,
                                      9817491932198370423, 4593380528125082431,
                                      16408922859458223821]
    s = WL.Stream(1002, "H_pol")
    assert s.words(0, 64).tolist() == _splitmix64_reference(s.key, 64)
    # any window of the stream equals the same words drawn from the start
    assert s.words(37, 5).tolist() == s.words(0, 42)[37:].tolist()


def test_box_muller_pairs():
    s = WL.Stream(5, "t")
    z = s.normal_pairs(0, 4096)
    w = s.words(0, 4096)
    u1 = ((w >> np.uint64(32)).astype(np.float64) + 0.5) * 2.0 ** -32
    # each pair lies on the circle of radius sqrt(-2 ln u1)
    r2 = z[0::2] ** 2 + z[1::2] ** 2
    assert np.allclose(r2, -2.0 * np.log(u1), rtol=1e-12, atol=1e-300)
    big = s.normal_pairs(0, 1 << 19)
    assert abs(big.mean()) < 5e-3 and abs(big.std() - 1.0) < 5e-3
    # fourth moment of a normal is 3
    assert abs(np.mean(big ** 4) - 3.0) < 0.05


def test_bf16_rounding_is_torchs():
    g = torch.Generator().manual_seed(1)
    x = torch.randn(100000, generator=g) * torch.exp2(torch.randint(-20, 20, (100000,),
                                                                    generator=g).float())
    # exact ties between bf16 neighbours round to even
    ties = torch.tensor([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 0.0, -0.0])
    x = torch.cat([x, ties])
    mine = WL._bf16_bits(x.numpy())
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_integer_draws_are_in_range_and_uniform():
    s = WL.Stream(9, "ids")
    v = s.below(200000, 1000)
    assert v.min() >= 0 and v.max() < 1000
    counts = np.bincount(v.astype(np.int64), minlength=1000)
    assert counts.min() > 120 and counts.max() < 290        # mean 200
    u = s.unit(100000)
    assert u.min() >= 0.0 and u.max() < 1.0 and abs(u.mean() - 0.5) < 5e-3


def test_inputs_do_not_depend_on_thread_count(monkeypatch):
    w = WL.SMALL["gpt-oss-small"]
    a = WL.input_digest(WL.make_inputs(w))
    monkeypatch.setattr(WL, "_threads", lambda: 1)
    monkeypatch.setattr(WL, "_PAIRS_PER_TASK", 777)
    assert WL.input_digest(WL.make_inputs(w)) == a


def test_workload_recipes():
    w = WL.SMALL["qwen2.5-small"]
    inp = WL.make_inputs(w)
    H = inp["H_pol"].float()
    assert inp["H_pol"].dtype == torch.bfloat16 and inp["W"].shape == (w.V, w.d)
    assert abs(H.mean().item()) < 0.01 and abs(H.std().item() - 1) < 0.01
    assert abs(inp["W"].float().std().item() - w.w_std) < 2e-4
    noise = (inp["H_ref"].float() - H) / 0.05
    assert abs(noise.std().item() - 1) < 0.02
    m = inp["mask"].reshape(w.B, w.T)
    lengths = m.sum(1)
    assert lengths.min() >= w.pad_lo and lengths.max() <= w.pad_hi
    # right padding: every row is a prefix of ones
    assert bool(torch.all(m[:, :-1] >= m[:, 1:]))
    assert set(inp["rewards"].tolist()) <= set(w.reward_values)
    tiny = WL.make_inputs(WL.TINY)
    assert tiny["H_pol"].dtype == torch.float32 and int(tiny["mask"].sum()) == 480
    q3 = WL.make_inputs(WL.SMALL["qwen3-small"])
    assert q3["rewards"] is None and q3["adv"].shape == (1,)
    assert int(q3["mask"].sum()) == 990


def test_zipf_ids_follow_the_power_law():
    w = WL.GPTOSS_20B.scaled("zipf-check", prompts=1, G=1, T=200000, d=16, V=5000,
                             pad_lo=200000, pad_hi=200000)
    ids = WL._zipf_ids(w.seed, w.N, w.V, w.zipf_s)
    counts = np.bincount(ids, minlength=w.V).astype(np.float64)
    k = np.arange(1, w.V + 1, dtype=np.float64)
    pmf = k ** -w.zipf_s / np.sum(k ** -w.zipf_s)
    # the most frequent ranks within a few standard errors of the pmf
    for r in range(5):
        expect = pmf[r] * w.N
        assert abs(counts[r] - expect) < 5 * np.sqrt(expect), r
    assert ids.min() >= 0 and ids.max() < w.V


@pytest.mark.parametrize("w", [WL.QWEN25_1P5B, WL.LLAMA31_8B_20K, WL.QWEN3_8B_110K,
                               WL.GPTOSS_20B], ids=lambda w: w.name)
def test_golden_files_match_the_generator(w):
    """The stored full-size oracle values were computed on this generator's
    inputs: their valid-token count is this mask's, and the float32
    advantages they record are the oracle's advantages of this generator's
    rewards (or the supplied advantages). The input digest itself is checked
    where the full inputs are drawn, beside the GPU run."""
    import json
    import os

    from oracle import grpo_oracle as O
    path = os.path.join(os.path.dirname(__file__), "golden", "fullsize_%s.json" % w.name)
    if not os.path.exists(path):
        pytest.skip("golden values not written yet")
    rec = json.load(open(path))
    assert rec["workload"] == w.name and len(rec["input_digest"]) == 64
    assert rec["n_valid"] == int(WL.make_mask(w).sum())
    rewards, adv = WL.make_rewards(w)
    if adv is None:
        adv = O.advantages(rewards, w.G, w.eps, w.std_unbiased).astype(np.float32)
    assert [float(a) for a in adv] == rec["adv_float32"]
