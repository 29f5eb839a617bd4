"""Pins of the oracle's stochastic acceptance: the Philox4x32-10 noise, the
two-level Gumbel-max draw from softmax(logits / temperature), and the walk
that follows the draws, checked against the literal rejection rule of the
speculative-decoding tutorial (section 2.3) enumerated exactly."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from tests import indep


def test_philox_known_answers():
    # Known-answer vectors published with Philox4x32-10 (Salmon, Moraes, Dror
    # and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011, and
    # the Random123 release that accompanies it).
    ctr = np.array([[0, 0, 0, 0], [0xFFFFFFFF] * 4,
                    [0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344]], np.uint32)
    key = np.array([[0, 0], [0xFFFFFFFF] * 2, [0xA4093822, 0x299F31D0]], np.uint32)
    want = np.array([[0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8],
                     [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD],
                     [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]], np.uint32)
    np.testing.assert_array_equal(oracle.philox4x32_10(ctr, key), want)


_TRITON_PHILOX = r"""
import os, sys
os.environ["TRITON_INTERPRET"] = "1"
import numpy as np, torch, triton, triton.language as tl

@triton.jit
def k(c_ptr, out_ptr, seed, N: tl.constexpr):
    i = tl.arange(0, N)
    c0 = tl.load(c_ptr + 4 * i).to(tl.uint32, bitcast=True)
    c1 = tl.load(c_ptr + 4 * i + 1).to(tl.uint32, bitcast=True)
    c2 = tl.load(c_ptr + 4 * i + 2).to(tl.uint32, bitcast=True)
    c3 = tl.load(c_ptr + 4 * i + 3).to(tl.uint32, bitcast=True)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3, 10)
    tl.store(out_ptr + 4 * i, a.to(tl.int32, bitcast=True))
    tl.store(out_ptr + 4 * i + 1, b.to(tl.int32, bitcast=True))
    tl.store(out_ptr + 4 * i + 2, c.to(tl.int32, bitcast=True))
    tl.store(out_ptr + 4 * i + 3, d.to(tl.int32, bitcast=True))

ctr = np.frombuffer(bytes.fromhex(sys.argv[1]), dtype=np.uint32).copy()
seed = int(sys.argv[2])
c = torch.from_numpy(ctr.view(np.int32))
out = torch.zeros_like(c)
k[(1,)](c, out, seed, N=c.numel() // 4)
print(out.numpy().view(np.uint32).tobytes().hex())
"""


def test_philox_against_an_independent_implementation():
    """Triton's Philox4x32-10 (run on the CPU by its interpreter) on random
    counters; its key is (low, high) 32 bits of the seed."""
    pytest.importorskip("triton")
    rng = np.random.default_rng(5)
    ctr = rng.integers(0, 2**32, size=(16, 4), dtype=np.uint64).astype(np.uint32)
    for seed in (0, 0x299F31D0A4093822, 2**64 - 1):
        env = dict(os.environ, TRITON_INTERPRET="1")
        r = subprocess.run([sys.executable, "-c", _TRITON_PHILOX, ctr.tobytes().hex(), str(seed)],
                           capture_output=True, text=True, env=env, timeout=600)
        if r.returncode != 0:
            pytest.skip("triton interpreter unavailable: " + r.stderr.strip()[-200:])
        got = np.frombuffer(bytes.fromhex(r.stdout.strip().splitlines()[-1]),
                            dtype=np.uint32).reshape(16, 4)
        key = np.tile(np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32), (16, 1))
        np.testing.assert_array_equal(oracle.philox4x32_10(ctr, key), got)


def _chi2(counts, probs):
    exp = probs * counts.sum()
    return float(((counts - exp) ** 2 / exp).sum())


@pytest.mark.parametrize("temperature", [0.5, 1.0, 2.5])
def test_draws_follow_the_tempered_softmax(temperature):
    """Many independent draws (one per request index) of one row of 10 logits
    cut into chunks of 4, 4 and 2 tokens: the frequencies match
    softmax(l / temperature) (chi-square, 9 degrees of freedom; 33.7 is the
    1e-4 quantile)."""
    l = torch.tensor([0.3, -1.2, 2.0, 0.0, 1.1, -0.4, 0.9, -2.5, 1.6, 0.2])
    n = 40000
    logits = l.repeat(n, 1, 1)                              # [n][1][10]
    smp, _ = oracle.sample_rows(logits, np.ones(n, np.int32), np.full(n, 7, np.int32),
                                temperature, seed=0x1234_5678_9ABC, chunk=4)
    counts = np.bincount(smp[:, 0], minlength=10).astype(np.float64)
    p = torch.softmax(l.double() / temperature, 0).numpy()
    assert _chi2(counts, p) < 33.7


def test_one_chunk_and_many_chunks_give_the_same_law():
    l = torch.tensor([1.0, 0.5, -0.5, 2.0, 0.0, -1.0, 1.5])
    n = 30000
    logits = l.repeat(n, 1, 1)
    p = torch.softmax(l.double(), 0).numpy()
    for chunk in (1, 3, 7):
        smp, _ = oracle.sample_rows(logits, np.ones(n, np.int32), np.zeros(n, np.int32), 1.0,
                                    seed=99, chunk=chunk)
        counts = np.bincount(smp[:, 0], minlength=7).astype(np.float64)
        assert _chi2(counts, p) < 27.9          # 6 degrees of freedom, 1e-4 quantile


def test_noise_changes_with_every_counter_word():
    l = torch.zeros(1, 2, 5000)
    base, _ = oracle.sample_rows(l, np.array([2]), np.array([3]), 1.0, seed=1)
    assert base[0, 0] != base[0, 1]                         # row
    other_pos, _ = oracle.sample_rows(l, np.array([2]), np.array([4]), 1.0, seed=1)
    other_seed, _ = oracle.sample_rows(l, np.array([2]), np.array([3]), 1.0, seed=2)
    two, _ = oracle.sample_rows(l.repeat(2, 1, 1), np.array([2, 2]), np.array([3, 3]), 1.0, 1)
    assert (other_pos != base).any() and (other_seed != base).any()
    assert (two[1] != two[0]).any()                          # request
    assert (two[0] == base[0]).all()


def test_low_temperature_is_the_argmax():
    g = torch.Generator().manual_seed(3)
    logits = torch.randn(4, 6, 9000, generator=g)
    smp, _ = oracle.sample_rows(logits, np.full(4, 6, np.int32), np.arange(4, dtype=np.int32),
                                1e-3, seed=11)
    am, margin = oracle.argmax(logits)
    ok = margin > 0.05
    assert ok.sum() > 20
    np.testing.assert_array_equal(smp[ok], am[ok])


def test_padding_rows_and_gaps():
    g = torch.Generator().manual_seed(4)
    logits = torch.randn(2, 4, 6000, generator=g)
    nn = np.array([3, 1], np.int32)
    kv = np.array([10, 20], np.int32)
    smp, mar = oracle.sample_rows(logits, nn, kv, 0.8, seed=5)
    assert (smp[0, 3:] == -1).all() and (smp[1, 1:] == -1).all()
    assert np.isinf(mar[0, 3:]).all()
    for b in range(2):
        for t in range(nn[b]):
            gap = oracle.sample_gaps(logits[b, t], t, b, kv[b], 0.8, 5, int(smp[b, t]))
            assert gap == (0.0, 0.0)
            other = (int(smp[b, t]) + 4097) % 6000              # the other chunk
            cg, tg = oracle.sample_gaps(logits[b, t], t, b, kv[b], 0.8, 5, other)
            assert cg > 0.0 or tg > 0.0
            assert min(cg, tg) >= 0.0


def _tiny_tree():
    # root(0) -> 1 (token 2), 2 (token 0); 1 -> 3 (token 4), 4 (token 1);
    # 3 -> 5 (token 3); m = 3, vocabulary 5
    tree = dict(node_tok=np.array([[1, 2, 0, 4, 1, 3]], np.int32),
                node_parent=np.array([[-1, 0, 0, 1, 1, 3]], np.int32),
                n_nodes=np.array([6], np.int32))
    return tree, 3


@pytest.mark.parametrize("temperature", [0.7, 1.5])
def test_walk_over_draws_follows_the_rejection_rule(temperature):
    """The oracle's stochastic acceptance (draw at every row, follow the
    matching child) against the exact law of the tutorial's rejection rule
    with fixed drafts: chi-square over the outcomes (accepted tokens + bonus)."""
    tree, m = _tiny_tree()
    g = torch.Generator().manual_seed(8)
    rows = torch.randn(6, 5, generator=g) * 1.5
    rows[0, 2] += 1.0                      # make deep paths likely enough
    rows[1, 4] += 1.0
    rows[3, 3] += 1.5
    law = indep.rejection_outcomes(tree["node_tok"][0], tree["node_parent"][0], 6,
                                   torch.softmax(rows.double() / temperature, -1).numpy(), m)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    n = 40000
    nb = {k: np.repeat(v, n, 0) for k, v in tree.items()}
    smp, _ = oracle.sample_rows(rows.repeat(n, 1, 1), nb["n_nodes"], np.full(n, 17, np.int32),
                                temperature, seed=2024, chunk=2)
    acc = oracle.accept(nb, smp, m)
    seen = {}
    for b in range(n):
        key = tuple(int(x) for x in acc["out_tok"][b, :acc["accept_len"][b]])
        seen[key] = seen.get(key, 0) + 1
    assert set(seen) <= set(law)
    # bins with expected count >= 20, the rest merged into one
    big = [k for k, v in law.items() if v * n >= 20]
    rest_p = 1.0 - sum(law[k] for k in big)
    counts = np.array([seen.get(k, 0) for k in big] + [n - sum(seen.get(k, 0) for k in big)],
                      np.float64)
    probs = np.array([law[k] for k in big] + [rest_p])
    keep = probs > 0
    dof = int(keep.sum()) - 1
    # 1e-4 quantile of chi-square by the Wilson-Hilferty approximation
    crit = dof * (1 - 2 / (9 * dof) + 3.719 * np.sqrt(2 / (9 * dof))) ** 3
    assert _chi2(counts[keep], probs[keep]) < crit
    # and the mean accepted length matches the law's
    tau_law = sum(p * len(k) for k, p in law.items())
    assert abs(acc["accept_len"].mean() - tau_law) < 0.03
