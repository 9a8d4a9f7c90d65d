"""Pins for the oracle's random stream and Gumbel-max sampler (CPU only).

Philox-4x32-10 is pinned against NVIDIA's curand *host* generator
(CURAND_RNG_PSEUDO_PHILOX4_32_10, run as a library on the CPU): with its default
ordering, output 4*s + w of a batch is word w of Philox(counter=(0,0,s,0),
key=seed), and a generator offset of 262144*i moves counter word 0 to i (with
carry into word 1).  That is an implementation written independently of ours.
"""
import ctypes
import ctypes.util
import os

import numpy as np
import pytest
from scipy import stats
from scipy.special import logsumexp, softmax

import oracle


def _curand():
    for path in ("/usr/local/cuda/lib64/libcurand.so", ctypes.util.find_library("curand")):
        if path and os.path.exists(path):
            try:
                return ctypes.CDLL(path)
            except OSError:
                pass
    pytest.skip("libcurand not available")


def _curand_words(seed: int, offset: int, n: int) -> np.ndarray:
    cur = _curand()
    gen = ctypes.c_void_p()
    assert cur.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0  # PHILOX4_32_10
    try:
        assert cur.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert cur.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        buf = np.zeros(n, dtype=np.uint32)
        assert cur.curandGenerate(gen, buf.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
        return buf
    finally:
        cur.curandDestroyGenerator(gen)


@pytest.mark.parametrize("seed", [0, 1, 0x123456789ABCDEF, 0xFFFFFFFFFFFFFFFF, 0xDEADBEEF00000000])
def test_philox_matches_curand_subsequences(seed):
    key = (seed & 0xFFFFFFFF, seed >> 32)
    words = _curand_words(seed, 0, 4 * 300)
    for s in range(300):
        got = oracle.philox4x32_10((0, 0, s, 0), key)
        assert list(got) == list(words[4 * s: 4 * s + 4]), s


@pytest.mark.parametrize("c0,c1,s", [(1, 0, 0), (5, 0, 7), (4096, 0, 123), ((1 << 32) - 1, 0, 9),
                                     (0, 1, 0), (3, 1, 17), (7, 2, 1000)])
def test_philox_matches_curand_counter_words_0_and_1(c0, c1, s):
    seed = 0x0123456789ABCDEF
    key = (seed & 0xFFFFFFFF, seed >> 32)
    offset = 262144 * (c0 + (c1 << 32)) + 4 * s
    words = _curand_words(seed, offset, 4)
    assert list(oracle.philox4x32_10((c0, c1, s, 0), key)) == list(words)


def test_uniform_is_open_interval_odd_multiple():
    seed = 77
    key = (seed & 0xFFFFFFFF, seed >> 32)
    for v in range(64):
        for purpose in range(4):
            u = oracle.uniform(seed, v, 3, 11, purpose)
            word = int(oracle.philox4x32_10((v // 4, 3, 11, purpose), key)[v % 4])
            scaled = u * 2.0 ** 24
            assert 0.0 < u < 1.0
            assert scaled == int(scaled) and int(scaled) % 2 == 1
            # the 23 low bits of the word select the odd multiple
            assert (int(scaled) - 1) // 2 == word & 0x7FFFFF


def test_uniform_streams_differ_by_purpose_position_request():
    vals = {oracle.uniform(5, 0, j, rid, p) for j in range(3) for rid in range(3) for p in range(4)}
    assert len(vals) == 36


def test_uniform_distribution_chisquare():
    u = np.array([oracle.uniform(9, v, 1, 2, 0) for v in range(40000)])
    counts, _ = np.histogram(u, bins=20, range=(0, 1))
    assert stats.chisquare(counts).pvalue > 1e-3


@pytest.mark.parametrize("V,temp", [(8, 1.0), (5, 0.5), (12, 2.0)])
def test_gumbel_max_draft_matches_softmax(V, temp):
    """x_1 ~ softmax(U/T) over 2e5 independent requests (no bias: A = C = 0)."""
    rng = np.random.default_rng(V)
    R = 200_000
    Urow = rng.normal(0, 1.5, size=V).astype(np.float32)
    U = np.broadcast_to(Urow, (R, 1, V))
    A = np.zeros((1, V, 1), np.float32)
    out = oracle.draft(U, A, A, np.zeros(R, np.int32), [temp], seed=1234, rid_base=0)
    p = softmax(Urow.astype(np.float64) / temp)
    counts = np.bincount(out.x[:, 0], minlength=V)
    assert stats.chisquare(counts, p * R).pvalue > 1e-3
    # q_tok and lse are the closed forms of the sampled token
    z = Urow.astype(np.float64) / temp
    assert np.allclose(out.lse[:, 0], logsumexp(z), rtol=0, atol=1e-12)
    assert np.allclose(out.q_tok[:, 0], p[out.x[:, 0]], rtol=1e-12, atol=0)


def test_gumbel_argmax_excludes_neg_inf_and_reports_gap():
    lw = np.array([-np.inf, 0.0, -np.inf, 0.5])
    seen = set()
    for rid in range(200):
        idx, gap = oracle.gumbel_argmax(lw, 3, 1, rid, 2)
        seen.add(idx)
        assert gap > 0
    assert seen == {1, 3}
    idx, gap = oracle.gumbel_argmax(np.array([-np.inf, 1.0]), 3, 1, 0, 2)
    assert idx == 1 and gap == np.inf


def test_gumbel_argmax_of_dominant_logit():
    lw = np.zeros(16)
    lw[9] = 40.0  # Gumbel noise spans [-2.9, 16.7] for this stream
    assert all(oracle.gumbel_argmax(lw, s, 1, 0, 0)[0] == 9 for s in range(50))


def test_gumbel_noise_value_is_minus_log_minus_log_u():
    """G = -ln(-ln u): with a single candidate per position the score gap is inf,
    but with two equal logits the winner is the larger u (G is increasing in u)."""
    for rid in range(100):
        u0 = oracle.uniform(4, 0, 1, rid, 0)
        u1 = oracle.uniform(4, 1, 1, rid, 0)
        idx, gap = oracle.gumbel_argmax(np.zeros(2), 4, 1, rid, 0)
        assert idx == (0 if u0 > u1 else 1)
        g0, g1 = -np.log(-np.log(u0)), -np.log(-np.log(u1))
        assert abs(gap - abs(g0 - g1)) < 1e-12
