"""The seeded input generator (ftgen) against the distributions the workloads
call for: standard normals, uniforms and permutations from counter-addressed
streams, x rounded to bf16, and the Zipf popularity bias of the router logits.
The generator feeds both the GPU library and the oracle, so these checks pin
the workloads, not the parity."""
import numpy as np
import scipy.stats
import torch

import ftgen


def test_normals_are_standard_normal():
    z = ftgen.normal(7, 3, 1 << 20).astype(np.float64)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1.0) < 5e-3
    assert scipy.stats.kstest(z, "norm").statistic < 3e-3


def test_uniforms_are_uniform_and_streams_are_independent():
    u = ftgen.uniform(7, 3, 1 << 20).astype(np.float64)
    assert u.min() >= 0.0 and u.max() < 1.0
    assert scipy.stats.kstest(u, "uniform").statistic < 3e-3
    v = ftgen.uniform(7, 4, 1 << 20).astype(np.float64)
    assert abs(np.corrcoef(u, v)[0, 1]) < 5e-3
    w = ftgen.uniform(8, 3, 1 << 20).astype(np.float64)
    assert abs(np.corrcoef(u, w)[0, 1]) < 5e-3
    # counter addressing: any window is the same counters of the whole stream
    np.testing.assert_array_equal(ftgen.uniform(7, 3, 100, ctr0=1000), ftgen.uniform(7, 3, 1100)[1000:])
    np.testing.assert_array_equal(ftgen.normal(7, 3, 64, ctr0=4096), ftgen.normal(7, 3, 4160)[4096:])


def test_permutations_are_uniform_permutations():
    E, n = 8, 4000
    counts = np.zeros((E, E), np.int64)
    for st in range(n):
        p = ftgen.permutation(5, st, E)
        assert sorted(p.tolist()) == list(range(E))
        counts[np.arange(E), p] += 1
    # each value lands in each position 1/E of the time (5 sigma)
    mean, sd = n / E, (n * (1 / E) * (1 - 1 / E)) ** 0.5
    assert np.all(np.abs(counts - mean) < 5 * sd)


def test_x_is_the_normals_rounded_to_bf16():
    T, H, step, layer = 64, 256, 3, 5
    bits = ftgen.x_bf16(11, T, H, step, layer)
    z = ftgen.normal(11, ftgen._sid(ftgen._K_X, layer, step), T * H).reshape(T, H)
    ref = torch.from_numpy(z).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, ref)
    # (layer, step) address independent streams
    assert not np.array_equal(ftgen.x_bf16(11, T, H, step, layer + 1), bits)


def test_zipf_bias_gives_zipf_popularity():
    E, s = 128, 1.1
    b = ftgen.zipf_bias(3, E, s, 0).astype(np.float64)
    p = np.exp(b)
    assert abs(p.sum() - 1.0) < 1e-5
    ranked = np.sort(p)[::-1]
    np.testing.assert_allclose(ranked / ranked[0], np.arange(1, E + 1, dtype=np.float64) ** -s, rtol=1e-5)
    # the logits' column means recover the bias under N(0,1) noise (4096 tokens: 5 sigma = 0.08)
    lg = ftgen.router_logits(3, 4096, E, 0, 0, s)
    np.testing.assert_allclose(lg.mean(axis=0), b, atol=0.08)
    np.testing.assert_allclose(lg.std(axis=0), 1.0, atol=0.08)
    # a new epoch re-draws the ranks; layers have their own
    assert not np.array_equal(ftgen.zipf_bias(3, E, s, 0, epoch=1), ftgen.zipf_bias(3, E, s, 0))
    assert not np.array_equal(ftgen.zipf_bias(3, E, s, 1), ftgen.zipf_bias(3, E, s, 0))
