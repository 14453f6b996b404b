"""The seeded input generator (synth.py) against its stated recipe.

- SplitMix64 matches the published reference outputs for seed 0
  (0xe220a8397b1dcdaf, 0x6e789e6aa1b965f4, 0x06c45d188009454f).
- The weight generators: field ranges and determinism.
- The activations: N(0, sigma^2) moments, and round(0.01 K) outlier columns
  scaled x8.
- The router: top_k distinct experts per token, uniform without skew, and
  weighted toward low expert ids with skew.
- The benchmark workloads: shapes, seeds (1000 + i for weights, (1000 + i) * 100
  + 7 for X; 1004 and 100400 + M for the sweep), scales and outlier columns."""
import numpy as np
import pytest

import synth


def test_splitmix64_reference_vectors():
    z = synth.splitmix64(0, 3)
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    # a window of the stream equals the same outputs taken from its start
    assert np.array_equal(synth.splitmix64(7, 5, start=3), synth.splitmix64(7, 8)[3:])


def test_uniform_and_normal_moments():
    u = synth.uniform01(11, 200000)
    assert u.min() >= 0.0 and u.max() < 1.0 and abs(u.mean() - 0.5) < 0.005
    z = synth.normal(12, 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert abs(np.mean(z ** 4) - 3.0) < 0.1          # Gaussian kurtosis


def fp16_field(w, off):
    return w[:, off:off + 2].copy().view(np.float16).astype(np.float64).ravel()


def test_q4k_fields():
    N, K = 64, 1024
    w = synth.gen_q4k(N, K, 3)
    assert w.shape == (N, (K // 256) * 144) and np.array_equal(w, synth.gen_q4k(N, K, 3))
    assert not np.array_equal(w, synth.gen_q4k(N, K, 4))
    blocks = w.reshape(-1, 144)
    d, dmin = fp16_field(blocks, 0), fp16_field(blocks, 2)
    lo, hi = float(np.float16(1e-4)), float(np.float16(1e-3))
    assert d.min() >= lo and d.max() <= hi and dmin.min() >= lo and dmin.max() <= hi
    assert abs(d.mean() - 5.5e-4) < 3e-5                        # uniform on [1e-4, 1e-3]
    q = np.concatenate([blocks[:, 16:] & 15, blocks[:, 16:] >> 4]).ravel()
    assert np.bincount(q, minlength=16).min() > 0.9 * q.size / 16  # 4-bit codes uniform


def test_q6k_fields():
    N, K = 64, 1024
    w = synth.gen_q6k(N, K, 5).reshape(-1, 210)
    sc = w[:, 192:208].view(np.int8).ravel()
    assert sc.min() == -32 and sc.max() == 31                   # int8 sub-scales uniform on [-32, 31]
    d = fp16_field(w, 208)
    assert d.min() >= float(np.float16(1e-4)) and d.max() <= float(np.float16(1e-3))


def test_q6k_full_scale_fields():
    w = synth.gen_q6k(64, 1024, 5, full_scales=True).reshape(-1, 210)
    sc = w[:, 192:208].view(np.int8).ravel().astype(np.int64)
    assert sc.min() == -128 and sc.max() == 127                 # the whole int8 range
    assert np.bincount(sc + 128, minlength=256).min() > 0        # every value drawn
    assert abs((np.abs(sc) > 64).mean() - 127 / 256) < 0.03     # about half beyond +-64
    # the other fields are those of the plain generator
    w0 = synth.gen_q6k(64, 1024, 5).reshape(-1, 210)
    assert np.array_equal(np.delete(w, np.s_[192:208], axis=1), np.delete(w0, np.s_[192:208], axis=1))


def test_ptq1_fields():
    w = synth.gen_ptq1(32, 1024, 6).reshape(-1, 28)
    assert w[:, :24].max() < 243 and w[:, 24:26].max() < 81
    d = fp16_field(w, 26)
    assert d.min() >= float(np.float16(1e-3)) and d.max() <= float(np.float16(1e-2))


def test_activations_and_outliers():
    M, K = 64, 2048
    x = synth.gen_x(M, K, 7, sigma=0.5)
    assert x.dtype == np.float32 and abs(x.std() - 0.5) < 0.01
    xo = synth.gen_x(M, K, 7, outlier_frac=0.01)
    cols = synth.outlier_columns(K, 7)
    assert len(cols) == round(0.01 * K) == 20 and len(set(cols.tolist())) == 20
    base = synth.gen_x(M, K, 7)
    assert np.array_equal(xo[:, cols], base[:, cols] * np.float32(8.0))
    rest = np.setdiff1d(np.arange(K), cols)
    assert np.array_equal(xo[:, rest], base[:, rest])


def test_router():
    M, top_k, E = 4000, 2, 8
    ids = synth.gen_ids(M, top_k, E, 9)
    assert ids.shape == (M, top_k) and ids.min() >= 0 and ids.max() < E
    assert np.all(ids[:, 0] != ids[:, 1])                        # distinct experts per token
    counts = np.bincount(ids.ravel(), minlength=E)
    assert counts.min() > 0.9 * counts.mean()                    # skew 0: uniform
    skewed = np.bincount(synth.gen_ids(M, top_k, E, 9, skew=2.0).ravel(), minlength=E)
    assert skewed[0] > 3 * skewed[E - 1] and np.all(np.diff(skewed) <= 50)


@pytest.mark.parametrize("i,wl,shape,wtype,sigma,outliers",
                         [(0, synth.C0, (64, 2048, 2048), 4, 1.0, 0.0), (1, synth.C1, (512, 2048, 11008), 4, 1.0, 0.01),
                          (2, synth.C2, (512, 11008, 2048), 6, 1.0, 0.0), (3, synth.C3, (2048, 4096, 14336), 4, 0.5, 0.0)])
def test_benchmark_workloads(i, wl, shape, wtype, sigma, outliers):
    # seeds 1000 + i for the weights, (1000 + i) * 100 + 7 for X
    assert (wl.M, wl.K, wl.N) == shape and wl.wtype == wtype
    assert (wl.w_seed, wl.x_seed) == (1000 + i, (1000 + i) * 100 + 7)
    assert wl.sigma == sigma and wl.outlier_frac == outliers


def test_sweep_workloads():
    # the K = N = 5120 sweep: one weight matrix (seed 1004), X seeded per M
    assert synth.SWEEP_M == (1, 4, 8, 64, 512, 2048, 8192)
    for m in synth.SWEEP_M:
        wl = synth.sweep(m)
        assert (wl.M, wl.K, wl.N, wl.wtype) == (m, 5120, 5120, 4)
        assert (wl.w_seed, wl.x_seed) == (1004, 100400 + m)
