"""The seeded input generator: determinism, the planted recipes, and
bit-identical points from the host and the device."""
import numpy as np
import pytest

import datagen


def test_points_deterministic_and_index_addressable():
    wl = datagen.WORKLOADS["embed_diag"].with_n(5000)
    mix = datagen.planted(wl)
    a = datagen.points(mix, 0, 300)
    b = datagen.points(mix, 100, 50)
    c = datagen.points_at(mix, np.arange(100, 150))
    assert (a[100:150] == b).all() and (b == c).all()
    assert (datagen.points(datagen.planted(wl), 0, 300) == a).all()


def test_sphere_points_unit_norm():
    wl = datagen.WORKLOADS["embed_diag"].with_n(2000)
    mix = datagen.planted(wl)
    x = datagen.to_double(mix, datagen.points(mix, 0, 2000))
    assert np.abs(np.linalg.norm(x, axis=1) - 1).max() < 5e-3  # fp16 storage
    assert np.abs(np.linalg.norm(mix.mu, axis=1) - 1).max() < 1e-12


def test_planted_moments_diag():
    wl = datagen.WORKLOADS["tiny_diag"].with_n(200_000)
    mix = datagen.planted(wl)
    x = datagen.to_double(mix, datagen.points(mix, 0, wl.N))
    # nearest planted centre recovers the draw's component (well separated)
    d = ((x[:, None, :] - mix.mu[None]) ** 2 / (mix.sd[None] ** 2)).sum(-1)
    z = d.argmin(1)
    frac = np.bincount(z, minlength=wl.K) / wl.N
    assert np.abs(frac - mix.weights).max() < 0.01
    for k in range(wl.K):
        xs = x[z == k]
        assert np.abs(xs.mean(0) - mix.mu[k]).max() < 6 * mix.sd[k].max() / np.sqrt(len(xs))
        assert np.abs(xs.var(0) / mix.sd[k] ** 2 - 1).max() < 0.1


def test_planted_full_covariance():
    wl = datagen.WORKLOADS["full_cov"].with_n(100_000)
    mix = datagen.planted(wl)
    assert np.allclose(np.einsum("kij,klj->kil", mix.chol, mix.chol), mix.sigma, atol=1e-10)
    x = datagen.to_double(mix, datagen.points(mix, 0, 20_000))
    assert np.isfinite(x).all()


def test_dirichlet_weights_and_ivf_midpoints():
    wl = datagen.WORKLOADS["large_diag"].with_n(1000)
    mix = datagen.planted(wl)
    assert abs(mix.weights.sum() - 1) < 1e-12 and (mix.weights > 0).all()
    # Dirichlet(0.5) over 1024 components is skewed: its largest weights are far above 1/K
    assert mix.weights.max() > 5.0 / wl.K
    wl5 = datagen.WORKLOADS["ivf_assign"].with_n(4_000)
    mix5 = datagen.planted(wl5)
    x = datagen.to_double(mix5, datagen.points(mix5, 0, wl5.N))
    # mixture draws sit within ~128 sigma^2 <= 32 of their centre; midpoints
    # of two centres ~|mu_a - mu_b|^2/4 ~ 64 from every centre: ~10% of points
    d2 = ((x * x).sum(1)[:, None] - 2 * x @ mix5.mu.T + (mix5.mu ** 2).sum(1)[None]).min(1)
    assert 0.06 < (d2 > 48).mean() < 0.14


def test_init_params():
    wl = datagen.WORKLOADS["tiny_diag"]
    mix = datagen.planted(wl)
    pi, mu, var = datagen.init_params(mix)
    assert pi.shape == (wl.K,) and np.allclose(pi, 1.0 / wl.K)
    assert len({tuple(r) for r in mu}) == wl.K
    x = datagen.to_double(mix, datagen.points(mix, 0, wl.N))
    assert np.allclose(var[0], x.var(0), rtol=1e-5)


def test_rounding_matches_numpy_f16():
    lib = datagen.host_lib()
    vals = np.concatenate([np.random.default_rng(0).standard_normal(20000) * 10,
                           np.random.default_rng(1).standard_normal(2000) * 1e-6,
                           [65504.0, 65519.99, 6.1e-5, 5.96e-8, 2.98e-8, 0.0, -0.0]])
    ours = np.array([lib.gen_to_f16_host(float(v)) for v in vals], dtype=np.uint16)
    ref = vals.astype(np.float16).view(np.uint16)
    assert (ours == ref).all()


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(datagen.WORKLOADS))
def test_device_points_bit_identical(name):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    wl = datagen.WORKLOADS[name]
    mix = datagen.planted(wl)
    keep, ptrs = datagen.upload_tables(mix)
    start, count = max(0, wl.N - 3000), 3000
    esz = 4 if wl.dtype == datagen.F32 else 2
    out = torch.empty(count * wl.D * esz, dtype=torch.uint8, device="cuda")
    datagen.device_points(mix, start, count, out.data_ptr(), 0, ptrs)
    torch.cuda.synchronize()
    dev = out.cpu().numpy().view(np.float32 if wl.dtype == datagen.F32 else np.uint16)
    host = datagen.points(mix, start, count).reshape(-1)
    assert (dev.view(np.uint32 if esz == 4 else np.uint16) ==
            host.view(np.uint32 if esz == 4 else np.uint16)).all()
