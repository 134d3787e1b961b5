"""The tensor-core building blocks (swizzled shared-memory operands and
their descriptors, tcgen05.mma into tensor memory, mbarrier completion,
tcgen05.ld) give exactly A B^T on inputs whose products and sums are exact
in fp16 / fp32."""
import numpy as np
import pytest
import torch

import soft_clustering_gb300 as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from soft_clustering_gb300 import build
    build.build()


@pytest.mark.parametrize("kdim", [64, 128, 256, 80, 144, 272])
@pytest.mark.parametrize("n", [64, 128])
def test_tc_gemm_exact(kdim, n):
    rng = np.random.default_rng(kdim * 1000 + n)
    A = (rng.integers(-8, 9, (128, kdim)) * 0.25).astype(np.float16)
    B = (rng.integers(-8, 9, (n, kdim)) * 0.125).astype(np.float16)
    want = A.astype(np.float64) @ B.astype(np.float64).T
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    dC = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert G.gmm_debug_tc_gemm(dA, dB, dC, kdim, n, st) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = dC.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]
