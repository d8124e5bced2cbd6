"""GPU: the tensor-core building blocks (descriptors, MMA kinds, tf32 split)
against numpy, through the self-test entry point."""
import ctypes as C

import numpy as np
import pytest
import torch

from _gpu import dev, need_gpu

pytestmark = pytest.mark.gpu

TF32, TF32X3, BF16 = 0, 1, 2
MN_SWAP = 0


def _run(kind, n, k, a_mn, b_mn, seed=0, mn_swap=MN_SWAP):
    from offline_rl_step_gb300 import _abi
    need_gpu()
    lib = _abi.load()
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((128, k)).astype(np.float32)
    b = rng.standard_normal((n, k)).astype(np.float32)
    d = torch.zeros(128, n, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ta, tb = dev(a), dev(b)
    code = lib.ofrl_selftest_umma(C.c_void_p(ta.data_ptr()), C.c_void_p(tb.data_ptr()), C.c_void_p(d.data_ptr()),
                                  n, k, kind, a_mn, b_mn, mn_swap, C.c_void_p(flag.data_ptr()),
                                  C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    torch.cuda.synchronize()
    assert int(flag.item()) == 0, "MMA completion wait gave up"
    return d.cpu().numpy().astype(np.float64), a.astype(np.float64) @ b.astype(np.float64).T, a, b


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("n,k", [(128, 32), (64, 32), (16, 16)])
def test_umma_bf16_both_majors(a_mn, b_mn, n, k):
    _check(BF16, a_mn, b_mn, n, k)


@pytest.mark.parametrize("kind", [TF32, TF32X3])
@pytest.mark.parametrize("n,k", [(128, 32), (64, 32), (16, 16)])
def test_umma_tf32_k_major(kind, n, k):
    _check(kind, 0, 0, n, k)


def test_umma_wrong_mn_assignment_is_detected():
    got, want, a, b = _run(BF16, 64, 32, 1, 1, seed=5, mn_swap=1)
    scale = np.abs(a).astype(np.float64) @ np.abs(b).astype(np.float64).T
    assert (np.abs(got - want) / scale).max() > 0.1


def _check(kind, a_mn, b_mn, n, k):
    got, want, a, b = _run(kind, n, k, a_mn, b_mn, seed=n + k + kind)
    scale = np.abs(a).astype(np.float64) @ np.abs(b).astype(np.float64).T
    err = np.abs(got - want) / scale
    tol = {TF32: 2e-3, TF32X3: 1e-6, BF16: 1.6e-2}[kind]
    assert err.max() < tol, f"max error / sum|terms| = {err.max():.3g}"


@pytest.mark.parametrize("kind,k", [(TF32, 64), (BF16, 64)])
def test_umma_wide_n(kind, k):
    got, want, a, b = _run(kind, 256, k, 0, 0, seed=7)
    scale = np.abs(a).astype(np.float64) @ np.abs(b).astype(np.float64).T
    assert (np.abs(got - want) / scale).max() < {TF32: 2e-3, BF16: 1.6e-2}[kind]
