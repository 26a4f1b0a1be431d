"""Tensor-core building blocks on the GPU (tcgen05 MMA with A in shared memory
or in TMEM, the 128-byte-swizzled K-major operand layout, fp16 and bf16, TMEM
load/store, bounded mbarrier waits, 1-D bulk copies) against torch."""
import ctypes
import os
import subprocess

import pytest
import torch

from linear_attention_recurrence_prefill_gb300 import build as libbuild

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "umma_selftest.cu")
OUT = os.path.join(HERE, "_build", "libumma_selftest.so")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    deps = [SRC, os.path.join(libbuild.CSRC, "umma.cuh")]
    if not os.path.exists(OUT) or any(os.path.getmtime(d) > os.path.getmtime(OUT) for d in deps):
        cmd = [libbuild.nvcc(), *libbuild.flags(), "-shared", "-cudart", "shared", SRC, "-o", OUT]
        subprocess.run(cmd, check=True)
    l = ctypes.CDLL(OUT)
    vp, ci = ctypes.c_void_p, ctypes.c_int
    l.selftest_mma.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, ci]
    l.selftest_mma.restype = ci
    l.selftest_bulk.argtypes = [vp, vp, ctypes.POINTER(ci), ci]
    l.selftest_bulk.restype = ci
    return l


@pytest.mark.parametrize("a_in_tmem", [0, 1], ids=["A_smem", "A_tmem"])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("N,K", [(16, 128), (64, 64), (64, 128), (128, 128), (32, 64)])
def test_mma(lib, a_in_tmem, dtype, N, K):
    g = torch.Generator(device="cuda").manual_seed(N * 1000 + K)
    A = torch.randn((128, K), generator=g, device="cuda").to(dtype)
    B = torch.randn((N, K), generator=g, device="cuda").to(dtype)
    D = torch.full((128, N), float("nan"), device="cuda")
    rc = lib.selftest_mma(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, K,
                          int(dtype == torch.bfloat16), a_in_tmem, 0, 0)
    assert rc == 0, f"selftest_mma returned {rc}"
    ref = A.double() @ B.double().T
    err = (D.double() - ref).abs().max().item()
    assert err < 1e-3 * max(1.0, ref.abs().max().item()), f"max abs error {err}"


@pytest.mark.parametrize("a_mn,b_mn", [(1, 0), (0, 1), (1, 1)], ids=["A_mn", "B_mn", "AB_mn"])
@pytest.mark.parametrize("N,K", [(64, 64), (128, 64), (128, 128), (64, 128)])
def test_mma_mn_major(lib, a_mn, b_mn, N, K):
    """MN-major operands (the layout the prefill uses for V, K~ and K^)."""
    g = torch.Generator(device="cuda").manual_seed(7 * N + K + 10 * a_mn + 20 * b_mn)
    A = torch.randn((128, K), generator=g, device="cuda").half()
    B = torch.randn((N, K), generator=g, device="cuda").half()
    D = torch.full((128, N), float("nan"), device="cuda")
    rc = lib.selftest_mma(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, K, 0, 0, a_mn, b_mn)
    assert rc == 0, f"selftest_mma returned {rc}"
    ref = A.double() @ B.double().T
    err = (D.double() - ref).abs().max().item()
    assert err < 1e-3 * max(1.0, ref.abs().max().item()), f"max abs error {err}"


def test_bulk_copy_round_trip(lib):
    sizes = [16384, 16384, 16384, 16384, 8192, 512]
    total = sum(sizes)
    src = torch.randint(0, 255, (total,), dtype=torch.uint8, device="cuda")
    dst = torch.zeros_like(src)
    arr = (ctypes.c_int * len(sizes))(*sizes)
    rc = lib.selftest_bulk(src.data_ptr(), dst.data_ptr(), arr, len(sizes))
    assert rc == 0
    assert torch.equal(src, dst)
