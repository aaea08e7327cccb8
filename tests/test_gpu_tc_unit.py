"""Unit test of the tcgen05 building blocks (descriptors, MMA, commit, TMEM load
and store) on small GEMMs against torch's matmul of the same BF16 operands."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    out = tmp_path_factory.mktemp("tc") / "libtc_gemm_test.so"
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", os.path.join(HERE, "cuda", "tc_gemm_test.cu"), "-o", str(out)],
                   check=True)
    L = ctypes.CDLL(str(out))
    L.tc_gemm_test.restype = ctypes.c_int
    L.tc_gemm_test.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                                        ctypes.c_void_p]
    L.tc_gemm_ta_test.restype = ctypes.c_int
    L.tc_gemm_ta_test.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    return L


@pytest.mark.parametrize("N,K,pad", [(64, 128, 0), (128, 64, 0), (64, 64, 0), (128, 128, 0), (192, 64, 0),
                                     (128, 128, 1), (64, 128, 1)])
def test_tc_gemm_matches_torch(lib, N, K, pad):
    torch.manual_seed(N + K)
    A = torch.randn(128, K, device="cuda").to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda").to(torch.bfloat16)
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.tc_gemm_test(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, K, pad, status.data_ptr(),
                          torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and int(status.item()) == 0
    ref = 3.0 * (A.double() @ B.double().T)
    err = (D.double() - ref).abs().max().item() / ref.abs().max().item()
    print(f"tcgen05 GEMM 128x{N}x{K} ({'padded' if pad else 'dense'} layout): rel err {err:.2e}")
    assert err < 1e-5


@pytest.mark.parametrize("N,K", [(64, 128), (128, 128), (192, 64), (128, 64)])
def test_tc_gemm_tmem_a_matches_torch(lib, N, K):
    """A operand in tensor memory (BF16 pairs per column, one row per lane)."""
    torch.manual_seed(7 * N + K)
    A = torch.randn(128, K, device="cuda").to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda").to(torch.bfloat16)
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.tc_gemm_ta_test(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, K, status.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and int(status.item()) == 0
    ref = A.double() @ B.double().T
    err = (D.double() - ref).abs().max().item() / ref.abs().max().item()
    print(f"tcgen05 GEMM 128x{N}x{K}, A in tensor memory: rel err {err:.2e}")
    assert err < 1e-5
