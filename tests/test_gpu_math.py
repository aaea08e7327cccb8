"""The FMA-pipe reciprocal used by the prefill's SiLU and gate sigmoids, checked on the
GPU against the correctly rounded reciprocal over its whole input range [1, 2^126]."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    out = tmp_path_factory.mktemp("math") / "libmath_test.so"
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", os.path.join(HERE, "cuda", "math_test.cu"), "-o", str(out)], check=True)
    L = ctypes.CDLL(str(out))
    L.rcp_newton_test.restype = ctypes.c_int
    L.rcp_newton_test.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    return L


def test_rcp_newton_within_two_ulp(lib):
    rng = np.random.default_rng(7)
    mant = np.linspace(1.0, 2.0, 1 << 16, endpoint=False)  # every exponent's mantissa range, densely
    x = np.concatenate([np.exp2(rng.uniform(0.0, 126.0, 1 << 20)),
                        mant, mant * 2.0 ** 60, mant * 2.0 ** 125,
                        np.exp2(np.arange(0, 127)), [1.0, 1.5, 1.9999999, 2.0 ** 126]]).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    y = torch.empty_like(xd)
    assert lib.rcp_newton_test(xd.data_ptr(), y.data_ptr(), x.size, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    exact = 1.0 / x.astype(np.float64)
    ulp = np.spacing(exact.astype(np.float32)).astype(np.float64)
    err_ulp = np.abs(got - exact) / ulp
    cuda_div = (1.0 / xd).cpu().numpy().astype(np.float64)  # the IEEE division of the CUDA toolchain
    print(f"rcp_newton: max error {err_ulp.max():.2f} ulp over {x.size} inputs; "
          f"max |diff| to CUDA 1/x {np.max(np.abs(got - cuda_div) / ulp):.2f} ulp")
    assert err_ulp.max() <= 2.0
