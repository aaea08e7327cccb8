"""Failure detection without a GPU fault: a device-side wait that nothing satisfies gives
up after its iteration limit, records KDA_ERR_TIMEOUT in the error word the host reads,
and returns, leaving the context usable. The kernel (tests/cuda/wait_timeout_test.cu) uses
the library's own bounded mbarrier wait; the limit here is small (2^14 polls), so the test
takes milliseconds and cannot hang the GPU."""
import ctypes
import os
import subprocess

import pytest
import torch

import linear_attention_mixer_gb300 as K

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    out = tmp_path_factory.mktemp("wait") / "libwait_timeout_test.so"
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", os.path.join(HERE, "cuda", "wait_timeout_test.cu"), "-o", str(out)],
                   check=True)
    L = ctypes.CDLL(str(out))
    L.wait_timeout_test.restype = ctypes.c_int
    L.wait_timeout_test.argtypes = [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    return L


@pytest.mark.parametrize("arrive", [0, 1])
def test_unsatisfied_wait_times_out_and_reports(lib, arrive):
    limit = 1 << 14
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    polls = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.wait_timeout_test(err.data_ptr(), limit, arrive, polls.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()  # returns: the kernel ended by itself
    assert rc == 0
    if arrive:
        assert int(err.item()) == K.KDA_OK and 1 <= int(polls.item()) < limit
    else:
        assert int(err.item()) == K.KDA_ERR_TIMEOUT and int(polls.item()) == limit
    # the context is still usable: a library call and a torch kernel both run
    cfg = K.kda_config(2, 128, K.KDA_F32)
    st = K.kda_state_alloc(cfg, 1)
    try:
        K.kda_state_reset(st, [0])
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    assert float((torch.ones(1024, device="cuda") * 2).sum().item()) == 2048.0
