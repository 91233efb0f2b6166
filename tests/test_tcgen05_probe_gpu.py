"""tcgen05 / TMEM helper check: a one-CTA bf16 GEMM through the library's descriptor and
instruction encodings (tests/cuda/umma_probe.cu) equals an fp32 matmul of the same values."""
import ctypes
import os
import subprocess

import pytest
import torch

from gated_deltanet_linear_rule_gb300 import build

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe():
    src = os.path.join(HERE, "cuda", "umma_probe.cu")
    out_dir = os.path.join(HERE, "cuda", "_build")
    os.makedirs(out_dir, exist_ok=True)
    lib = os.path.join(out_dir, "libumma_probe.so")
    cmd = [build.nvcc(), *build.ARCH, "-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I", build.INCLUDE,
           "-I", build.CSRC, src, "-o", lib]
    subprocess.run(cmd, check=True, capture_output=True)
    L = ctypes.CDLL(lib)
    L.umma_probe_gemm.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_void_p]
    return L


CASES = [(64, 64, 0, 0), (64, 128, 0, 0), (128, 128, 0, 0), (256, 64, 0, 0), (256, 128, 0, 0),
         (128, 64, 0, 1), (128, 128, 0, 1), (64, 64, 0, 1), (128, 64, 1, 0), (128, 64, 1, 1), (128, 128, 1, 1)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("N,K,a_mn,b_mn", CASES)
def test_umma_gemm_matches_fp32_matmul(probe, N, K, a_mn, b_mn, dtype):
    """a_mn / b_mn: the operand is staged MN-major (transposed) and the MMA told so."""
    g = torch.Generator(device="cuda").manual_seed(N * 1000 + K)
    A = torch.randn((128, K), device="cuda", generator=g).to(dtype)
    B = torch.randn((N, K), device="cuda", generator=g).to(dtype)
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    half = 1 if dtype == torch.float16 else 0
    assert probe.umma_probe_gemm(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, K, half, a_mn, b_mn,
                                 status.data_ptr(), s) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "the MMA completion wait timed out"
    ref = A.float() @ B.float().T
    err = (D - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, f"tcgen05 GEMM N={N} K={K} a_mn={a_mn} b_mn={b_mn}: relative error {err:.3e}"
