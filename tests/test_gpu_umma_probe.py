"""tcgen05 operand layouts: each (A, B) K-major / MN-major combination the
tensor-core forward uses, with its descriptors, against a host matmul of the
same BF16 values."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe():
    src = os.path.join(HERE, "cuda", "umma_probe.cu")
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libumma_probe.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-shared", "-Xcompiler", "-fPIC", src, "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.umma_probe.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p] * 3
    lib.umma_probe.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("N,K,a_mn,b_mn,neg", [
    (64, 128, 0, 0, 0),    # [K;Q] K^T and S Q^T
    (64, 64, 1, 0, 0),     # K^T T''^T, V^T T'^T
    (64, 128, 0, 1, 1),    # -S W^T
    (128, 64, 0, 1, 0),    # (Delta^T diag(dec)) K
    (64, 64, 0, 0, 0),     # Delta^T Ahat^T
    (128, 128, 1, 1, 0),
])
def test_umma_layouts(probe, N, K, a_mn, b_mn, neg):
    g = torch.Generator().manual_seed(N + K + a_mn * 2 + b_mn)
    A = torch.randn(128, K, generator=g).bfloat16()
    B = torch.randn(K, N, generator=g).bfloat16()
    Ad, Bd = A.cuda(), B.cuda()
    Dd = torch.zeros(128, N, device="cuda")
    rc = probe.umma_probe(N, K, a_mn, b_mn, neg, Ad.data_ptr(), Bd.data_ptr(), Dd.data_ptr())
    assert rc == 0
    ref = (A.double() @ B.double()) * (-1 if neg else 1)
    err = (Dd.cpu().double() - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, err


@pytest.mark.parametrize("nthreads", [128, 256])
@pytest.mark.parametrize("inplace", [0, 1])
def test_solve64_tc(probe, nthreads, inplace):
    """(I + A)^{-1} of a chunk-like strictly lower A: diagonal blocks in FP32,
    block merges on TF32 tensor cores -> relative error well under BF16's."""
    probe.solve_probe.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    g = torch.Generator().manual_seed(nthreads)
    k = torch.nn.functional.normalize(torch.randn(64, 128, generator=g), dim=-1).double()
    beta = torch.sigmoid(torch.randn(64, generator=g)).double()
    gam = torch.cumsum(-torch.nn.functional.softplus(torch.randn(64, generator=g)), 0).double()
    A = torch.tril(beta[:, None] * torch.exp(gam[:, None] - gam[None, :]).clamp(max=1) * (k @ k.T), -1)
    Td = torch.zeros(64, 64, device="cuda")
    Ad = A.float().cuda()
    assert probe.solve_probe(Ad.data_ptr(), Td.data_ptr(), nthreads, inplace) == 0
    ref = torch.linalg.inv(torch.eye(64, dtype=torch.float64) + A)
    err = (Td.cpu().double() - ref).abs().max().item() / ref.abs().max().item()
    assert err < 2e-3, err
    assert torch.equal(torch.triu(Td.cpu(), 1), torch.zeros(64, 64))


@pytest.mark.parametrize("N,K,b_mn,neg", [
    (64, 128, 1, 1),     # -S W^T with S (BF16) in TMEM
    (64, 128, 0, 0),     # S Qg^T with S in TMEM
    (128, 64, 1, 0),     # (Delta^T diag(dec)) K with Delta^T in TMEM
    (64, 64, 0, 0),      # Delta^T Ahat^T with Delta^T in TMEM
])
def test_umma_a_from_tmem(probe, N, K, b_mn, neg):
    probe.umma_probe_ta.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p] * 3
    g = torch.Generator().manual_seed(7 * N + K + b_mn)
    A = torch.randn(128, K, generator=g).bfloat16()
    B = torch.randn(K, N, generator=g).bfloat16()
    Ad, Bd = A.cuda(), B.cuda()      # keep the device copies alive during the call
    Dd = torch.zeros(128, N, device="cuda")
    rc = probe.umma_probe_ta(N, K, b_mn, neg, Ad.data_ptr(), Bd.data_ptr(), Dd.data_ptr())
    assert rc == 0
    ref = (A.double() @ B.double()) * (-1 if neg else 1)
    err = (Dd.cpu().double() - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, err
