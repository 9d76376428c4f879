"""tcgen05 building blocks (swizzled fill, K-major and MN-major descriptors, per-block
accumulators, TMEM loads) on one CTA, checked against a float32 matmul of the same fp16 operands."""
import ctypes as C
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _build():
    out = os.path.join(ROOT, "_build", "tc_selftest.so")
    src = os.path.join(HERE, "cuda", "tc_selftest.cu")
    hdr = os.path.join(ROOT, "sparse_mla_decode_paged_gb300", "csrc", "smla_ptx.cuh")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not os.path.exists(out) or os.path.getmtime(out) < max(os.path.getmtime(src), os.path.getmtime(hdr)):
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                        "-Xcompiler", "-fPIC", "-cudart", "shared",
                        "-I", os.path.dirname(hdr), src, "-o", out], check=True)
    lib = C.CDLL(out)
    lib.tc_selftest.argtypes = [C.c_void_p] * 6
    return lib


def test_qk_blocks_and_pv_layouts():
    lib = _build()
    g = torch.Generator().manual_seed(7)
    A = torch.randn(128, 576, generator=g).half()
    Q = torch.randn(32, 576, generator=g).half()
    P = torch.rand(4, 128, 32, generator=g).half()
    S = torch.full((5, 128, 32), float("nan"), device="cuda")
    O = torch.full((512, 32), float("nan"), device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    dA, dQ, dP = A.cuda(), Q.cuda(), P.cuda()
    rc = lib.tc_selftest(dA.data_ptr(), dQ.data_ptr(), dP.data_ptr(), S.data_ptr(), O.data_ptr(), st.data_ptr())
    assert rc == 0 and int(st.item()) == 0
    S, O = S.cpu(), O.cpu()
    Af, Qf = A.float(), Q.float()
    for b in range(4):
        ref = Af[:, 128 * b:128 * b + 128] @ Qf[:, 128 * b:128 * b + 128].T
        assert torch.allclose(S[b], ref, rtol=1e-4, atol=1e-3), (b, (S[b] - ref).abs().max())
    ref = Af[:, 512:] @ Qf[:, 512:].T
    assert torch.allclose(S[4], ref, rtol=1e-4, atol=1e-3), (S[4] - ref).abs().max()
    for j in range(4):
        ref = Af[:, 128 * j:128 * j + 128].T @ P[j].float()
        assert torch.allclose(O[128 * j:128 * j + 128], ref, rtol=1e-4, atol=1e-3), (j, (O[128 * j:128 * j + 128] - ref).abs().max())
