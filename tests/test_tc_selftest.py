"""tcgen05 building blocks (swizzled fill, smem/instruction descriptors, TMEM loads) on one CTA,
checked against a float32 matmul of the same fp16 operands."""
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
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                        "-Xcompiler", "-fPIC", "-cudart", "shared",
                        "-I", os.path.join(ROOT, "sparse_mla_decode_paged_gb300", "csrc"), src, "-o", out], check=True)
    lib = C.CDLL(out)
    lib.tc_selftest.argtypes = [C.c_int] + [C.c_void_p] * 6
    return lib


def _run(lib, variant):
    g = torch.Generator().manual_seed(7)
    A = torch.randn(128, 576, generator=g).half()
    Q = torch.randn(64, 576, generator=g).half()
    P = torch.rand(128, 64, generator=g).half()
    dA, dQ, dP = A.cuda(), Q.cuda(), P.cuda()
    S = torch.full((128, 64), float("nan"), device="cuda")
    O = torch.full((512, 64), float("nan"), device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = lib.tc_selftest(variant, dA.data_ptr(), dQ.data_ptr(), dP.data_ptr(), S.data_ptr(), O.data_ptr(),
                         st.data_ptr())
    assert rc == 0 and int(st.item()) == 0
    S_ref = A.float() @ Q.float().T
    O_ref = A[:, :512].float().T @ P.float()
    return S.cpu(), O.cpu(), S_ref, O_ref


def test_qk_and_pv_layouts():
    lib = _build()
    S, O, S_ref, O_ref = _run(lib, 0)
    assert torch.allclose(S, S_ref, rtol=1e-4, atol=1e-3), (S - S_ref).abs().max()
    assert torch.allclose(O, O_ref, rtol=1e-4, atol=1e-3), (O - O_ref).abs().max()
