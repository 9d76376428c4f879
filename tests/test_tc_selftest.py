"""tcgen05 building blocks (swizzled fill, K-major and MN-major descriptors, A operand from TMEM,
TMEM loads and stores) on one CTA, checked against a float32 matmul of the same fp16 operands."""
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
    lib.tc_selftest.argtypes = [C.c_void_p] * 7
    return lib


def test_qk_correction_and_pv_layouts():
    lib = _build()
    g = torch.Generator().manual_seed(7)
    A = torch.randn(128, 576, generator=g).half()
    Q = torch.randn(64, 576, generator=g).half()
    L = (torch.randn(128, 512, generator=g) * 1e-3).half()
    P = torch.rand(128, 64, generator=g).half()
    S = torch.full((128, 64), float("nan"), device="cuda")
    O = torch.full((512, 64), float("nan"), device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    d = [x.cuda() for x in (A, Q, L, P)]
    rc = lib.tc_selftest(*[x.data_ptr() for x in d], S.data_ptr(), O.data_ptr(), st.data_ptr())
    assert rc == 0 and int(st.item()) == 0
    S, O = S.cpu().double(), O.cpu().double()
    Ad, Qd, Ld, Pd = (x.double() for x in (A, Q, L, P))
    S_ref = Ad @ Qd.T + Ld @ Qd[:, :512].T
    assert torch.allclose(S, S_ref, rtol=1e-5, atol=1e-4), (S - S_ref).abs().max()
    O_ref = Ad[:, :512].T @ Pd
    assert torch.allclose(O, O_ref, rtol=1e-5, atol=1e-4), (O - O_ref).abs().max()
