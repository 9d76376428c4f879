"""The split kernel's tcgen05 layouts (its own layout header: swizzled K tile and Q, K-major and
MN-major descriptors, P * mant buffers with 128-, 64- and 32-byte swizzle spans, the rope folded
into score buffer 0, TMEM loads of 16 and 32 columns) on one CTA per head-group size, checked against
a float64 matmul of the same fp16 operands."""
import ctypes as C
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "sparse_mla_decode_paged_gb300", "csrc")


def _build():
    out = os.path.join(ROOT, "_build", "tc_selftest.so")
    src = os.path.join(HERE, "cuda", "tc_selftest.cu")
    deps = [src] + [os.path.join(CSRC, h) for h in ("smla_ptx.cuh", "smla_split_layout.cuh")]
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not os.path.exists(out) or os.path.getmtime(out) < max(os.path.getmtime(d) for d in deps):
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                        "-Xcompiler", "-fPIC", "-cudart", "shared", "-I", CSRC, src, "-o", out], check=True)
    lib = C.CDLL(out)
    lib.tc_selftest.argtypes = [C.c_int] + [C.c_void_p] * 6
    return lib


@pytest.mark.parametrize("nh", [16, 32, 64])
def test_qk_and_pv_layouts_of_the_split_kernel(nh):
    lib = _build()
    g = torch.Generator().manual_seed(7 + nh)
    K = torch.randn(128, 576, generator=g).half()
    Q = torch.randn(nh, 576, generator=g).half()
    Pm = torch.rand(4, 128, nh, generator=g).half()
    S = torch.full((4, 128, nh), float("nan"), device="cuda")
    O = torch.full((512, nh), float("nan"), device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    d = [x.cuda().contiguous() for x in (K, Q, Pm)]
    rc = lib.tc_selftest(nh, *[x.data_ptr() for x in d], S.data_ptr(), O.data_ptr(), st.data_ptr())
    assert rc == 0 and int(st.item()) == 0
    S, O = S.cpu().double(), O.cpu().double()
    Kd, Qd, Pd = (x.double() for x in (K, Q, Pm))
    for b in range(4):
        ref = Kd[:, 128 * b:128 * b + 128] @ Qd[:, 128 * b:128 * b + 128].T
        if b == 0:
            ref = ref + Kd[:, 512:] @ Qd[:, 512:].T           # the rope accumulates into block 0
        assert torch.allclose(S[b], ref, rtol=1e-5, atol=1e-4), (b, (S[b] - ref).abs().max())
        o_ref = Kd[:, 128 * b:128 * b + 128].T @ Pd[b]
        assert torch.allclose(O[128 * b:128 * b + 128], o_ref, rtol=1e-5, atol=1e-4), \
            (b, (O[128 * b:128 * b + 128] - o_ref).abs().max())
