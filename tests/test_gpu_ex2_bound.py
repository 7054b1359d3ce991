"""The online-softmax filter assumes |ex2.approx(x) / 2^x - 1| <= 2^-21 for
x in [-126, 0]; measure the special-function unit's actual error on the GPU
(against double-precision exp2) and require a 2x margin below that bound."""

import ctypes
import os
import subprocess

import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytestmark = pytest.mark.skip("needs a GPU")
else:
    pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_ex2_relative_error_within_bound(tmp_path):
    so = str(tmp_path / "ex2_check.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                    "-Xcompiler", "-fPIC", "-o", so, os.path.join(HERE, "cuda", "ex2_check.cu")],
                   check=True)
    lib = ctypes.CDLL(so)
    lib.ex2_max_rel_err.argtypes = [ctypes.c_ulonglong, ctypes.POINTER(ctypes.c_double)]
    out = ctypes.c_double()
    assert lib.ex2_max_rel_err(1 << 25, ctypes.byref(out)) == 0
    print(f"max relative error of ex2.approx.ftz.f32: {out.value:.3e} (2^{__import__('math').log2(out.value):.2f})")
    assert out.value <= 2.0 ** -22
