"""The online-softmax filter assumes |ex2.approx(x) / 2^x - 1| <= 2^-21 for
x in [-126, 0]; measure the special-function unit's error on the GPU against
double-precision exp2 on every f32 argument of that range (about 1.1e9 of
them), and require a 2x margin below the assumed bound."""

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
    lib.ex2_max_rel_err.argtypes = [ctypes.POINTER(ctypes.c_double)]
    out = (ctypes.c_double * 3)()
    assert lib.ex2_max_rel_err(out) == 0
    worst, arg, count = out[0], out[1], out[2]
    assert count == 0xC2FC0000 - 0x80000000 + 2  # every f32 in [-126, 0], both zeros
    print(f"max relative error of ex2.approx.ftz.f32 over {count:.0f} arguments: {worst:.3e} "
          f"(2^{__import__('math').log2(worst):.2f}) at x = {arg!r}")
    assert 0 < worst <= 2.0 ** -22
