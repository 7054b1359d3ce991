"""Build libsv.so in-tree with nvcc for sm_103a (no cmake; the verify, gate and filter translation units)."""

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG_DIR, "csrc")
LIB_DIR = os.path.join(PKG_DIR, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libsv.so")
SOURCES = [os.path.join(CSRC, f) for f in ("sv_api.cu", "sv_gate.cu", "sv_filter.cu", "sv_lm_head.cu", "sv_static.cu", "sv_penalties.cu", "sv_rows.cu")]
HEADERS = [os.path.join(CSRC, f) for f in ("sv_kernel.cuh", "sv_verify.cuh", "sv_rows.cuh", "sv_topk.cuh", "sv_ptx.cuh", "sv_host.h")] + [
    os.path.join(os.path.dirname(PKG_DIR), "include", h) for h in ("sv.h", "sv_gate.h", "sv_filter.h", "sv_lm_head.h", "sv_penalties.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc_path():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or add /usr/local/cuda/bin to PATH)")


def _stale():
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in SOURCES + HEADERS)


def build(force=False, verbose=False):
    """Compile the library if it is missing or older than its sources: one
    nvcc process per translation unit in parallel, then one link."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    nvcc = nvcc_path()
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(LIB_DIR, os.path.splitext(os.path.basename(src))[0] + ".o")
        cmd = [nvcc, *NVCC_FLAGS[:-1], "-c", "-o", obj, src]  # no -shared for the objects
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        objs.append(obj)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)))
    logs = []
    failed = []
    for src, pr in procs:
        out, err = pr.communicate()
        logs.append(out + err)
        if pr.returncode != 0:
            failed.append(f"{src}:\n{out}{err}")
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = LIB_PATH + ".tmp"
    res = subprocess.run([nvcc, *NVCC_FLAGS, "-o", tmp, *objs], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc link failed:\n" + res.stdout + res.stderr)
    os.replace(tmp, LIB_PATH)
    for obj in objs:
        os.remove(obj)
    if verbose:
        print("".join(logs) + res.stdout + res.stderr)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
