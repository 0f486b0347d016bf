"""In-tree build of the native libraries with nvcc for sm_103a.

* ``tensor_transformer_forward_gb300/_lib/libtpfwd.so`` -- the C-ABI library
  (``include/tpfwd.h``) and its kernels.
* ``synth/_lib/libtpsynth.so`` -- the device half of the seeded input
  generator (``synth/csrc/synth_fill.cu``).

Translation units compile in parallel; a library is rebuilt when any of its
sources or headers is newer than it.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
from typing import List

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libtpfwd.so")
SYNTH_DIR = os.path.join(ROOT, "synth")
SYNTH_LIB_PATH = os.path.join(SYNTH_DIR, "_lib", "libtpsynth.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build tpfwd")


def _sources(d: str, exts=(".cu",)) -> List[str]:
    return sorted(os.path.join(d, f) for f in os.listdir(d) if f.endswith(exts))


def _stale(target: str, deps: List[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(p) > t for p in deps)


def _compile(src: str, obj: str, extra: List[str]) -> None:
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")


def _build_lib(srcs: List[str], headers: List[str], out: str, obj_dir: str, extra: List[str],
               verbose: bool) -> str:
    if not _stale(out, srcs + headers):
        return out
    os.makedirs(obj_dir, exist_ok=True)
    os.makedirs(os.path.dirname(out), exist_ok=True)
    objs = [os.path.join(obj_dir, os.path.basename(s) + ".o") for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        list(ex.map(lambda so: _compile(so[0], so[1], extra), zip(srcs, objs)))
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed for {os.path.basename(out)}:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, out)
    if verbose:
        print(f"built {out}")
    return out


def build(verbose: bool = False) -> List[str]:
    headers = _sources(CSRC, (".cuh", ".h")) + [os.path.join(ROOT, "include", "tpfwd.h")]
    lib = _build_lib(_sources(CSRC), headers, LIB_PATH, os.path.join(LIB_DIR, "obj"),
                     ["-I", os.path.join(ROOT, "include")], verbose)
    synth_src = _sources(os.path.join(SYNTH_DIR, "csrc"))
    slib = _build_lib(synth_src, [], SYNTH_LIB_PATH, os.path.join(SYNTH_DIR, "_lib", "obj"), [], verbose)
    return [lib, slib]


if __name__ == "__main__":
    build(verbose=True)
