"""Builds libfa_gb300.so in-tree with nvcc for sm_103a.

The library has one translation unit (``csrc/fa_api.cu``); the ptxas
resource report of the last build is kept in ``_build/ptxas.txt`` at the
repository root.
"""
from __future__ import annotations

import os
import re
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libfa_gb300.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
# the same sources with the device-side invariant checks (FA_DEBUG = 1)
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libfa_gb300_debug.so")
DEBUG_FLAGS = ["-DFA_DEBUG=1"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMPILE_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa_gb300.so")


def _sources():
    deps = [os.path.join(INCLUDE, "fa_gb300.h")]
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            deps.append(os.path.join(CSRC, name))
    return deps


STAMP_PATH = LIB_PATH + ".sha256"


def source_hash(debug: bool = False) -> str:
    """SHA-256 over the library's sources (names and contents), the compile
    command's flags and this machine's architecture: the stamp a built
    library must carry to be reused."""
    import hashlib
    import platform
    h = hashlib.sha256()
    h.update(" ".join(ARCH_FLAGS + COMPILE_FLAGS + (DEBUG_FLAGS if debug else [])).encode())
    h.update(platform.machine().encode())
    for path in _sources():
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode() + b"\0" + f.read())
    return h.hexdigest()


def needs_build(debug: bool = False) -> bool:
    """True unless the library exists and its stamp matches the sources (file
    times are not trusted: a copied tree can carry a library newer than
    sources it was not built from)."""
    lib = DEBUG_LIB_PATH if debug else LIB_PATH
    stamp = lib + ".sha256"
    if not (os.path.exists(lib) and os.path.exists(stamp)):
        return True
    with open(stamp) as f:
        return f.read().strip() != source_hash(debug)


# Registers per thread the attention kernel must launch with, by its last
# template argument (softmax threads per row): its warpgroups re-split this
# budget with setmaxnreg (fa_fwd_kernel.cuh, WarpLayout::kLaunchRegs), and a
# smaller launch budget would leave the increasing warpgroups waiting for
# registers that never come.
KERNEL_LAUNCH_REGS = {1: 168, 2: 96}


def _expected_regs(mangled: str) -> int:
    m = re.search(r"fa_fwd_kernelILi\d+ELb[01]ELi\d+ELi(\d+)(?:ELb[01]|ELi\d+)?EE", mangled)
    if not m:
        raise RuntimeError(f"cannot read the template arguments of {mangled}")
    return KERNEL_LAUNCH_REGS[int(m.group(1))]


def check_launch_registers(ptxas_log: str) -> None:
    """Raise unless every fa_fwd_kernel instantiation launches with the
    register count its setmaxnreg split assumes."""
    current = None
    seen = 0
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current is not None:
            if "fa_fwd_kernel" in current:
                seen += 1
                want = _expected_regs(current)
                if int(m.group(1)) != want:
                    raise RuntimeError(
                        f"{current} uses {m.group(1)} registers per thread, not "
                        f"{want}: its setmaxnreg split would not fit")
            current = None
    if seen == 0:
        raise RuntimeError("no fa_fwd_kernel register report in the ptxas output")


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile the library unless it exists with the stamp of the current
    sources; ``debug`` builds libfa_gb300_debug.so, the same sources with the
    device-side invariant checks (FA_DEBUG = 1)."""
    lib = DEBUG_LIB_PATH if debug else LIB_PATH
    if not force and not needs_build(debug):
        return lib
    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    tmp = lib + ".tmp"
    stamp = source_hash(debug)
    cmd = [_nvcc(), *ARCH_FLAGS, *COMPILE_FLAGS, *(DEBUG_FLAGS if debug else []), "-Xptxas", "-v",
           "-I", INCLUDE, "-o", tmp, os.path.join(CSRC, "fa_api.cu")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(out_dir, "ptxas_debug.txt" if debug else "ptxas.txt"), "w") as f:
        f.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stderr[-4000:]}")
    try:
        check_launch_registers(res.stdout + res.stderr)
    except RuntimeError:
        os.remove(tmp)
        raise
    os.replace(tmp, lib)
    with open(lib + ".sha256", "w") as f:
        f.write(stamp + "\n")
    if verbose:
        print(res.stderr)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
