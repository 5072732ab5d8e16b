"""Build libskattn.so in-tree: nvcc for sm_103a (tcgen05/TMA kernels and the C
ABI), g++ for the host scheduler.  Translation units compile in parallel."""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libskattn.so")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_SOURCES = ["api.cu", "fwd_decode.cu", "fwd_prefill.cu", "fwd_prefill_persistent.cu", "fwd_latent.cu", "combine.cu",
              "noalloc.cu", "linear_attn.cu", "linear_attn_tc.cu"]
CXX_SOURCES = ["plan.cpp"]


def _nvcc():
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda_home, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _sources_mtime():
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n%s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit and link libskattn.so; returns its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _sources_mtime():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-I" + INCLUDE, "-I" + CSRC]
    jobs = []
    for src in CU_SOURCES:
        obj = os.path.join(OUT_DIR, src + ".o")
        jobs.append(([nvcc] + ARCH + common + ["-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
                                               "-c", os.path.join(CSRC, src), "-o", obj], obj))
    for src in CXX_SOURCES:
        obj = os.path.join(OUT_DIR, src + ".o")
        jobs.append((["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-I" + INCLUDE, "-I" + CSRC, "-c",
                      os.path.join(CSRC, src), "-o", obj], obj))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
        logs = list(ex.map(lambda j: _run(j[0]), jobs))
    with open(os.path.join(OUT_DIR, "ptxas.log"), "w") as f:
        f.write("\n".join(logs))
    if verbose:
        print("\n".join(logs))
    tmp = LIB + ".tmp%d" % os.getpid()
    _run([nvcc] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", tmp] + [o for _, o in jobs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
