"""Build the C-ABI shared library (libfr_gb300.so) in-tree for sm_103a.

Each .cu under csrc/ compiles to an object in parallel, then the objects link
into gqa_kv_head_gb300/_build/libfr_gb300.so. The CUDA runtime is linked
statically, so the library loads on a machine without a GPU driver (the
driver is needed only once a CUDA call is made).
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB_NAME = "libfr_gb300.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# host code: no floating-point contraction, so host-side fp32 steps give the
# same bits on every host architecture
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-Xcompiler", "-ffp-contract=off",
         "--expt-relaxed-constexpr"]


TRACE_BUILD = os.path.join(HERE, "_build_trace")


def library_path(trace=False):
    return os.path.join(TRACE_BUILD if trace else BUILD, LIB_NAME)


def _nvcc():
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return p


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def is_stale(trace=False):
    lib = library_path(trace)
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in _deps())


def build(force=False, verbose=False, ptxas_verbose=False, trace=False):
    """Compile and link if any source is newer than the library. Returns its path.
    trace=True builds the timeline-instrumented variant (FR_TRACE) into its own
    directory; the library itself never has it."""
    if not force and not is_stale(trace):
        return library_path(trace)
    out_dir = TRACE_BUILD if trace else BUILD
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if trace:
        extra = extra + ["-DFR_TRACE"]

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, _sources()))
    objs = [o for o, _ in results]
    if verbose or ptxas_verbose:
        for _, log in results:
            if log:
                print(log)
    tmp = library_path(trace) + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, library_path(trace))
    return library_path(trace)


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
