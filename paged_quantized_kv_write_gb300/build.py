"""Build libpagedkv.so (the CUDA kernels and the C ABI) in-tree with nvcc.

Targets sm_103a only.  Translation units compile in parallel, then link into
paged_quantized_kv_write_gb300/_lib/libpagedkv.so.  The CUDA runtime is
linked statically, so the library needs only the driver at run time.

A second library, _lib/libpagedkv_test.so, is the test build: the same
sources compiled with PKV_TEST_HOOKS, plus the two comparators the product
never selects (the CUDA-core decode in pkv_simt.cu and the tcgen05 decode in
pkv_decode_tc.cu, chosen there with PKV_DECODE_MODE=simt|tc) and the switch
that drops one tensor-core commit to exercise the bounded waits
(PKV_TEST_DROP_COMMIT).  Only the tests load it.

    python paged_quantized_kv_write_gb300/build.py [--force] [--verbose-ptxas] [--product-only]

(run it by path: importing the package itself needs the built library)
"""

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
OBJ_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpagedkv.so")
TEST_LIB = os.path.join(OUT_DIR, "libpagedkv_test.so")
# comparators: compiled into the test build only
COMPARATORS = ("pkv_simt.cu", "pkv_decode_tc.cu")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xcompiler", "-Wall", f"-I{INCLUDE}"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedkv.so")
    return cand


def sources(test: bool = False):
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith(".cu") and (test or f not in COMPARATORS))


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "pagedkv.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale(target: str) -> bool:
    if not os.path.exists(target) or os.environ.get("PKV_NVCC_EXTRA"):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose_ptxas: bool = False, test: bool = True) -> str:
    """Build the product library and (test=True) the test library; return the
    product library's path."""
    targets = [(LIB, False)] + ([(TEST_LIB, True)] if test else [])
    todo = [(lib, t) for lib, t in targets if force or _stale(lib)]
    if not todo:
        return LIB
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    # tuning hook: extra nvcc flags (e.g. -DPKV_STAGES_FP8=6) from the environment
    extra += os.environ.get("PKV_NVCC_EXTRA", "").split()

    def compile_one(job):
        src, t = job
        obj_dir = os.path.join(OBJ_DIR, "test" if t else "product")
        os.makedirs(obj_dir, exist_ok=True)
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        defs = ["-DPKV_TEST_HOOKS"] if t else []
        cmd = [nvcc, *ARCH, *FLAGS, *defs, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    jobs = [(src, t) for _, t in todo for src in sources(t)]
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        results = dict(zip(jobs, ex.map(compile_one, jobs)))
    if verbose_ptxas:
        for job, (_, log) in results.items():
            if not job[1]:
                sys.stdout.write(log)
    for lib, t in todo:
        tmp = lib + f".tmp{os.getpid()}"
        objs = [results[(src, t)][0] for src in sources(t)]
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="--verbose-ptxas" in sys.argv,
                test="--product-only" not in sys.argv))
