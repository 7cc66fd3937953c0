"""Builds libmk.so (the megakernel and its C ABI) in-tree for sm_103a."""
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libmk.so")
SOURCES = ["megakernel.cu", "megakernel_nuc.cu", "plan.cu", "noalloc.cu", "serve.cu"]
HEADERS = [os.path.join(CSRC, "mk_internal.h"), os.path.join(CSRC, "megakernel.cuh"), os.path.join(ROOT, "include", "mk.h")]
NVFLAGS = ["-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
           "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def build(force: bool = False, verbose: bool = False) -> str:
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    newest = max(os.path.getmtime(f) for f in srcs + HEADERS + [__file__])
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    bdir = os.path.join(HERE, "_build")
    os.makedirs(bdir, exist_ok=True)
    objs = [os.path.join(bdir, os.path.splitext(s)[0] + ".o") for s in SOURCES]

    def compile_one(i):
        cmd = ["nvcc", *NVFLAGS, "-c", srcs[i], "-o", objs[i]]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {SOURCES[i]}:\n{r.stderr}")
        return r.stderr

    with ThreadPoolExecutor(len(srcs)) as ex:
        logs = list(ex.map(compile_one, range(len(srcs))))
    if verbose:
        for lg in logs:
            print(lg)
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run(["nvcc", "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", tmp,
                    "-lcudart", "-lpthread"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True)
