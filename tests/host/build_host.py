"""Builds the cache's host planner against a host-memory stand-in for the
CUDA runtime (``fake_cuda.cpp``), with g++ and no GPU, into
``tests/host/_build/libakv_host.so``.  Test infrastructure: only the
planner's host state is meaningful in this build (no kernel runs)."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
CSRC = os.path.join(ROOT, "agent_kv_cache_gb300", "csrc")
OUT = os.path.join(HERE, "_build", "libakv_host.so")
SOURCES = [os.path.join(CSRC, "akv_host.cpp"), os.path.join(CSRC, "akv_prefix.cpp"),
           os.path.join(HERE, "fake_cuda.cpp")]


def build():
    deps = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".h")]
    deps.append(os.path.join(ROOT, "include", "akv.h"))
    if os.path.exists(OUT) and all(os.path.getmtime(d) <= os.path.getmtime(OUT) for d in deps):
        return OUT
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    # -Bsymbolic: the planner's CUDA calls bind to the stand-in even in a
    # process that has loaded the real runtime
    cmd = ["g++", "-std=c++17", "-O1", "-g", "-fPIC", "-shared", "-Wl,--no-undefined",
           "-Wl,-Bsymbolic",
           "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-I", os.path.join(cuda, "include"),
           *SOURCES, "-o", OUT + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:
        raise RuntimeError("host-only build failed:\n" + r.stdout + r.stderr)
    os.replace(OUT + ".tmp", OUT)
    return OUT


if __name__ == "__main__":
    print(build())
