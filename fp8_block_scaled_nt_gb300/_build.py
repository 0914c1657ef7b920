"""Build ``libfp8g.so`` (the C-ABI library) in-tree for sm_103a with nvcc."""
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libfp8g.so")
SOURCES = [os.path.join(CSRC, "fp8g_api.cu")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home():
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home:
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _inputs():
    files = list(SOURCES)
    for d in (CSRC, INCLUDE):
        files += [os.path.join(d, f) for f in os.listdir(d)
                  if f.endswith((".cuh", ".h", ".cu"))]
    return files


def _stale():
    if not os.path.exists(LIB):
        return True
    newest = max(os.path.getmtime(f) for f in _inputs())
    return os.path.getmtime(LIB) < newest


def nvcc_command(out, extra=()):
    home = cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    if not os.path.exists(nvcc):
        nvcc = "nvcc"
    libdir = os.path.join(home, "lib64")
    return ([nvcc] + ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                             "-shared", "-cudart", "shared", "-I", INCLUDE,
                             "-Xlinker", "-rpath," + libdir, "-o", out]
            + list(extra) + SOURCES)


def build(force=False, verbose=False):
    """Compile the library if missing or older than its sources; return its path."""
    if not force and not _stale():
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = nvcc_command(tmp, ["-Xptxas", "-v"] if verbose else [])
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    if verbose:
        print(r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
