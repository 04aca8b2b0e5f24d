"""Build the synthetic-input fill libraries in place (host: gcc, device: nvcc)."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def _stale(out, srcs):
    return not os.path.exists(out) or any(
        os.path.getmtime(s) > os.path.getmtime(out) for s in srcs)


def build_host(force=False):
    out = os.path.join(HERE, "libsynth_host.so")
    srcs = [os.path.join(HERE, f) for f in ("synth_host.c", "synth.h", "synth_recipe.h")]
    if force or _stale(out, srcs):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-o", out, srcs[0]])
    return out


def build_device(force=False):
    out = os.path.join(HERE, "libsynth_dev.so")
    srcs = [os.path.join(HERE, f) for f in ("synth_dev.cu", "synth.h", "synth_recipe.h")]
    if force or _stale(out, srcs):
        subprocess.check_call([NVCC, "-O2", "-std=c++17", "-gencode",
                               "arch=compute_103a,code=sm_103a", "-fmad=false", "-shared",
                               "-Xcompiler", "-fPIC", "-o", out, srcs[0]])
    return out


def build(force=False):
    return build_host(force), build_device(force)


if __name__ == "__main__":
    print(build(force=True))
