"""Build libpa.so in-tree with nvcc for sm_103a.

The library is a handful of translation units compiled in parallel (the decode
kernel instantiations are split by dtype and head_size) and linked into
``paged_kv_cache_136_gb300/_lib/libpa.so``, plus ``_lib/pa_latency``, a host
program that times the C ABI on the 4-sequence workload.  Run ``python
paged_kv_cache_136_gb300/build.py`` or call :func:`build`.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIB_DIR, "libpa.so")
LATENCY_TOOL = os.path.join(LIB_DIR, "pa_latency")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC]

UNITS = [
    ("pa_api", "pa_api.cu", []),
    ("pa_noalloc", "pa_noalloc.cu", []),
    ("pa_decode_f16_d64", "pa_decode_inst.cu", ["-DPA_INST_DTYPE=0", "-DPA_INST_D=64"]),
    ("pa_decode_f16_d128", "pa_decode_inst.cu", ["-DPA_INST_DTYPE=0", "-DPA_INST_D=128"]),
    ("pa_decode_bf16_d64", "pa_decode_inst.cu", ["-DPA_INST_DTYPE=1", "-DPA_INST_D=64"]),
    ("pa_decode_bf16_d128", "pa_decode_inst.cu", ["-DPA_INST_DTYPE=1", "-DPA_INST_D=128"]),
    ("pa_prefill_f16", "pa_prefill_inst.cu", ["-DPA_INST_DTYPE=0"]),
    ("pa_decode_fp8_f16", "pa_decode_fp8_inst.cu", ["-DPA_INST_DTYPE=0"]),
    ("pa_decode_fp8_bf16", "pa_decode_fp8_inst.cu", ["-DPA_INST_DTYPE=1"]),
    ("pa_prefill_bf16", "pa_prefill_inst.cu", ["-DPA_INST_DTYPE=1"]),
]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources() -> list[str]:
    return (glob.glob(os.path.join(CSRC, "*")) + [os.path.join(INCLUDE, "pa.h"),
                                                  os.path.abspath(__file__)])


def _stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(LATENCY_TOOL):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(LATENCY_TOOL))
    return any(os.path.getmtime(s) > t for s in _sources())


def _compile(unit, verbose: bool):
    name, src, defs = unit
    obj = os.path.join(OBJ_DIR, name + ".o")
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {name}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _compile_tool() -> str:
    """Object of the host program that times the C ABI (csrc/pa_latency.cu)."""
    obj = os.path.join(OBJ_DIR, "pa_latency.o")
    cmd = [_nvcc(), *ARCH, "-O2", "-std=c++17", "-I", INCLUDE, "-c",
           os.path.join(CSRC, "pa_latency.cu"), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for pa_latency:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libpa.so if any source changed; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(UNITS) + 1) as ex:
        tool_obj = ex.submit(_compile_tool)
        results = list(ex.map(lambda u: _compile(u, verbose), UNITS))
        tool_obj = tool_obj.result()
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    # The C-ABI latency tool links against the library it measures.
    tmp = LATENCY_TOOL + f".{os.getpid()}.tmp"
    cmd = [_nvcc(), *ARCH, tool_obj, "-L", LIB_DIR, "-lpa", "-Xlinker", "-rpath=$ORIGIN", "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LATENCY_TOOL)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
