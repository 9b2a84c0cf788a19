"""Build the CUDA executor library (libcmdexec.so) in-tree.

Each executor source compiles once per tier and op-set variant
(CMDX_TIER, CMDX_EXT; the tile executor also per view variant, CMDX_ND):
the per-tier interpreters are large, so this spreads them over parallel
compiler processes. With the host sources, all compile in parallel for
sm_103a only, then link into one shared library next to this file.
Float arithmetic is compiled with contraction off (-fmad=false) and without
fast-math, so denormals are kept and every add/sub/mul rounds once.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
OBJ_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libcmdexec.so")

# (source, the defines of each object built from it), longest compiles first
def _objs(tiers, nds=(None,)):
    out = []
    for t in tiers:
        for ext in (1, 0):
            for nd in nds:
                d = dict(CMDX_TIER=t)
                if nd is not None:
                    d["CMDX_ND"] = nd
                d["CMDX_EXT"] = ext
                out.append(d)
    return out


CU_SOURCES = [("exec_tile2d.cu", _objs((2,), (0, 1))), ("exec_generic.cu", _objs((2,))),
              ("exec_contig.cu", _objs((2,))), ("exec_contig.cu", [dict(CMDX_TIER=0, CMDX_EXT=1, CMDX_OCC4=1)]),
              ("exec_contig.cu", [dict(CMDX_TIER=1, CMDX_EXT=0, CMDX_HALF16=1)]),
              ("exec_tile2d.cu", _objs((1, 0), (0, 1))),
              ("exec_generic.cu", _objs((4, 3, 1, 0))), ("exec_contig.cu", _objs((4, 3, 1, 0))),
              ("static_scratch.cu", [{}])]
CPP_SOURCES = ["cmd_api.cpp", "cmd_yaml.cpp", "exec_host.cpp"]
HEADERS = ["cmd_internal.h", "exec_common.cuh", "exec_pipe.cuh", "exec_tile2d.h", "interp_asm.cuh", "gen_interp.py"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    env = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if env and os.path.isdir(env):
        return env
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _sources():
    return ([os.path.join(CSRC, s) for s in sorted({c for c, _ in CU_SOURCES}) + CPP_SOURCES + HEADERS]
            + [os.path.join(ROOT, "include", "cmd.h"), os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(s) <= t for s in _sources())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libcmdexec.so unless it is newer than every source."""
    gen = os.path.join(CSRC, "gen_interp.py")
    inc_file = os.path.join(CSRC, "interp_asm.cuh")
    if not os.path.exists(inc_file) or os.path.getmtime(inc_file) < os.path.getmtime(gen):
        subprocess.run(["python3", gen], check=True, capture_output=True)
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(OBJ_DIR, exist_ok=True)
    home = cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    inc = ["-I" + os.path.join(home, "include"), "-I" + os.path.join(ROOT, "include")]
    jobs = []
    for s, variants in CU_SOURCES:
        for defs in variants:
            stem = s + "".join(f".{k[5:].lower()}{v}" for k, v in defs.items())
            obj = os.path.join(OBJ_DIR, stem + ".o")
            log = os.path.join(OBJ_DIR, stem + ".ptxas.txt")
            cmd = ([nvcc] + ARCH + ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-prec-div=true",
                                    "-prec-sqrt=true", "-ftz=false", "-Xptxas", "-v", "-Xcompiler", "-fPIC",
                                    "-c", os.path.join(CSRC, s), "-o", obj] + inc
                   + [f"-D{k}={v}" for k, v in defs.items()])
            jobs.append((cmd, obj, log))
    for s in CPP_SOURCES:
        obj = os.path.join(OBJ_DIR, s + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-Wextra", "-Wno-unused-parameter",
               "-c", os.path.join(CSRC, s), "-o", obj] + inc
        jobs.append((cmd, obj, None))

    def run(job):
        cmd, obj, log = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        if log:
            with open(log, "w") as f:
                f.write(r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(run, jobs))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart_static", "-lrt", "-lpthread", "-ldl"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
