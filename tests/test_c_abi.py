"""The C ABI used from C (host only, no GPU): tests/c_abi_host.c is compiled
with gcc against include/cmd.h, linked to the built library and run; it
builds a Command, lowers it, plans launches (aligned, shifted, a size
mismatch, an overlapping store), round-trips the text form and checks the
error paths."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

import tensor_command_execution_gb300 as T

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_c_program_against_the_library(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    T.lib()  # builds the library when it is missing or stale
    lib = T.library_path()
    exe = str(tmp_path / "c_abi_host")
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-O1", "-I", os.path.join(ROOT, "include"),
           os.path.join(HERE, "c_abi_host.c"), "-o", exe, "-L", os.path.dirname(lib),
           "-l:" + os.path.basename(lib), "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
