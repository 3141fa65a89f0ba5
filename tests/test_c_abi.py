"""The boundary from plain C: include/rmsnorm.h compiles as C99 and as C++17
with warnings as errors, and a C program linked to librmsnorm.so gets the
library's host-side argument checks (tests/c_abi_check.c).  No GPU: every
call in the program fails validation or is an empty batch."""
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
INCLUDE = ROOT / "include"
PKG = ROOT / "row_wise_normalization_rms_gb300"


@pytest.fixture(scope="module")
def lib_path():
    from row_wise_normalization_rms_gb300 import build

    return build.build()


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_against_the_header_and_library(lib_path, tmp_path):
    exe = tmp_path / "c_abi_check"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Wpedantic", "-Werror", f"-I{INCLUDE}",
           str(ROOT / "tests" / "c_abi_check.c"), f"-L{lib_path.parent}", f"-l:{lib_path.name}",
           f"-Wl,-rpath,{lib_path.parent}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    assert run.stdout.strip() == "ok"


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_header_is_valid_cxx(tmp_path):
    src = tmp_path / "inc.cc"
    src.write_text('#include "rmsnorm.h"\nint main() { return rms_status_string(RMS_OK) ? 0 : 1; }\n')
    r = subprocess.run(["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        f"-I{INCLUDE}", str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
