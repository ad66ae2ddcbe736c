"""The C ABI from plain C: tests/c_abi_check.c is compiled as C11 with
warnings as errors against include/dvl.h, linked to the library and run.
It calls only host entry points (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_is_c11_and_host_calls_work(tmp_path):
    from draft_vocab_lm_gb300 import build
    lib = build.build()
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "c_abi_check")
    libdir = os.path.dirname(lib)
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_check.c"),
                    "-L", libdir, "-ldvl", f"-Wl,-rpath,{libdir}", "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "c abi ok"
