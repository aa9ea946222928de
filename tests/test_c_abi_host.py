"""The boundary is a C ABI: a plain C99 program (tests/c_abi_host.c) compiles
against include/kascade.h with -pedantic -Werror, links libkascade.so and
passes its host-side checks (validation before launch, workspace sizing,
status strings, the anchor DP). No GPU."""
import os
import shutil
import subprocess

import pytest

import __graft_entry__

ROOT = __graft_entry__.ROOT
PKG = os.path.join(ROOT, "long_context_anchor_gb300")


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return os.path.join(PKG, "libkascade.so")


def test_c_program_against_the_header_and_library(lib, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "c_abi_host")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_host.c"),
           "-L", PKG, "-lkascade", "-Wl,-rpath," + PKG, "-lm", "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "0 failure(s)" in run.stdout
    assert run.stdout.count("ok ") >= 20
