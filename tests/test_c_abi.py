"""The boundary from plain C: a C99 program (tests/c_abi/host_calls.c)
built with gcc against include/layoutmove.h, linked to liblayoutmove.so,
calls the host side of the ABI and prints what it gets (no GPU needed)."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    from layout_driven_movement_gb300 import _build
    lib = _build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path_factory.mktemp("c_abi") / "host_calls")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    f"-I{ROOT}/include",
                    os.path.join(ROOT, "tests", "c_abi", "host_calls.c"),
                    lib, f"-Wl,-rpath,{os.path.dirname(lib)}", "-o", exe],
                   check=True, capture_output=True, timeout=300)
    return exe


def test_c_program_drives_the_host_abi(program):
    r = subprocess.run([program], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    out = dict(line.split(" ", 1) for line in r.stdout.splitlines())
    # the padded composition of the TV layout and the bf16 tiling, closed
    # forms of "CUTE布局代数" §2.2 and §3.2
    assert out["compose"] == "((4,8),2):((18,1),9)"
    assert out["zipped_divide"] == "((64,64),(128,128)):((8192,1),(524288,64))"
    assert out["plan_path"] == "STAGED"
    assert out["banks"] == "8 1"           # 32 rows of an 8-wide tile
    assert out["local_partition"] == "(2,4):(32,2) 9"
    assert out["bad"] == "LM_E_INVALID"
    assert out["bad_out_null"] == "1"       # a failed call leaves no handle
    assert out["version"]
