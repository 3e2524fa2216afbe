"""The header is plain C: a C11 client (tests/abi_host_check.c) compiles
with -Wall -Werror against include/fsdp.h, links against libfsdpreduce.so
and runs its host-only checks (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client_compiles_links_and_runs(tmp_path):
    import __graft_entry__ as g
    g.build()
    from sharded_fsdp_reduce_gb300 import _lib
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    exe = tmp_path / "abi_host_check"
    libdir = os.path.dirname(_lib.LIB_PATH)
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "abi_host_check.c"),
                    "-o", str(exe), "-L", libdir, "-lfsdpreduce", f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
