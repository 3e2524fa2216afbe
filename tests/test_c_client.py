"""The header is plain C: a C11 client (tests/abi_host_check.c) compiles
with -Wall -Werror against include/fsdp.h, links against libfsdpreduce.so
and runs its host-only checks (no GPU needed); a second one
(tests/abi_gpu_check.c, -m gpu) runs the step on device buffers of its own,
with no Python in the process, and its results are checked against the
oracle."""
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


@pytest.mark.gpu
def test_c_client_runs_the_step_on_the_gpu(tmp_path, orc):
    # tests/abi_gpu_check.c: buffers from the CUDA runtime, the step through
    # the C ABI, results written to a file; bit-exact against the oracle
    import numpy as np
    import __graft_entry__ as g
    g.build()
    from sharded_fsdp_reduce_gb300 import _lib, build as B
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    cuda = os.path.dirname(os.path.dirname(B.nvcc()))
    cudalib = next((d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                    if os.path.exists(os.path.join(d, "libcudart.so"))), None)
    assert cudalib is not None, "libcudart.so not found beside nvcc"
    exe = tmp_path / "abi_gpu_check"
    libdir = os.path.dirname(_lib.LIB_PATH)
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    os.path.join(ROOT, "tests", "abi_gpu_check.c"), "-o", str(exe),
                    "-L", libdir, "-lfsdpreduce", f"-Wl,-rpath,{libdir}",
                    "-L", cudalib, "-lcudart", f"-Wl,-rpath,{cudalib}"], check=True)
    out = tmp_path / "out.bin"
    r = subprocess.run([str(exe), str(out)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
    N, P, PPAD = 2, 4099, 4100
    raw = out.read_bytes()
    f32 = np.frombuffer(raw, np.float32, 3 * PPAD).reshape(3, PPAD)
    b16 = np.frombuffer(raw, np.uint16, 3 * PPAD, offset=12 * PPAD).reshape(3, PPAD)
    nf, wt = (int(x) for x in np.frombuffer(raw, np.uint32, 2, offset=18 * PPAD))
    # the same inputs, rebuilt here, through the oracle
    j = np.arange(PPAD)
    p = np.where(j < P, ((j * 5) % 201 - 100) / np.float32(2048.0), 0).astype(np.float32)
    m = np.zeros(PPAD, np.float32)
    v = np.zeros(PPAD, np.float32)
    for t in (1, 2, 3):
        grads = []
        for q in range(N):
            x = (((j * 7 + q * 13 + t * 29) % 97 - 48) / np.float32(1024.0)).astype(np.float32)
            bits = (x.view(np.uint32) >> 16).astype(np.uint16)
            bits[P:] = 0
            grads.append(bits)
        shards, full = orc.fsdp_step(grads, "bf16", N, p, m, v, "bf16", orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, t))
    np.testing.assert_array_equal(f32[0].view(np.uint32), p.view(np.uint32))
    np.testing.assert_array_equal(f32[1].view(np.uint32), m.view(np.uint32))
    np.testing.assert_array_equal(f32[2].view(np.uint32), v.view(np.uint32))
    np.testing.assert_array_equal(b16[0], shards)
    np.testing.assert_array_equal(b16[1], full)
    np.testing.assert_array_equal(b16[2], full)
    assert nf == 0
    assert wt == 0  # no bounded wait of the gathers gave up
