"""The C ABI from a plain C program (tests/csrc/abi_client.c): no Python or
PyTorch between the caller and the library.

The client is compiled with gcc against include/vqx.h, libvqx.so and the CUDA
runtime, run on planes this test writes, and its printed records are compared
with the oracle: the five exact sums bit for bit, every double bit for bit
(the frames stay in the exact range), and the integer psnr likewise.
"""
import os
import shutil
import struct
import subprocess

import numpy as np
import pytest

from exact_full_reference_gb300 import build as vb
from exact_full_reference_gb300 import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc", "abi_client.c")

DOUBLES = ("noise", "mse", "psnr", "psnr_uncapped", "ref_mean", "ref_meansq", "dist_mean",
           "dist_meansq")
UNITS = ("noise_units", "ref_sum", "dist_sum", "ref_sumsq", "dist_sumsq")


def cuda_home():
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_client(out_dir):
    lib = vb.build_library()
    exe = os.path.join(out_dir, "abi_client")
    cuda = cuda_home()
    libdirs = [d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                           os.path.join(cuda, "targets", "sbsa-linux", "lib"),
                           os.path.join(cuda, "targets", "x86_64-linux", "lib")) if os.path.isdir(d)]
    cmd = ["gcc", "-O2", "-std=c11", "-I" + os.path.join(ROOT, "include"),
           "-I" + os.path.join(cuda, "include"), "-o", exe, SRC, lib]
    cmd += ["-L" + d for d in libdirs] + ["-lcudart"]
    cmd += ["-Wl,-rpath," + os.path.dirname(lib)] + ["-Wl,-rpath," + d for d in libdirs]
    subprocess.run(cmd, check=True)
    return exe


def test_client_source_uses_only_the_header():
    """The client includes vqx.h and the CUDA runtime header, nothing of the
    library's sources."""
    with open(SRC) as f:
        src = f.read()
    includes = [line.split()[1] for line in src.splitlines() if line.startswith("#include")]
    assert '"vqx.h"' in includes
    assert not any("csrc" in i or ".cuh" in i for i in includes)


@pytest.mark.gpu
@pytest.mark.parametrize("name,frames", [("576x324_8bit_x1", None), ("1920x1080_10bit_x48", [0, 1, 2]),
                                         ("1920x1080_16bit_x64", [0, 63])])
def test_c_client_matches_the_oracle(tmp_path, orc, name, frames):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    w = wl.WORKLOADS[name]
    ref, dist = w.generate(frames)
    n = ref.shape[0]
    path = tmp_path / "planes.bin"
    with open(path, "wb") as f:
        f.write(np.ascontiguousarray(ref).tobytes())
        f.write(np.ascontiguousarray(dist).tobytes())
    exe = build_client(str(tmp_path))
    res = subprocess.run([exe, str(path), str(w.width), str(w.height), str(w.bpc), str(n)],
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    lines = res.stdout.split("\n")
    frames_out = [l.split() for l in lines if l.startswith("frame ")]
    assert len(frames_out) == n
    tail = [l for l in lines if l.startswith("errors ")][0].split()
    assert tail[1] == "ok"
    sc, un = orc.frames(ref, dist, w.bpc)
    ip = orc.int_psnr_frames(ref, dist, w.bpc)
    for f, row in enumerate(frames_out):
        vals = row[2:]
        for k, name_u in enumerate(UNITS):
            assert int(vals[k]) == int(un[f][name_u]), (f, name_u)
        assert int(vals[5]) == 0
        for k, name_d in enumerate(DOUBLES):
            got = struct.unpack("<d", struct.pack("<Q", int(vals[6 + k], 16)))[0]
            assert struct.pack("<d", got) == struct.pack("<d", float(sc[f][name_d])), (f, name_d)
        assert int(vals[14]) == int(ip[f]["sse"])
        for k, name_i in enumerate(("mse", "psnr", "psnr_uncapped")):
            got = struct.unpack("<d", struct.pack("<Q", int(vals[15 + k], 16)))[0]
            assert struct.pack("<d", got) == struct.pack("<d", float(ip[f][name_i])), (f, name_i)
