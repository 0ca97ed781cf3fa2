"""libosm from plain C: tests/c_abi_consumer.c includes only osm.h and the CUDA
runtime header, links libosm.so, allocates its own device buffers and checks
the attention forward and row softmax against direct double-precision sums."""
import os
import shutil
import subprocess

import pytest

import exact_tiled_attention_osm_gb300 as osm

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_plain_c_consumer(cuda_ok, tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    osm.load_library()  # builds libosm.so if it is not there yet
    libdir = os.path.dirname(osm.LIB_PATH)
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "c_abi_consumer")
    subprocess.run([gcc, "-O2", "-std=c11", "-Wall", "-Wextra", "-Werror",
                    os.path.join(HERE, "c_abi_consumer.c"), "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), "-L", libdir, "-losm",
                    "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
                    "-Wl,-rpath," + libdir + ":" + os.path.join(cuda, "lib64"), "-o", exe],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    print(r.stdout, r.stderr)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("OK")
