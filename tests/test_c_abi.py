"""The C ABI from plain C: the header compiles as C99 (no GPU), and a C
program drives the library end to end against the oracle (GPU)."""
import os
import shutil
import subprocess

import pytest

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def test_header_compiles_as_c99(tmp_path):
    src = tmp_path / "inc.c"
    src.write_text('#include "pagedattn.h"\nint main(void) { pa_pool* p = 0; (void)p; '
                   'return PA_OK + (int)PA_DTYPE_BF16 * 0; }\n')
    cc = shutil.which("gcc") or shutil.which("cc")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(REPO, "include"), "-c", str(src), "-o",
                    str(tmp_path / "inc.o")], check=True)


@pytest.mark.gpu
def test_c_client_end_to_end(pa_lib, cuda_device, tmp_path):
    lib_dir = os.path.dirname(pa_lib.library_path())
    exe = tmp_path / "pa_c_client"
    cmd = ["gcc", "-std=c11", "-O2", "-I", os.path.join(REPO, "include"),
           "-I", os.path.join(CUDA, "include"),
           os.path.join(REPO, "tests", "c_abi", "pa_c_client.c"),
           os.path.join(REPO, "oracle", "pa_oracle.c"), "-fopenmp",
           "-L", lib_dir, "-lpagedattn", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + lib_dir + ":" + os.path.join(CUDA, "lib64"), "-lm", "-o", str(exe)]
    subprocess.run(cmd, check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "c client ok" in res.stdout
