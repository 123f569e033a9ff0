"""The C ABI from plain C: tests/c_client/abi_client.c is compiled with gcc as C11 against
include/*.h alone, linked to libgdn_decode.so, and run without a GPU. The argument structs must
have the same size in C as inside the library, and the host-side checks must refuse bad calls
with the documented status codes before any CUDA work."""
import os
import shutil
import subprocess

import pytest

from ssm_recurrent_decode_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def client_output(tmp_path_factory):
    if not shutil.which("gcc"):
        pytest.skip("gcc is needed to build the C client")
    lib = _build.build()
    exe = tmp_path_factory.mktemp("c_client") / "abi_client"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_client", "abi_client.c"), "-o", str(exe),
                    "-L", os.path.dirname(lib), "-lgdn_decode", f"-Wl,-rpath,{os.path.dirname(lib)}"],
                   check=True)
    run = subprocess.run([str(exe)], capture_output=True, text=True, check=True)
    return dict(line.split(" ", 1) for line in run.stdout.strip().splitlines())


def test_struct_sizes_agree_between_c_and_the_library(client_output):
    assert client_output["c_sizes"] == client_output["lib_sizes"]
    import ssm_recurrent_decode_gb300 as gdn
    assert int(client_output["version"]) == gdn.ABI_VERSION


def test_host_checks_from_c(client_output):
    assert int(client_output["null_args"]) == -1          # GDN_ERR_NULL
    assert int(client_output["bad_K"]) == -2              # GDN_ERR_SHAPE
    assert int(client_output["bad_dtype"]) == -3          # GDN_ERR_DTYPE
    assert int(client_output["misaligned_state"]) == -4   # GDN_ERR_ALIGN
    assert int(client_output["bad_gate_mode"]) == -6      # GDN_ERR_ARG
    assert int(client_output["null_indices"]) == -1
    assert int(client_output["empty_batch"]) == 0         # nothing to launch
    assert int(client_output["front_width"]) == 4 * 32 * 128 + 2 * 32
    assert "NULL" in client_output["strerror_null"]
