"""The C ABI from a plain C99 program: include/mlp.h compiles as strict C
and the library links and answers its host-side calls (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

import activated_mlp_gemms_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    if not os.path.exists(m.LIB_PATH):
        from activated_mlp_gemms_gb300 import _build
        _build.build()
    exe = str(tmp_path_factory.mktemp("c_abi") / "abi_host")
    libdir = os.path.dirname(m.LIB_PATH)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_host.c"),
           "-o", exe, "-L", libdir, "-lmlp", "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    return dict(line.split(" ", 1) for line in r.stdout.strip().splitlines())


def test_workspace_sizes_match_the_binding(results):
    p = m.problem(2048, 4096, 11008)
    assert int(results["ws_fwd"]) == m.mlp_workspace_size(p, m.MODE_FWD)
    assert int(results["ws_bwd"]) == m.mlp_workspace_size(p, m.MODE_BWD)
    assert int(results["ws_null"]) == 0


def test_strings(results):
    assert results["status_ok"] == m.lib().mlp_status_string(0).decode()
    assert results["version"] == m.lib().mlp_version().decode()


def test_validation_before_any_launch(results):
    assert int(results["fwd_null_problem"]) == -1   # MLP_ERR_INVALID_ARG
    assert int(results["fwd_null_x"]) == -1
    assert int(results["fwd_bad_h"]) == -2          # MLP_ERR_ALIGNMENT
