"""The C ABI from plain C: tests/c_abi_host.c includes include/kvc.h, compiles as
C99 with warnings as errors (so the header is valid C, not only C++), links
against libkvc.so and runs its host-only calls without a GPU. Its pyramid
budgets are compared with the oracle's planner; its validation and null-handle
statuses with the header's documented codes."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "kv_cache_compression_snapkv_gb300")
LIB = os.path.join(PKG, "libkvc.so")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(LIB):
        pytest.skip("libkvc.so not built")
    exe = str(tmp_path_factory.mktemp("cabi") / "c_abi_host")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_host.c"),
           "-L", PKG, "-lkvc", f"-Wl,-rpath,{PKG}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _run(exe, *args):
    r = subprocess.run([exe, *map(str, args)], capture_output=True, text=True, timeout=120)
    return r.returncode, r.stdout


@pytest.mark.parametrize("L,avg,depth,n,alpha", [
    (32, 1024, 8, 131072, 64), (32, 512, 8, 32768, 32), (7, 96, 3, 500, 16), (1, 64, 2, 1000, 8)])
def test_pyramid_budgets_from_c(client, L, avg, depth, n, alpha):
    from oracle import plan_budgets
    rc, out = _run(client, "budgets", L, avg, depth, n, alpha)
    assert rc == 0, out
    got = [int(x) for x in out.split()]
    assert got == plan_budgets(L, "pyramid", avg, depth, 32, max_budget=n - alpha)
    if (L, avg) == (32, 1024):
        assert got[0] == 1920 and got[-1] == 128 and sum(got) == 32 * 1024


def test_validation_and_null_handles_from_c(client):
    rc, out = _run(client, "checks")
    assert rc == 0, out
    vals = dict(line.split(" ", 1) for line in out.strip().splitlines())
    assert vals["bad_head_dim"] == "2"            # KVC_E_SHAPE
    assert vals["too_many_new_tokens"] == "2"     # KVC_E_SHAPE (beyond KVC_MAX_NEW_TOKENS)
    assert vals["uneven_budget"] == "1"           # KVC_E_ARG (not a multiple of the group)
    assert vals["null_out"] == "1"
    assert vals["append_null"] == "1"
    assert vals["decode_null"] == "1"
    assert vals["free_null"] == "0"
    assert vals["checked_build"] in ("0", "1")
    assert int(vals["launches"]) >= 0
    assert vals["status_capacity"] == "capacity exceeded"
