"""The C ABI from C itself, without the Python binding.

* include/arf.h compiles as strict C99 and as C++17 with every warning an
  error.
* tests/c_abi/host_calls.c, a plain C program linked against libarf.so,
  makes the host-only calls (status strings, shape rules, planner, plan
  checker, staging sizes); its results equal those of the same calls made
  through the binding. No GPU needed.
* tests/c_abi/device_run.c runs the epilogue from C on device buffers of the
  CUDA runtime and checks it against the C oracle, linked into the same
  program (GPU only).
"""
import os
import subprocess

import pytest

import all_reduce_residual_gb300 as arf
import oracle
from all_reduce_residual_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
CDIR = os.path.join(ROOT, "tests", "c_abi")
LIBDIR = os.path.dirname(_binding.LIB_PATH)
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def lib():
    build.build()
    arf.load()
    return LIBDIR


def _cc(args, cwd):
    r = subprocess.run(args, cwd=cwd, capture_output=True, text=True)
    assert r.returncode == 0, f"{' '.join(args)}\n{r.stdout}\n{r.stderr}"


def test_header_compiles_as_strict_c_and_cpp(tmp_path):
    src = tmp_path / "inc.c"
    src.write_text('#include "arf.h"\nint main(void) { return (int)sizeof(arf_run_opts_t) > 0 ? 0 : 1; }\n')
    _cc(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I", INCLUDE, str(src)],
        tmp_path)
    cpp = tmp_path / "inc.cpp"
    cpp.write_text(src.read_text())
    _cc(["g++", "-std=c++17", "-pedantic", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I", INCLUDE, str(cpp)],
        tmp_path)


def _run_host_calls(tmp_path, libdir):
    exe = tmp_path / "host_calls"
    _cc(["gcc", "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, os.path.join(CDIR, "host_calls.c"),
         "-L", libdir, "-larf", f"-Wl,-rpath,{libdir}", "-o", str(exe)], tmp_path)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    return [ln.split(" ", 2) if ln.startswith("status") else ln.split() for ln in r.stdout.splitlines()]


SHAPES = [(arf.ARF_ALLREDUCE, 4, 5851, 7168, arf.ARF_BF16), (arf.ARF_AR_RESIDUAL_RMSNORM, 4, 5851, 7168, arf.ARF_BF16),
          (arf.ARF_AR_RESIDUAL_RMSNORM, 16, 585, 7168, arf.ARF_FP16), (arf.ARF_AR_RESIDUAL_RMSNORM, 8, 1, 7168, arf.ARF_BF16),
          (arf.ARF_ALLREDUCE, 2, 4096, 4098, arf.ARF_BF16), (arf.ARF_AR_RESIDUAL_RMSNORM, 3, 2000, 7168, arf.ARF_BF16),
          (arf.ARF_AR_RESIDUAL_RMSNORM, 65, 8, 1024, arf.ARF_BF16), (arf.ARF_AR_RESIDUAL_RMSNORM, 2, 8, 0, arf.ARF_BF16)]


def test_host_calls_from_c_match_the_binding(tmp_path, lib):
    out = _run_host_calls(tmp_path, lib)
    gb300 = arf.DeviceCaps(num_sms=152, max_cluster=16, max_threads_per_sm=2048, max_smem_per_block=232448)
    small = arf.DeviceCaps(num_sms=20, max_cluster=1, max_threads_per_sm=1536, max_smem_per_block=101376)
    lines = {}
    for f in out:
        lines.setdefault(f[0], []).append(f[1:])
    for code, text in lines["status"]:
        assert text == arf.arf_status_string(int(code)), code
    sup = {int(i): int(s) for i, s in lines["supports"]}
    plans = {tag: [int(x) for x in rest] for tag, *rest in lines["plan"]}
    checks = {int(i): int(s) for i, s in lines["check"]}
    staging = {int(i): int(b) for i, b in lines["staging"]}
    for i, (pat, W, M, H, dt) in enumerate(SHAPES):
        assert sup[i] == arf.arf_supports(None, pat, W, M, H, dt), i
        if sup[i] != arf.ARF_OK:
            assert f"gb300_{i}" not in plans
            continue
        for tag, caps, fn in ((f"gb300_{i}", gb300, arf.arf_plan_for_caps), (f"small_{i}", small, arf.arf_plan_rules)):
            p = arf.Plan()
            st = fn(caps, pat, W, M, H, dt, p)
            assert plans[tag][0] == st, tag
            assert plans[tag][1:] == [p.path, p.threads, p.vpt, p.cluster, p.grid, p.w_spec, p.stages], tag
        assert checks[i] == arf.ARF_OK
        assert staging[i] == arf.arf_host_staging_bytes(pat, W, M, H, dt)
    assert int(lines["static_staging"][0][0]) == arf.arf_static_staging_bytes()
    assert int(lines["null_ws"][0][0]) == arf.ARF_ERR_INVALID_ARG


@pytest.mark.gpu
def test_device_run_from_c_matches_the_oracle(tmp_path, lib):
    exe = tmp_path / "device_run"
    orc = tmp_path / "arf_oracle.o"
    _cc(["gcc", *[f for f in oracle.CFLAGS if f not in ("-fPIC", "-shared")], "-c", "-I", os.path.dirname(oracle.SRC),
         oracle.SRC, "-o", str(orc)], tmp_path)
    _cc(["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, "-I", os.path.dirname(oracle.SRC),
         "-I", os.path.join(CUDA_HOME, "include"), os.path.join(CDIR, "device_run.c"), str(orc),
         "-L", lib, "-larf", "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart", "-lm",
         f"-Wl,-rpath,{lib}", f"-Wl,-rpath,{os.path.join(CUDA_HOME, 'lib64')}", "-o", str(exe)], tmp_path)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count("OK ") == 7, r.stdout
