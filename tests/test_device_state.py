"""Per-device launch state of the library (csrc/device_state.h), checked on the host: function
attributes, SM counts, the library's side stream and the static scratch address are kept per device
ordinal and per context, set up once even under concurrent host threads. No GPU: the table is plain
C++, compiled here with g++ and run."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "routing_dispatch_expert_gb300", "csrc")


def test_per_device_table_is_indexed_by_device_and_context(tmp_path):
    exe = tmp_path / "device_state_check"
    subprocess.check_call(["g++", "-std=c++17", "-O1", "-pthread", "-I", CSRC,
                           os.path.join(ROOT, "tests", "device_state_check.cpp"), "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip() == "ok"


def test_launchers_keep_no_process_wide_launch_flags():
    """Every launcher that sets a function attribute or caches a device property does so through a
    PerDevice table, not a process-wide static flag."""
    for name in os.listdir(CSRC):
        if not name.endswith(".cu"):
            continue
        src = open(os.path.join(CSRC, name)).read()
        for bad in ("static bool attr", "static int max_pairs", "static int n = 0"):
            assert bad not in src, f"{name}: {bad}"
        if "cudaFuncSetAttribute" in src:
            assert "PerDevice<" in src, name
