"""Host-side validation cost of the C ABI (SURVEY's "< 1 us per call" bar for the launch path,
the figure TileLang reports for its host-side checks).  A small C program (tests/c/) calls
csa_decode_step and csa_sparse_attn with arguments that pass every check but the last (a
workspace one byte short), so each call runs the whole validation and launches nothing; the
mean per call must stay under 1 us.  It runs on a GPU machine, where the library's per-device
lookups (SM count, device error word) are cached as they are in real use."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_validation_under_one_microsecond(tmp_path):
    from compressed_sparse_attention_csa_gb300 import _lib
    _lib.load()
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    pkg = os.path.join(ROOT, "compressed_sparse_attention_csa_gb300")
    exe = str(tmp_path / "validation_timing")
    subprocess.check_call([gcc, "-O2", "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "validation_timing.c"),
                           "-L", pkg, "-lcsa", "-Wl,-rpath," + pkg, "-o", exe])
    env = dict(os.environ)
    cuda_lib = [d for d in ("/usr/local/cuda/lib64", "/usr/local/cuda/lib") if os.path.isdir(d)]
    env["LD_LIBRARY_PATH"] = ":".join(cuda_lib + [env.get("LD_LIBRARY_PATH", "")])
    out = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    vals = dict(line.split() for line in out.stdout.strip().splitlines())
    print(vals)
    assert float(vals["decode_step_ns"]) < 1000.0
    assert float(vals["sparse_attn_ns"]) < 1000.0
