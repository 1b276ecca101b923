"""The quantiser's 6-candidate block scale: Markstein's correction step gives the E4M3 code of
the correctly rounded a / 6 for every binary32 a >= 0 (the Four Over Six choice of the pages is
made on those codes).  The check program evaluates both forms on all 2^31 + 1 inputs."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.gpu
def test_scale_division_codes_equal_for_every_input(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "scale_division_check")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe,
                    os.path.join(HERE, "scale_division_check.cu")], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    fields = out.stdout.split()
    counts = dict(zip(fields[0::2], map(int, fields[1::2])))
    assert counts["code_mismatches"] == 0
    # the quotient itself is not always correctly rounded (last place), so the check has teeth
    assert 0 < counts["quotient_mismatches"] < 2**22
