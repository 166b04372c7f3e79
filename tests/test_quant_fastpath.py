"""The GPU kernels form activation codes as rint(x * fl(127 / amax)) and
fall back to the exact division x / fl(amax / 127) only near a tie
(common.cuh, quant8_group4).  The reading of the pages' in-kernel
quantisation ("Що змінює ML Drift для on-device AI-інференсу на вашому
телефоні?", tech.dede.sh, section "Stage-aware оптимізація для великих
мовних моделей") is the division.  quant_fastpath.c compares the two for
every pair of positive fp16 values x <= amax; they must never differ."""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_reciprocal_codes_equal_division_codes_exhaustively():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "quant_fastpath")
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", exe,
                        os.path.join(HERE, "quant_fastpath.c"), "-lm"], check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    pairs, bad, slow = (int(v) for v in r.stdout.split())
    assert pairs == 0x7BFF * (0x7BFF + 1) // 2          # every 0 < x <= amax
    assert bad == 0, f"{bad} codes differ from the division"
    assert r.returncode == 0
    # the fallback is rare (it only guards near-ties)
    assert 0 < slow < pairs // 1000
