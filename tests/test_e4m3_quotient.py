"""The GPU FP8 quantiser forms v / s without a division (Markstein's
corrected product with the rounded reciprocal, two fused multiply-adds).
tests/e4m3_quotient_check.c checks, for every bf16 block maximum with scale
s >= 2^-112 and every bf16 value up to it, that this gives the same E4M3
code as the IEEE fp32 quotient the blockwise FP8 recipe specifies
("Scalable Training of Mixture-of-Experts Models with Megatron Core", §5).
Runs on the host in about 20 s."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_markstein_quotient_gives_ieee_e4m3_codes_for_all_bf16(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "e4m3_quotient_check")
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-o", exe, os.path.join(HERE, "e4m3_quotient_check.c"),
                    "-lm"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout
    assert "E4M3 differences 0" in r.stdout
