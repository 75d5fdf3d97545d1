"""The fp8 dispatch quantises with an FMA-corrected product in place of an
IEEE division per element (Markstein's method; see quantise16_e4m3 in the
package's CUDA sources). quotient_check.c walks the whole input domain of
that step (every bf16 amax whose scale takes the fast path, every bf16 x of
either sign with |x| <= amax) on the host and asserts that the e4m3 code can
never differ from the one of the IEEE quotient. The GPU parity tests then
check the kernels' codes against the oracle bit for bit."""
import os
import re
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _build(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = os.path.join(HERE, "quotient_check.c")
    exe = str(tmp_path / "quotient_check")
    base = [cc, "-O2", "-ffp-contract=off", src, "-o", exe, "-lm"]
    if subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True).returncode != 0:
        subprocess.run(base, check=True, capture_output=True)
    return exe


def test_fma_corrected_quotient_gives_the_ieee_codes_on_the_whole_domain(tmp_path):
    exe = _build(tmp_path)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    m = re.search(r"amax (\d+) pairs (\d+) differ (\d+) violations (\d+)", out.stdout)
    assert m, out.stdout + out.stderr
    n_amax, pairs, differ, violations = map(int, m.groups())
    # every positive finite bf16 amax from about 2^-91 up: 219 binades of 128
    assert n_amax > 28000
    assert pairs > 10**9
    # the fp32 quotients do differ by an ulp in places; the codes never do
    assert differ > 0
    assert violations == 0 and out.returncode == 0
