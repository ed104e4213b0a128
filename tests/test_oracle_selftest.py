"""The oracle's C++ self-test program (oracle/selftest.cc): brute force over
every routing of 3 tokens to 2 of 3 experts at N = 1 and N = 3, routing
errors, combine closed forms and hand-worked bf16 / E4M3 conversions, checked
without Python in between."""
import subprocess


def test_oracle_selftest_program_passes(oracle_mod):
    r = subprocess.run([oracle_mod.SELFTEST], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failed" in r.stdout
