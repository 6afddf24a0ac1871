"""The SLORA_DEBUG build on the GPU, in a process of its own (the library is
chosen when the binding loads it): tests/debug_build_check.py."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_catches_planted_page_indices():
    from lora_adapters_gb300 import build

    build.build(debug=True)
    env = dict(os.environ, SLORA_DEBUG="1")
    res = subprocess.run([sys.executable, "-m", "tests.debug_build_check"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert "debug build OK" in res.stdout
