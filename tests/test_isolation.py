"""The oracle and the product path share no code and do not use each other.

The package and its CUDA sources never import, load or include anything of the oracle;
the oracle never imports the package or includes its sources; and the package imports
and plans with the oracle made unimportable.  Only the seeded input generator (synth)
serves both, and it holds none of the method's arithmetic.
"""
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "kv_cache_incremental_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def sources(folder, exts):
    for base, _, files in os.walk(folder):
        if "_build" in base or "__pycache__" in base:
            continue
        for f in files:
            if f.endswith(exts):
                yield os.path.join(base, f)


def test_package_sources_do_not_reach_the_oracle():
    for path in sources(PKG, (".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
        text = open(path).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), path
        assert "liboracle" not in text and "oracle.c" not in text, path
        assert not re.search(r'#include\s+"[^"]*oracle', text), path


def test_oracle_sources_do_not_reach_the_package():
    for path in sources(ORACLE, (".py", ".c", ".h")):
        text = open(path).read()
        assert "kv_cache_incremental_gb300" not in text and "libkvinc" not in text, path
        assert not re.search(r'#include\s+"[^"]*(csrc|kvinc)', text), path


def test_package_works_with_the_oracle_unimportable():
    code = (
        "import sys\n"
        "sys.modules['oracle'] = None\n"      # any import of the oracle now raises
        "import kv_cache_incremental_gb300 as kvi\n"
        "p = kvi.plan_decode(152, 32, 8, 128, 0, kvi.KV_GLOBAL, [4095])\n"
        "assert p['n_splits'] == [8], p\n"
        "assert 'oracle' not in [m for m in sys.modules if sys.modules[m] is not None]\n"
        "print('ok')\n")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True,
                         text=True, timeout=300)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stderr[-2000:]
