"""The oracle's pins must catch plausible mistakes in the oracle itself.

Each case compiles the oracle source with one planted mistake (selected by
the ORACLE_PLANT macro; never defined in the library the other tests load),
points the oracle package at that build, and requires the pin suite
(tests/test_oracle.py) to FAIL. Everything runs on the CPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "sinkattn_oracle.cpp")

PLANTS = {
    1: "sink column dropped from the denominator",
    2: "sink multiplied by sm_scale",
    3: "query head h reads KV head h % Hkv instead of h // G",
    4: "causal mask aligned top-left instead of bottom-right",
    5: "window admits one key too many",
    6: "merge counts the sink once per split",
    7: "sm_scale not applied to the logits",
    8: "lse excludes the sink column",
    9: "FP8 keys scaled by the value scale and values by the key scale",
    10: "e4m3 exponent bias 8 instead of 7",
}


@pytest.mark.parametrize("plant", sorted(PLANTS), ids=lambda p: PLANTS[p].replace(" ", "_"))
def test_pins_catch_planted_mistake(tmp_path, plant):
    lib = tmp_path / ("liboracle_plant%d.so" % plant)
    subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp",
                    "-DORACLE_PLANT=%d" % plant, SRC, "-o", str(lib)], check=True)
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, ("pins did not catch: %s\n%s" % (PLANTS[plant], r.stdout[-2000:]))
    assert "failed" in r.stdout
