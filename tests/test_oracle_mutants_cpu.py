"""The oracle's pins catch planted mistakes.

A pin that cannot fail pins nothing. tests/_oracle_mutants.py lists small,
plausible mistakes in the oracle's functions (a dropped term, a wrong sign or
index, swapped operands, an off-by-one bound, a wrong constant); here the four
pin files run once per mistake, in a child pytest process whose oracle has
that mistake made in memory, and every run must fail. A control run loads the
same plugin with no mistake and must pass, so the failures come from the
mistakes and not from the plugin. No GPU needed.
"""
import os
import re
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import _oracle_mutants as M

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
PIN_FILES = ["test_oracle_pins.py", "test_oracle_fp8_pins.py", "test_oracle_nvfp4_pins.py",
             "test_oracle_attn_pins.py"]


def _run_pins(mutant):
    env = dict(os.environ)
    env.pop(M.ENV, None)
    if mutant:
        env[M.ENV] = mutant
    env["PYTHONPATH"] = os.pathsep.join([ROOT, HERE] + ([env["PYTHONPATH"]]
                                                         if env.get("PYTHONPATH") else []))
    env.pop("PYTEST_ADDOPTS", None)
    cmd = [sys.executable, "-m", "pytest", "-p", "_oracle_mutants", "-p", "no:cacheprovider",
           "-x", "-q", "-m", "not gpu"] + [os.path.join(HERE, f) for f in PIN_FILES]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:] + r.stderr[-2000:]


def test_every_oracle_function_has_a_planted_mistake():
    with open(os.path.join(ROOT, "oracle", "beam_oracle.py"), encoding="utf-8") as f:
        src = f.read()
    functions = set(re.findall(r"^def (\w+)\(", src, flags=re.M))
    targeted = {fn for fn, _, _ in M.MUTANTS.values()}
    assert functions - targeted == set()
    for name in M.MUTANTS:               # each edit applies where it says
        assert M.mutated_source(src, name) != src


def test_pins_pass_with_the_plugin_and_no_mistake():
    code, out = _run_pins(None)
    assert code == 0, out


def test_pins_catch_every_planted_mistake():
    names = sorted(M.MUTANTS)
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as pool:
        results = dict(zip(names, pool.map(_run_pins, names)))
    survivors = [n for n, (code, _) in results.items() if code == 0]
    broken = {n: out for n, (code, out) in results.items() if code not in (0, 1)}
    assert not broken, "pytest did not run cleanly for: " + ", ".join(
        f"{n}:\n{o}" for n, o in broken.items())
    assert not survivors, "the pins did not catch: " + ", ".join(survivors)
