"""Runs the oracle's pins against an edited private copy of the oracle.

Used by the planted-mistake tests: a copy of the oracle's source with an edit
applied is executed as a fresh module, and the pin functions of
test_oracle_encodings.py and test_oracle_path.py (loaded here as private
modules, so pytest does not collect them twice) are called with that copy in
place of the oracle.  Nothing here changes the oracle the other tests import.
"""

import importlib.util
import os
import types

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE_PATH = os.path.join(os.path.dirname(HERE), "oracle", "mx_oracle.py")
PIN_FILES = ("test_oracle_encodings.py", "test_oracle_path.py", "test_oracle_kv.py")


def oracle_source():
    with open(ORACLE_PATH) as f:
        return f.read()


def oracle_from_source(src):
    mod = types.ModuleType("mx_oracle_planted")
    mod.__file__ = ORACLE_PATH
    exec(compile(src, ORACLE_PATH, "exec"), mod.__dict__)
    return mod


def oracle_copy(edits):
    """The oracle with each (text, replacement) applied; every text occurs once."""
    src = oracle_source()
    for old, new in edits:
        assert src.count(old) == 1, f"planted text not found exactly once: {old!r}"
        src = src.replace(old, new)
    return oracle_from_source(src)


def _load_pins():
    mods = []
    for name in PIN_FILES:
        spec = importlib.util.spec_from_file_location("pins_" + name[:-3], os.path.join(HERE, name))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mods.append(mod)
    return mods


PINS = _load_pins()


def _cases(mod):
    for name in sorted(n for n in dir(mod) if n.startswith("test_")):
        fn = getattr(mod, name)
        params = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if params:
            for v in params[0].args[1]:
                yield name, (lambda fn=fn, v=v: fn(v))
        else:
            yield name, fn


def failing_pins(oracle, stop_at_first):
    """Names of the pins that fail with `oracle` in place of the real one."""
    failed = []
    for mod in PINS:
        saved = mod.O
        mod.O = oracle
        try:
            for name, call in _cases(mod):
                try:
                    with np.errstate(all="ignore"):
                        call()
                except Exception:
                    failed.append(name)
                    if stop_at_first:
                        return failed
        finally:
            mod.O = saved
    return failed
