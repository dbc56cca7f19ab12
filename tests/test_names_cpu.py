"""Every global name that a function of the host-side Python modules reads is
defined at module level or is a builtin (catches harness breakage that only a
GPU run would otherwise reach)."""
import builtins
import importlib
import os
import symtable

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MODULES = ["bench", "__graft_entry__", "non_cartesian_mri_gather_gb300", "non_cartesian_mri_gather_gb300.build",
           "oracle", "inputs"]


def _globals_read(table):
    out = set()
    for child in table.get_children():
        if child.get_type() == "function":
            for sym in child.get_symbols():
                if sym.is_referenced() and sym.is_global() and not sym.is_assigned():
                    out.add(sym.get_name())
        out |= _globals_read(child)
    return out


@pytest.mark.parametrize("name", MODULES)
def test_no_undefined_globals(name):
    mod = importlib.import_module(name)
    path = mod.__file__
    table = symtable.symtable(open(path).read(), path, "exec")
    missing = sorted(n for n in _globals_read(table) if not hasattr(mod, n) and not hasattr(builtins, n))
    assert not missing, f"{name}: undefined globals {missing}"
