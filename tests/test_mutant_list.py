"""The oracle mutation check (tests/oracle_mutants.py) stays in step with the
oracle's sources: every planted mistake still names text that occurs exactly
once in its file and changes it (no GPU; the check itself takes minutes and
is run by hand)."""
import importlib.util
import os

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _mutants():
    spec = importlib.util.spec_from_file_location("oracle_mutants", os.path.join(HERE, "oracle_mutants.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.MUTANTS


@pytest.mark.parametrize("i,mutant", list(enumerate(_mutants())))
def test_mutant_text_occurs_once(i, mutant):
    path, old, new, what, equivalent = mutant
    assert path.startswith("oracle/") and old != new and what
    with open(os.path.join(ROOT, path)) as fh:
        assert fh.read().count(old) == 1, f"mutant {i} ({what})"
    assert equivalent is None or len(equivalent) > 20      # an equivalent mutant says why
