"""The oracle's pins catch plausible mistakes: each mutation in
``tests/oracle_mutations.py`` is planted in a child pytest run of the pin
suite (CPU only), and that run must fail."""
import os
import subprocess
import sys

import pytest

from tests.oracle_mutations import MUTATIONS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name):
    env = dict(os.environ, ET_ORACLE_MUTATION=name)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "tests.oracle_mutations",
                        "tests/test_oracle_pins.py", "-m", "not gpu"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"the pins did not notice: {name}\n{r.stdout[-2000:]}"


def test_pins_pass_without_mutation():
    env = {k: v for k, v in os.environ.items() if k != "ET_ORACLE_MUTATION"}
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "tests.oracle_mutations",
                        "tests/test_oracle_pins.py", "-m", "not gpu"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
