"""Child process of the oracle mutation test (tests/test_oracle_mutants.py).

    python tests/mutant_pins_main.py <path of a kda_oracle.c build>

Loads that build in place of the oracle's own and runs the pin suite against
it, leaving out the frozen regression values (written by the oracle itself).
Exit status: pytest's (0 every pin passed, 1 a pin failed).
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

if __name__ == "__main__":
    import oracle
    oracle.use_library(sys.argv[1])
    import pytest
    sys.exit(pytest.main([os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-x", "-q",
                          "-p", "no:cacheprovider", "-k", "not frozen"]))
