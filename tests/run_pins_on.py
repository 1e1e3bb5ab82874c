"""Run every oracle pin against one build of the oracle library.

    python tests/run_pins_on.py /path/to/liboracle.so

Exit status 0 if every pin holds, 1 if any pin fails (its name is printed).
test_oracle_mutants.py runs planted-mistake builds through this in a child
process, so that a mutant that crashes (for instance by reading outside its
arrays) is caught without taking the test session down with it.
"""

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
from oracle_pins import ALL_PINS  # noqa: E402


def main(path):
    orc = oracle.Oracle(path)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except Exception as e:  # an assertion or a refusal both count
            failed.append("%s: %s" % (pin.__name__, type(e).__name__))
    for f in failed:
        print("caught by", f)
    return 1 if failed else 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1]))
