"""How much of each parity bar a GPU test used.

A parity test computes, per compared tensor, error / allowed (1.0 = exactly
at the bar).  ``record`` prints those ratios (visible with ``pytest -s`` or
``-rA``) and, when the environment variable DIFFATTN_RATIO_LOG names a file,
appends one JSON line per call to it: the test id and the ratios.  The
design notes keep a table of the worst ratio per tensor built from such a
log, so each bar and the margin the kernels leave under it can be read
without rerunning anything.
"""

import json
import os


def record(ratios, tag=""):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").rsplit(" ", 1)[0]
    rounded = {k: round(float(v), 4) for k, v in ratios.items()}
    print(f"[bar ratios] {test} {tag} {rounded}")
    path = os.environ.get("DIFFATTN_RATIO_LOG")
    if path:
        with open(path, "a") as fh:
            fh.write(json.dumps({"test": test, "tag": tag, "ratios": rounded}) + "\n")
