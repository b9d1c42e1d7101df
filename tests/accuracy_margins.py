"""Turns the errors a GPU test run recorded (GDN_RECORD_MARGINS=<file>) into
the accuracy guard table tests/accuracy_margins.json: per parity case and
quantity, four times the largest error max|d| / max|ref| seen, at least 1e-4.

    GDN_RECORD_MARGINS=/tmp/m.jsonl python -m pytest tests -m gpu
    python tests/accuracy_margins.py /tmp/m.jsonl

With --merge, the cases of the file are added to (or replace theirs in) the
existing table, and every other case keeps its entry: for a run of new tests
only.
"""
import json
import os
import sys

FACTOR, FLOOR = 4.0, 1e-4


def main(path, merge=False):
    worst = {}
    with open(path) as f:
        for line in f:
            r = json.loads(line)
            key = (r["case"], r["quantity"])
            worst[key] = max(worst.get(key, 0.0), r["rel_to_max"])
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "accuracy_margins.json")
    margins = {}
    if merge:
        with open(out) as f:
            margins = json.load(f)["margins"]
        for case in {c for c, _ in worst}:
            margins.pop(case, None)
    for (case, q), e in sorted(worst.items()):
        margins.setdefault(case, {})[q] = float(f"{max(FACTOR * e, FLOOR):.3g}")
    margins = dict(sorted(margins.items()))
    with open(out, "w") as f:
        json.dump({"note": "largest error max|d|/max|ref| of each GPU parity case against the fp64 oracle, times "
                           f"{FACTOR:g} (floor {FLOOR:g}): an accuracy guard inside the parity bar",
                   "margins": margins}, f, indent=1, sort_keys=True)
        f.write("\n")
    print(f"{len(worst)} quantities in {len(margins)} cases -> {out}")


if __name__ == "__main__":
    main(sys.argv[1], merge="--merge" in sys.argv[2:])
