"""The oracle against the hand-derived fixtures in tests/golden (derivations on each line)."""
import os

import numpy as np

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_closed_forms_file():
    n = 0
    with open(os.path.join(GOLD, "e4m3_closed_forms.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            v, code = line.split()[:2]
            assert oracle.e4m3_encode(float(v)) == int(code, 16), line
            n += 1
    assert n >= 10


def test_schedule_worked_example_file():
    rows = {}
    tiles = []
    with open(os.path.join(GOLD, "schedule_worked_example.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "tile":
                tiles.append([int(v) for v in vals])
            else:
                rows[key] = [int(v) for v in vals]
    ids = np.array(rows["ids"], np.int32).reshape(3, 2)
    sch = oracle.schedule(ids, 3, 128, 128)
    assert sch["counts"].tolist() == rows["counts"]
    assert sch["offsets"].tolist() == rows["offsets"]
    assert sch["poff"].tolist() == rows["poff"]
    for key in ("perm@0", "perm@128", "perm@256"):
        at = int(key.split("@")[1])
        assert sch["perm"][at:at + len(rows[key])].tolist() == rows[key]
    assert sch["inv"].tolist() == rows["inv"]
    assert sch["tiles"].tolist() == tiles
