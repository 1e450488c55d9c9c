"""Values the pages print, stored under tests/golden/ with their citations, against the oracle and the
library (host-side, no GPU)."""
import os

import oracle
from beam_search_shared_gb300 import bsp

HERE = os.path.dirname(os.path.abspath(__file__))


def _rows(name):
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield tuple(int(x) for x in line.split())


def test_bucket_rows_printed_by_the_pages():
    rows = list(_rows("bucket_rows.txt"))
    assert len(rows) == 3
    for valid, capacity, bound in rows:
        assert oracle.bucket_rows(valid, capacity) == bound, (valid, capacity)
        assert bsp.bucket_rows(valid, capacity) == bound, (valid, capacity)


def test_tail_bound_printed_by_the_pages():
    import re
    limits = {}
    with open(os.path.join(HERE, "golden", "limits.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                limits[k] = int(v)
    assert bsp.MAX_TAIL == limits["max_tail"]
    header = open(os.path.join(HERE, "..", "include", "bsp.h")).read()
    assert int(re.search(r"#define BSP_MAX_TAIL (\d+)", header).group(1)) == limits["max_tail"]
