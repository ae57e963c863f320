"""The recorded DRAM traffic that bench.py reports beside its roofline
(profiles/traffic.json): every record names its workload, call and kernel
sources, the bytes are the read and write counters' sum, and each call is
recorded once per workload and source.  (A record whose source no longer
matches the kernels is kept but not reported.)"""

import json
import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

PATH = os.path.join(ROOT, "profiles", "traffic.json")


def _records():
    with open(PATH) as f:
        return json.load(f)


def test_records_are_well_formed():
    recs = _records()
    assert recs
    seen = set()
    for r in recs:
        for key in ("config", "T", "call", "source", "bytes_per_call", "dram_read", "dram_write", "command"):
            assert key in r, (key, r.get("config"), r.get("call"))
        assert r["config"] in synth.CONFIGS
        assert r["T"] == synth.CONFIGS[r["config"]].T  # full-size captures only
        assert re.fullmatch(r"[0-9a-f]{16}", r["source"])
        assert r["dram_read"] > 0 and r["dram_write"] > 0
        # (each figure is a mean over launches, rounded on its own)
        assert abs(r["bytes_per_call"] - (r["dram_read"] + r["dram_write"])) <= 1
        # DRAM bytes near the algorithmic bytes where the record carries them
        # (a call cannot move much less than its operands, nor many times more
        # without a defect worth a look)
        if r.get("algorithmic_bytes"):
            assert 0.8 < r["bytes_per_call"] / r["algorithmic_bytes"] < 2.0, r
        key = (r["config"], r["T"], r["call"], r["source"])
        assert key not in seen, key
        seen.add(key)

