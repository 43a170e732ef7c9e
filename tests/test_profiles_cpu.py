"""The committed ncu summaries: each names a known workload, records the hash
of the CUDA sources it was taken on, and gives its commands in full, through
committed files only, with ncu left off the clocks."""
import glob
import os
import re

import pytest

from weight_only_quantized_qgemv_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))
KNOWN = set(synth.WORKLOADS + synth.VARIANT_WORKLOADS + synth.PREFILL_WORKLOADS)


def test_there_are_profiles():
    assert len(PROFILES) >= 3


@pytest.mark.parametrize("path", PROFILES, ids=os.path.basename)
def test_profile_summary_format(path):
    text = open(path).read()
    m = re.search(r"^workload: (\S+)$", text, flags=re.M)
    assert m and m.group(1) in KNOWN, "names a workload of the bench"
    assert m.group(1) in os.path.basename(path), "the file is named for its workload"
    assert re.search(r"^source_hash: [0-9a-f]{16}$", text, flags=re.M)
    ncu = [ln for ln in text.splitlines() if re.match(r"\s*ncu\s", ln)]
    assert ncu, "gives the ncu command"
    for ln in ncu:
        assert "--clock-control none" in ln
    assert "python bench.py" in text
    assert "/root/" not in text and "_work/" not in text
    t = re.search(r"^traffic_bytes_per_launch: (\d+)$", text, flags=re.M)
    if t:
        assert int(t.group(1)) > 0
