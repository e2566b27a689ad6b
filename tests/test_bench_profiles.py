"""The bench's roofline `traffic` comes from committed ncu summaries under
profiles/, and only while the summary was taken on the kernel source that
runs now (its kernel_source_hash line).  These checks need no GPU."""
from __future__ import annotations

import os
import re

import bench

PROFILES = os.path.join(bench.ROOT, "profiles")

# (profile, kernel sources, traffic field) of each dominant kernel the bench reports
DOMINANT = [
    ("fattn_bwd_kernels_b2h16n4096d128_causal", bench.BWD_SOURCES, "dkdv_dram_bytes_per_launch"),
    ("fattn_linear_kernels_lin_b2h16n4096e64", bench.LINEAR_SOURCES, "output_dram_bytes_per_launch"),
    ("fattn_fwd_kernel_b2h16n4096d128_causal", bench.KERNEL_SOURCES, "dram_bytes_per_launch"),
]


def _fields(name):
    out = {}
    with open(os.path.join(PROFILES, name + ".txt")) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                out[k.strip()] = v.strip()
    return out


def test_summaries_name_their_command_and_hash():
    """Each summary of a dominant kernel gives the command that made it and
    the source hash and traffic the bench reads."""
    for name, _, field in DOMINANT:
        f = _fields(name)
        assert "python bench.py" in f.get("command", ""), name
        assert "--clock-control none" in f.get("ncu", ""), name
        assert len(f.get("kernel_source_hash", "").split()[0]) == 16, name
        assert float(f[field].split()[0]) > 0, name


def test_traffic_only_for_the_current_source():
    """A summary whose hash matches yields its traffic; with any other hash
    the bench reports null rather than counters of another kernel."""
    for name, sources, field in DOMINANT:
        f = _fields(name)
        current = f["kernel_source_hash"].split()[0] == bench.kernel_source_hash(sources)
        got = bench.ncu_traffic("", name, sources, field)
        if current:
            assert got == float(f[field].split()[0]), name
        else:
            assert got is None, name
    # a source list whose hash cannot match any summary
    assert bench.ncu_traffic("", DOMINANT[0][0], ("v_prepass.cuh",), DOMINANT[0][2]) is None


def _reads(name, f):
    """DRAM bytes read per launch, as the summary records them."""
    if "dram_bytes_read" in f:
        return float(f["dram_bytes_read"].split()[0])
    for v in f.values():
        m = re.search(r"dram read (\d+)", v)
        if m:
            return float(m.group(1))
    raise KeyError(name)


def test_traffic_is_near_the_algorithmic_bytes():
    """Counters that belong to the kernel: the DRAM bytes read per launch are
    at least the algorithmic bytes read (one pass over the inputs cannot be
    skipped), and reads plus writes stay under 2x the algorithmic bytes
    (re-reads that L2 misses).  Writes may fall short: what is still in L2
    when a kernel ends is not counted."""
    mb = 1 << 20
    algorithmic = {  # (bytes read, bytes written)
        # dK/dV: Q, K, V, dO read, dK, dV written
        "fattn_bwd_kernels_b2h16n4096d128_causal": (4 * 32 * mb, 2 * 32 * mb),
        # output kernel: Q, K, V read (the parts' totals are a few MB), O written
        "fattn_linear_kernels_lin_b2h16n4096e64": (3 * 32 * mb, 32 * mb),
        # attention: Q, K, V read, O written (and the LSE)
        "fattn_fwd_kernel_b2h16n4096d128_causal": (3 * 32 * mb, 32 * mb),
    }
    for name, _, field in DOMINANT:
        f = _fields(name)
        total = float(f[field].split()[0])
        rd, wr = algorithmic[name]
        assert _reads(name, f) >= 0.98 * rd, name
        assert total <= 2.0 * (rd + wr), name
