"""Host-side pieces of the benchmark: the algorithmic-byte formulas the
roofline divides by, the L2 rotation rule, and the committed ncu summaries the
bench line reads its traffic from (no GPU needed)."""
import os
import re

import numpy as np

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_metric_bytes_of_the_headline_configuration():
    # [B(K+1)V + BKV + BV] * 2 at B=256, K=5, V=128256: every target row, every
    # draft row and one stopping target row per sequence, in bf16
    B, K, V = 256, 5, 128256
    assert bench.metric_bytes(B, K, V) == (B * (K + 1) * V + B * K * V + B * V) * 2 == 788_004_864
    assert bench.sweep_bytes(B, K, V) == B * (2 * K + 1) * V * 2 == 722_337_792


def test_rotation_copies_span_twice_the_l2():
    two_l2 = 2 * bench.L2_BYTES
    for nbytes in (1, 3_000_000, 100_000_000, two_l2 - 1, two_l2, 10**10):
        c = bench.rotation_copies(nbytes)
        if nbytes < two_l2:
            assert c * nbytes >= two_l2 > (c - 1) * nbytes   # enough copies, and no more
        else:
            assert c == 1


def test_leading_true():
    f = np.array([[1, 1, 0, 1], [0, 1, 1, 1], [1, 1, 1, 1], [0, 0, 0, 0]], dtype=bool)
    np.testing.assert_array_equal(bench.leading_true(f), [2, 0, 4, 0])


def test_every_workload_names_a_committed_summary_with_its_counters():
    """Each workload's roofline reads `dram_bytes_per_launch` from its ncu
    summary under profiles/ while `source_sha` matches the kernel sources;
    the summaries named must exist and carry both keys in the expected form."""
    named = {wl.summary: wl for wl in bench.WORKLOADS.values() if wl.summary}
    assert "fused_sample_kernel_b256_v128256_k5_bf16.md" in named
    for summary, wl in named.items():
        path = os.path.join(ROOT, "profiles", summary)
        assert os.path.exists(path), summary
        text = open(path).read()
        sha = re.search(r"^source_sha: ([0-9a-f]{16})$", text, re.M)
        dram = re.search(r"^dram_bytes_per_launch: (\d+)$", text, re.M)
        assert sha and dram, summary
        assert int(dram.group(1)) > 0
        assert wl.sources, summary
        # the traffic is reported only while the sources hash to the summary's sha
        expect = int(dram.group(1)) if sha.group(1) == bench.source_sha(wl.sources) else None
        assert bench.profiled_traffic(summary, wl.sources) == expect


def test_profiles_hold_only_text_summaries():
    for name in os.listdir(os.path.join(ROOT, "profiles")):
        assert name.endswith((".md", ".txt")), name
