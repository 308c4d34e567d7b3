"""Host-side checks of bench.py's reporting (no GPU): the DRAM traffic the benchmark line reports is
taken from the committed ncu summary of the timed kernel only while a hash of the kernel's sources
matches the one recorded there, so the hash must cover every source file the kernel is built from."""
import os
import re

import bench

CSRC = os.path.join(bench.ROOT, "speculative_decoding_logit_gb300", "csrc")


def _local_includes(name, seen):
    if name in seen:
        return
    seen.add(name)
    with open(os.path.join(CSRC, name)) as f:
        text = f.read()
    for inc in re.findall(r'#include "([^"]+)"', text):
        if os.path.exists(os.path.join(CSRC, inc)):
            _local_includes(inc, seen)


def test_hash_covers_every_source_of_the_timed_kernel():
    seen = set()
    _local_includes("asv_jsd.cu", seen)
    assert seen <= set(bench.KERNEL_SOURCES), sorted(seen - set(bench.KERNEL_SOURCES))
    assert len(bench.kernel_source_hash()) == 16


def test_rapid_hash_covers_its_sources():
    seen = set()
    _local_includes("asv_rapid.cu", seen)
    srcs = set(bench.KERNEL_SOURCES_OF["rapid_kernel"])
    assert seen <= srcs, sorted(seen - srcs)
    assert bench.kernel_source_hash("rapid_kernel") != bench.kernel_source_hash("jsd_family")


def test_profile_records_hash_and_traffic():
    with open(os.path.join(bench.ROOT, "profiles", f"jsd_family_{bench.WORKLOAD}.md")) as f:
        text = f.read()
    assert re.search(r"kernel_source_sha256_16:\s*[0-9a-f]{16}", text)
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    # 64 requests x 3 rows x 151936 entries x 3 bf16 inputs: DRAM traffic is at least the input
    assert m and int(m.group(1)) >= 64 * 3 * 151936 * 3 * 2
