"""The committed ncu summaries describe the kernels as they are.

Each summary under profiles/ records the hash of the kernel sources it was
captured on (bench.kernel_source_hash: every .cu, .cuh and .h under csrc/).
A kernel change without a new capture would leave figures that describe
other code, and the bench line's roofline.traffic would silently turn null;
this test fails instead. It also checks that each summary gives the command
that produced it, with ncu's clocks left alone."""
import glob
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def test_every_summary_is_stamped_with_the_current_kernel_sources():
    assert PROFILES
    current = bench.kernel_source_hash()
    for path in PROFILES:
        text = open(path).read()
        stamps = re.findall(r"kernel_source_sha:\s*([0-9a-f]+)", text)
        assert stamps, os.path.basename(path) + ": no kernel_source_sha"
        assert set(stamps) == {current}, (os.path.basename(path), stamps, current)


def test_every_summary_gives_its_ncu_command_with_clock_control_none():
    for path in PROFILES:
        text = open(path).read()
        if os.path.basename(path).endswith("_mlp.md"):
            continue   # per-kernel traffic figures; their command is in the DRAM-traffic summary they cite
        joined = re.sub(r"\\\n", " ", text)          # shell line continuations
        cmds = [l for l in joined.splitlines() if re.match(r"\s*ncu\s", l) and " -i " not in l]
        assert cmds, os.path.basename(path) + ": no ncu command"
        for c in cmds:
            assert "--clock-control none" in c, (os.path.basename(path), c)


def test_bench_reads_traffic_for_every_kernel_of_the_step():
    for kernel in ("bf16_kmn", "bf16_kk", "bf16_mnmn", "f32_kmn"):
        t = bench.traffic_from_profiles(kernel)
        assert t is not None and t > 1e8, kernel
