"""The bench's workload table: names, positions (bench.py --config I) and the default workload."""
import os
import subprocess
import sys

from bwd_ssm_conv_gb300.workloads import WORKLOADS, workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_names_are_unique_and_resolve():
    names = [w.name for w in WORKLOADS]
    assert len(set(names)) == len(names) == 5
    for i, name in enumerate(names):
        assert workload(name) is WORKLOADS[i]


def test_default_workload_is_the_training_shaped_layer():
    sys.path.insert(0, ROOT)
    import bench

    w = workload(bench.DEFAULT_WORKLOAD)
    assert WORKLOADS.index(w) == 4  # --config 4 names the same workload
    assert (w.n_seqs, w.n_tok, w.n_head, w.head_dim, w.d_state, w.d_conv) == (16, 2048, 1536, 1, 16, 4)
    assert (w.io, w.chunk, w.has_z, w.has_D, w.fwd_only) == ("bf16", 256, True, True, False)


def test_command_line_lists_every_workload():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"],
                         capture_output=True, text=True, check=True, cwd=ROOT).stdout
    for w in WORKLOADS:
        assert w.name in out
