"""Host-side logic of bench.py that needs no GPU: profile validity and launch counting."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

KERNEL = """// header comment
__global__ void k(float* y) {  /* block
  comment */
  y[threadIdx.x] = 1.f;  // trailing
}
"""


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    csrc = tmp_path / "state_space_model_02_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def write_kernel(root, text):
    (root / "state_space_model_02_gb300" / "csrc" / "chunk_scan_tc.cu").write_text(text)


def test_digest_ignores_comments_and_whitespace(fake_root):
    write_kernel(fake_root, KERNEL)
    d0 = bench.source_digest("chunk_scan")
    write_kernel(fake_root, KERNEL.replace("// header comment", "// reworded header\n\n")
                 .replace("/* block\n  comment */", "/* other */").replace("  y[", "\ty["))
    assert bench.source_digest("chunk_scan") == d0


def test_digest_changes_with_the_code(fake_root):
    write_kernel(fake_root, KERNEL)
    d0 = bench.source_digest("chunk_scan")
    write_kernel(fake_root, KERNEL.replace("1.f", "2.f"))
    assert bench.source_digest("chunk_scan") != d0


def test_profiled_traffic_only_while_the_kernel_is_unchanged(fake_root):
    write_kernel(fake_root, KERNEL)
    summary = fake_root / "profiles" / "chunk_scan__some_workload.txt"
    summary.write_text("# ncu summary\nsource_sha256_16 = %s\ndram_bytes_per_launch = 1234\n"
                       % bench.source_digest("chunk_scan"))
    assert bench.profiled_traffic("chunk_scan", "some_workload") == 1234.0
    assert bench.profiled_traffic("chunk_scan", "other_workload") is None
    write_kernel(fake_root, KERNEL.replace("1.f", "3.f"))
    assert bench.profiled_traffic("chunk_scan", "some_workload") is None


@pytest.mark.parametrize("dstate,chunk,plan,launches", [
    (128, 256, 3, 1),   # one tensor-core launch
    (256, 256, 3, 2),   # the readout, then chunk_scan
    (512, 256, 3, 2),
    (192, 128, 3, 2),
    (512, 256, 1, 1),   # CUDA-core chunk_scan: one launch whatever the state size
    (64, 64, 0, 1),
])
def test_scan_launch_count(dstate, chunk, plan, launches):
    assert bench.scan_launches({"dstate": dstate, "chunk": chunk}, plan) == launches


def test_step_kernels_follow_the_plan():
    assert bench.step_kernels(3) == ("chunk_cumsum", "chunk_state", "state_passing", "chunk_scan")
    assert bench.step_kernels(7) == ("chunk_cumsum", "fwd_pass_state", "chunk_scan")
    assert bench.step_kernels(0) == bench.KERNELS
    by, fl = bench.algorithmic(dict(batch=2, seqlen=8192, nheads=80, headdim=64, dstate=128, ngroups=1,
                                    chunk=256, io_dtype="bf16", init=False))
    # the fused kernel moves chunk_state's inputs and state_passing's outputs, not S
    st = 2 * 32 * 80 * 64 * 128 * 2
    assert by["fwd_pass_state"] == by["chunk_state"] + 2 * 80 * 64 * 128 * 4
    # what fusing saves: S written and read back, and state_passing's own cs2 and extra state bytes
    assert by["chunk_state"] + by["state_passing"] - by["fwd_pass_state"] == \
        2 * st + 2 * 80 * 32 * 4 + 2 * 80 * 64 * 128 * 4
