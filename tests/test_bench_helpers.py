"""bench.py helpers that need no GPU: the comment-insensitive kernel-source
hash and the DRAM-traffic lookup that attaches a committed ncu figure to a
bench line only while it was taken on the current kernel source."""
import os

import pytest

from tests.conftest import ROOT


@pytest.fixture()
def bench(monkeypatch):
    import sys
    sys.path.insert(0, ROOT)
    import bench as b
    return b


def test_strip_comments_ignores_documentation_only(bench):
    code = "int f(int a) { return a + 1; }\n"
    doc = "/* a block\n comment */\n// a line comment\nint f(int a)   {\n  return a + 1; // trailing\n}\n\n"
    assert bench._strip_comments(code) == bench._strip_comments(doc)
    assert bench._strip_comments(code) != bench._strip_comments(code.replace("+ 1", "+ 2"))


def _tree(tmp_path, body):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cu").write_text(body)
    return tmp_path


def test_kernel_hash_follows_code_not_comments(bench, monkeypatch, tmp_path):
    root = _tree(tmp_path, "__global__ void k() { }\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.kernel_hash(["k.cu"])
    (root / "k.cu").write_text("// kernel k\n__global__ void k() { } /* nothing */\n")
    assert bench.kernel_hash(["k.cu"]) == h0
    (root / "k.cu").write_text("__global__ void k() { __syncthreads(); }\n")
    assert bench.kernel_hash(["k.cu"]) != h0


def test_profiled_traffic_only_for_the_profiled_source(bench, monkeypatch, tmp_path):
    root = _tree(tmp_path, "__global__ void k() { }\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    h = bench.kernel_hash(["k.cu"])
    (root / "profiles" / "row_x.md").write_text(
        f"# k\n\nkernel_source_sha256_16: {h}\ndram_bytes_per_launch: 123456\n")
    assert bench.profiled_traffic("x", ["k.cu"], prefix="row_") == 123456
    (root / "k.cu").write_text("__global__ void k() { int x = 1; }\n")   # the kernel changed
    assert bench.profiled_traffic("x", ["k.cu"], prefix="row_") is None
    assert bench.profiled_traffic("missing", ["k.cu"], prefix="row_") is None


def test_committed_profiles_are_well_formed(bench):
    """Every committed row summary that carries a traffic figure also carries
    the source hash it was taken on (16 hex digits)."""
    import re
    seen = 0
    for name in sorted(os.listdir(os.path.join(ROOT, "profiles"))):
        text = open(os.path.join(ROOT, "profiles", name), encoding="utf-8").read()
        if "dram_bytes_per_launch:" in text:
            seen += 1
            assert re.search(r"^kernel_source_sha256_16: [0-9a-f]{16}$", text, re.M), name
            assert re.search(r"^dram_bytes_per_launch: \d+$", text, re.M), name
    assert seen >= 9


def test_every_measured_row_has_a_profile_of_the_current_source(bench):
    """The bench line attaches DRAM traffic to a row only while its committed
    ncu summary was taken on the kernel source in the tree; a kernel change
    without a new capture would silently drop the figure, so every row that
    reports traffic must find one here."""
    ring = ["f32_64mib", "bf16_64mib", "weak"]
    rows = {"reduce_scatter_bf16_64mib": bench.KERNEL_SOURCES, "reduce_scatter_bidir_bf16_64mib": bench.KERNEL_SOURCES,
            "all_gather_f32_8mib": bench.KERNEL_SOURCES, "ppermute_f32_64mib": bench.KERNEL_SOURCES,
            "fused_f32_64mib": bench.FOLD_SOURCES, "psum_f32_64mib": bench.FOLD_SOURCES}
    for w in ring:
        assert bench.profiled_traffic(w) is not None, f"profiles/ring_allreduce_{w}.md"
    for name, sources in rows.items():
        assert bench.profiled_traffic(name, sources, prefix="") is not None, f"profiles/{name}.md"
