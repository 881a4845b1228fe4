"""bench.py reports a kernel's DRAM traffic from a committed ncu summary only
while the source spans the kernel is built and launched from are the ones
the summary was captured from."""
import pytest

import bench


def test_traffic_comes_from_the_matching_summary():
    t, src = bench.profiled_traffic("mha13b", "decode_bf16_persistent_kernel")
    if t is None:                           # the kernel's sources changed since the capture
        assert "changed since profiles/decode_bf16_persistent_kernel_mha13b.md" in src
    else:
        assert src == "profiles/decode_bf16_persistent_kernel_mha13b.md" and t > 600_000_000


def test_traffic_follows_the_recorded_fingerprint(monkeypatch):
    with open(bench.os.path.join(bench.ROOT, "profiles", "decode_bf16_persistent_kernel_mha13b.md")) as f:
        sha = [ln.split(": ", 1)[1].strip() for ln in f if ln.startswith("source_sha256: ")][0]
    monkeypatch.setattr(bench, "kernel_source_sha256", lambda kernel: sha)
    t, src = bench.profiled_traffic("mha13b", "decode_bf16_persistent_kernel")
    assert src == "profiles/decode_bf16_persistent_kernel_mha13b.md" and t > 600_000_000


def test_traffic_is_null_once_the_sources_change(monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_sha256", lambda kernel: "0" * 64)
    t, why = bench.profiled_traffic("mha13b", "decode_bf16_persistent_kernel")
    assert t is None and "changed" in why


def test_traffic_is_null_without_a_capture():
    t, why = bench.profiled_traffic("parallel_sampling", "decode_bf16_persistent_kernel")
    assert t is None and "no ncu capture" in why


@pytest.mark.parametrize("kernel", sorted(bench.KERNEL_SPANS))
def test_every_fingerprinted_definition_exists(kernel):
    assert len(bench.kernel_source_sha256(kernel)) == 64


def test_definition_spans_find_definitions_not_uses():
    src = """
    #define N_MAX 8
    constexpr int kBlock = 16;
    struct Thing { int a; int f() { return 1; } };
    __device__ int helper(int x) { if (x) { return 2; } return kBlock; }
    void user() { helper(3); int y = helper(4); Thing t; }
    int helper(int x);
    """
    assert [s.split()[0] for s in bench.definition_spans(src, "helper")] == ["helper(int"]
    assert bench.definition_spans(src, "helper")[0].rstrip().endswith("return kBlock; }")
    assert bench.definition_spans(src, "Thing")[0].endswith("return 1; } }")
    assert bench.definition_spans(src, "kBlock") == ["    constexpr int kBlock = 16;"]
    assert bench.definition_spans(src, "N_MAX") == ["    #define N_MAX 8"]


def test_a_change_outside_the_spans_keeps_the_fingerprint(monkeypatch, tmp_path):
    """Editing code the kernel does not depend on (here the prefill launch)
    leaves its fingerprint unchanged; editing its own body changes it."""
    import shutil
    root = tmp_path / "r"
    for f in {f for spans in bench.KERNEL_SPANS.values() for f in spans}:
        (root / f).parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(bench.os.path.join(bench.ROOT, f), root / f)
    monkeypatch.setattr(bench, "ROOT", str(root))
    k = "decode_bf16_persistent_kernel"
    before = bench.kernel_source_sha256(k)
    cu = root / bench._CSRC / "pkv.cu"
    text = cu.read_text()
    cu.write_text(text.replace("int paged_prefill_attention(", "int unused_marker = 1;\nint paged_prefill_attention(", 1))
    assert bench.kernel_source_sha256(k) == before
    kern = root / bench._CSRC / "pkv_kernels.cuh"
    t2 = kern.read_text()
    kern.write_text(t2.replace("if (i == cnt - 1) break;", "if (i == cnt - 1) { break; }", 1))
    assert bench.kernel_source_sha256(k) != before


def test_the_bench_names_kernels_the_sources_define():
    """Every kernel name the bench line can report is a __global__ of the library."""
    import re
    from paged_kv_cache_177_gb300 import workloads as W
    src = ""
    for name in ("pkv_kernels.cuh", "pkv_prefill_tc.cuh"):
        with open(bench.os.path.join(bench.ROOT, "paged_kv_cache_177_gb300", "csrc", name)) as f:
            src += f.read()
    defined = set(re.findall(r"__global__[^;{]*?\b(\w+_kernel)\s*\(", src, flags=re.S))
    names = {"decode_bf16_persistent_kernel", "decode_bf16_kernel", "lse_reduce_kernel", "kv_append_kernel",
             "move_blocks_kernel", "decode_bf16_cascade_kernel", "cascade_reduce_kernel", "prefill_tc_kernel",
             "prefill_tc_units_kernel"}
    names |= {bench.f32_kernel_name(W.spec(n, dtype="f32")) for n in W.SPECS}
    names |= set(bench.KERNEL_SPANS)
    assert names <= defined, names - defined
    assert bench.f32_kernel_name(W.spec("long_context")) == "decode_f32_tc_kernel"   # 64 / 8 heads
    assert bench.f32_kernel_name(W.spec("gqa8b")) == "decode_f32_staged_kernel"      # 32 / 8 heads
