"""bench.py reports a kernel's DRAM traffic from a committed ncu summary only
while the kernel sources are the ones the summary was captured from."""
import bench


def test_traffic_comes_from_the_matching_summary():
    t, src = bench.profiled_traffic("mha13b", "decode_bf16_persistent_kernel")
    if t is None:                           # the kernel sources changed since the capture
        assert "changed since profiles/decode_bf16_persistent_kernel_mha13b.md" in src
    else:
        assert src == "profiles/decode_bf16_persistent_kernel_mha13b.md" and t > 600_000_000


def test_traffic_follows_the_recorded_fingerprint(monkeypatch):
    with open(bench.os.path.join(bench.ROOT, "profiles", "decode_bf16_persistent_kernel_mha13b.md")) as f:
        sha = [ln.split(": ", 1)[1].strip() for ln in f if ln.startswith("source_sha256: ")][0]
    monkeypatch.setattr(bench, "kernel_sources_sha256", lambda: sha)
    t, src = bench.profiled_traffic("mha13b", "decode_bf16_persistent_kernel")
    assert src == "profiles/decode_bf16_persistent_kernel_mha13b.md" and t > 600_000_000


def test_traffic_is_null_once_the_sources_change(monkeypatch):
    monkeypatch.setattr(bench, "kernel_sources_sha256", lambda: "0" * 64)
    t, why = bench.profiled_traffic("mha13b", "decode_bf16_persistent_kernel")
    assert t is None and "changed" in why


def test_traffic_is_null_without_a_capture():
    t, why = bench.profiled_traffic("parallel_sampling", "decode_bf16_persistent_kernel")
    assert t is None and "no ncu capture" in why
