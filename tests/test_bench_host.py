"""Host-side logic of bench.py that needs no GPU: the algorithmic byte counts
the roofline divides by, and the rule that the ncu DRAM-traffic figure is
reported only for the kernel sources it was captured on."""
import bench


def test_algorithmic_bytes_of_the_workloads():
    # weights once + Q8_1 activations + fp32 outputs
    assert bench.alg_bytes(256, 1024, 1) == 256 * 4 * 54 + 32 * 36 + 4 * 256 == 57472
    assert bench.alg_bytes(5120, 6144, 1) == 5120 * 24 * 54 + 192 * 36 + 4 * 5120 == 6662912
    assert bench.alg_bytes(5120, 6144, 32) == 6635520 + 32 * 6912 + 32 * 20480


def test_traffic_reported_only_for_the_captured_sources(monkeypatch):
    digest = bench.decode_sources_digest()
    monkeypatch.setattr(bench, "DECODE_TRAFFIC", {"sha256": digest, "bytes": 123})
    assert bench.decode_traffic(None) == 123
    monkeypatch.setattr(bench, "DECODE_TRAFFIC", {"sha256": "0" * 64, "bytes": 123})
    assert bench.decode_traffic(None) is None
    assert bench.decode_traffic(456.0) == 456.0  # an explicit figure from a fresh capture


def test_digest_covers_every_decode_source(tmp_path, monkeypatch):
    base = bench.decode_sources_digest()
    assert len(base) == 64
    # Changing any one of the files changes the digest.
    for rel in bench.DECODE_SOURCES:
        src = bench.os.path.join(bench.ROOT, rel)
        copy = tmp_path / "root"
        (copy / bench.os.path.dirname(rel)).mkdir(parents=True, exist_ok=True)
        for other in bench.DECODE_SOURCES:
            dst = copy / other
            dst.parent.mkdir(parents=True, exist_ok=True)
            dst.write_bytes(open(bench.os.path.join(bench.ROOT, other), "rb").read())
        (copy / rel).write_bytes(open(src, "rb").read() + b"\n")
        monkeypatch.setattr(bench, "ROOT", str(copy))
        assert bench.decode_sources_digest() != base
        monkeypatch.setattr(bench, "ROOT", bench.os.path.dirname(bench.os.path.abspath(bench.__file__)))
