"""Host-side figures of bench.py that go into its JSON line (no GPU needed)."""
import bench


def test_algorithmic_bytes_of_the_wan_launch():
    # Q^, K^: 64 code bytes per token; V^: 128 channels x ceil(N/32)*32 tokens / 2;
    # three tensors' 512-byte scale atoms per 128-token tile; fp32 output
    bh, n = 40, 32760
    nt = 256
    codes = 2 * bh * n * 64 + bh * 128 * 32768 // 2
    assert bench.fwd_algorithmic_bytes(bh, n) == codes + 3 * bh * nt * 512 + bh * n * 128 * 4
    assert bench.fwd_algorithmic_bytes(bh, n) == 938_270_720  # the figure DESIGN and the profile quote
    # bf16 output halves the output bytes only
    assert bench.fwd_algorithmic_bytes(bh, n) - bench.fwd_algorithmic_bytes(bh, n, out_bytes=2) == bh * n * 128 * 2


def test_traffic_reported_only_for_the_captured_source_and_length():
    c = bench.FWD_TRAFFIC_CAPTURE
    got = bench.fwd_traffic(c["bh"], c["n"])
    if bench.kernel_fingerprint() == c["fingerprint"]:
        assert got == (c["read_bytes"], c["write_bytes"])
        # scaled per launch by B*H, null for another length
        r, w = bench.fwd_traffic(2 * c["bh"], c["n"])
        assert (r, w) == (2 * c["read_bytes"], 2 * c["write_bytes"])
        assert bench.fwd_traffic(c["bh"], c["n"] + 1) is None
    else:
        assert got is None


def test_fingerprint_ignores_comments(tmp_path, monkeypatch):
    import os
    import shutil

    src = os.path.join(bench.ROOT, "mxfp4_precision_attention_gb300", "csrc")
    dst = tmp_path / "mxfp4_precision_attention_gb300" / "csrc"
    dst.mkdir(parents=True)
    for name in bench.FWD_SOURCES:
        shutil.copy(os.path.join(src, name), dst / name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.kernel_fingerprint()
    f = dst / bench.FWD_SOURCES[0]
    f.write_text(f.read_text() + "\n// a comment only\n/* and a block comment */\n")
    assert bench.kernel_fingerprint() == base
    f.write_text(f.read_text() + "\nstatic const int extra_symbol = 1;\n")
    assert bench.kernel_fingerprint() != base
