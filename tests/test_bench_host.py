"""Host logic of bench.py (no GPU): the algorithmic byte counts behind the
roofline fractions, against the workloads' own sizes, and the JSON config fields."""
import bench
from selective_state_space_115_b300 import workloads as W


def test_scan_bytes_match_the_workload_sizes():
    """u, delta (, z) read and y written at io width, B and C read, fp32 A, D, bias:
    672.5 MB for the 2.8B-like layer, 101.3 MB for the 130M-like one, 1216.5 MB for
    the long sequence (no gate), 5.2 KB for the tiny case."""
    mb = lambda name: bench.scan_bytes(W.SCAN_CONFIGS[name]) / 1e6  # noqa: E731
    assert round(mb("2p8b"), 1) == 672.5
    assert round(mb("130m"), 1) == 101.3
    assert round(mb("long"), 1) == 1216.5
    assert round(bench.scan_bytes(W.SCAN_CONFIGS["tiny"]) / 1e3, 1) == 5.2


def test_decode_bytes_per_step():
    """h read and written (2 x 83.9 MB), u, delta, z, y per channel, B, C, params."""
    assert round(bench.decode_bytes(W.DECODE_CONFIGS["decode"]) / 1e6, 1) == 178.6


def test_gradient_bytes():
    cfg = W.SCAN_CONFIGS["2p8b"]
    s = 2
    e = cfg.batch * cfg.dim * cfg.seqlen
    expect = 7 * s * e + 4 * s * cfg.dstate * cfg.batch * cfg.seqlen + \
        8 * (cfg.dim * cfg.dstate + 2 * cfg.dim)
    assert bench.bwd_bytes(cfg) == expect


def test_gradient_split_rule():
    """The library splits the gradient's sequence when fewer than two 32-channel
    CTAs per SM exist (the long sequence), not for the 2.8B-like layer."""
    assert not bench.bwd_split(W.SCAN_CONFIGS["2p8b"])
    assert bench.bwd_split(W.SCAN_CONFIGS["long"])
    assert bench.bwd_split(W.SCAN_CONFIGS["130m"])
    assert not bench.bwd_split(W.SCAN_CONFIGS["tiny"])  # too short to split


def test_config_fields():
    c = bench.bench_config("note")
    for k in ("workload", "batch", "dim", "dstate", "seqlen", "io", "l2", "parallelism"):
        assert k in c, k
    assert c["batch"] == 8 and c["dim"] == 5120 and c["seqlen"] == 2048 and c["io"] == "bf16"
    assert "larger than L2" in c["l2"]


def test_source_hash_covers_each_profiled_kernel():
    for k in bench.KERNEL_SOURCES:
        h = bench.source_sha(k)
        assert len(h) == 16 and int(h, 16) >= 0


def test_roofline_binding_term_per_workload():
    """The slowest of bytes / HBM, exps / ex2 peak and 2 FMA per update / fp32 peak:
    the exps bind the 2.8B-like and long scans, the bytes the fp32 130M-like scan
    (148 SMs, 2032 MHz, 6484.9 GB/s)."""
    r = {n: bench.scan_roofline(W.SCAN_CONFIGS[n], 1.0, 148, 2032.0, 6484.9)
         for n in ("2p8b", "long", "130m")}
    assert r["2p8b"]["bound"] == "alu" and r["long"]["bound"] == "alu"
    assert r["130m"]["bound"] == "hbm"
    assert abs(r["2p8b"]["roof_us"]["ex2"] - 139.5) < 0.5
    assert abs(r["130m"]["roof_us"]["hbm"] - 15.6) < 0.1
    # at 1 ms per scan the 2.8B-like fraction is 139.5 us / 1 ms
    assert abs(r["2p8b"]["frac"] - r["2p8b"]["roof_us"]["ex2"] / 1000.0) < 1e-9


def test_link_floor():
    """End-to-end floor: the larger of the copy-in and copy-out times at the measured
    pinned-copy peaks."""
    link = {"h2d_gbs": 50.0, "d2h_gbs": 40.0, "bytes": 1}
    f = bench.link_fraction(link, h2d=500_000_000, d2h=100_000_000, e2e_s=0.02)
    assert abs(f["floor_ms"] - 10.0) < 1e-9 and abs(f["frac"] - 0.5) < 1e-9
    assert bench.link_fraction(None, 1, 1, 1.0) is None


def test_gradient_checkpoint_pass_launches():
    # the forward's kernels form the gradient's checkpoints where AUTO runs the forward
    # on the channel kernel (one launch, or the mixed split) or the segmented plan (its
    # two passes); elsewhere the gradient kernel forms them itself (no launch)
    assert bench.bwd_ckpt_pass_launches(W.SCAN_CONFIGS["2p8b"]) == 1
    assert bench.bwd_ckpt_pass_launches(W.SCAN_CONFIGS["long"]) == 2
    assert bench.bwd_ckpt_pass_launches(W.SCAN_CONFIGS["130m"]) == 0
