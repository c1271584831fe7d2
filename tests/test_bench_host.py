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
