"""The seeded synthetic inputs (no GPU): shapes, value recipes and determinism of
selective_state_space_115_b300.workloads, and the binding's argument checks that
run before any device call."""
import numpy as np
import pytest

from selective_state_space_115_b300 import workloads as W


def test_scan_recipe_2p8b():
    """B8 D5120 N16 L2048 bf16 with the gate: A[d,n] = -(n+1); the per-channel bias is
    the inverse softplus of dt log-uniform in [1e-3, 1e-1]; u, delta, B, C, z ~ N(0,1)."""
    cfg = W.SCAN_CONFIGS["2p8b"]
    assert (cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen, cfg.io, cfg.gate) == \
        (8, 5120, 16, 2048, W.BF16, True)
    x = W.make_scan_inputs(cfg, seed=0, batch=1, dim=256, seqlen=512)
    assert np.array_equal(x["A"], -np.tile(np.arange(1, 17, dtype=np.float32), (256, 1)))
    dt = np.log1p(np.exp(x["delta_bias"].astype(np.float64)))
    assert dt.min() >= 1e-3 * 0.999 and dt.max() <= 1e-1 * 1.001
    for k in ("u", "delta", "B", "C", "z"):
        v = W.to_f64(x[k], W.BF16)
        assert abs(v.mean()) < 0.05 and abs(v.std() - 1.0) < 0.05, k
    assert x["u"].dtype == np.uint16 and x["A"].dtype == np.float32


def test_tiny_recipe():
    """Tiny: B1 D4 N4 L64 fp32, bias 0, D = 1, no gate."""
    cfg = W.SCAN_CONFIGS["tiny"]
    x = W.make_scan_inputs(cfg, seed=0)
    assert x["u"].shape == (1, 4, 64) and x["z"] is None
    assert np.all(x["delta_bias"] == 0) and np.all(x["D"] == 1)


def test_inputs_are_deterministic_per_seed():
    cfg = W.SCAN_CONFIGS["130m"]
    a = W.make_scan_inputs(cfg, seed=3, batch=1, dim=32, seqlen=64)
    b = W.make_scan_inputs(cfg, seed=3, batch=1, dim=32, seqlen=64)
    c = W.make_scan_inputs(cfg, seed=4, batch=1, dim=32, seqlen=64)
    for k in a:
        if a[k] is not None:
            assert np.array_equal(a[k], b[k]), k
    assert not np.array_equal(a["u"], c["u"])
    g1 = W.make_scan_grads(cfg, seed=3, batch=1, dim=32, seqlen=64)
    g2 = W.make_scan_grads(cfg, seed=3, batch=1, dim=32, seqlen=64)
    assert np.array_equal(g1["dy"], g2["dy"]) and g1["dh_last"].shape == (1, 32, 16)


def test_decode_recipe():
    cfg = W.DECODE_CONFIGS["decode"]
    assert (cfg.batch, cfg.dim, cfg.dstate, cfg.steps) == (256, 5120, 16, 1024)
    st = W.make_decode_static(cfg, seed=0, batch=4, dim=64)
    assert abs(st["h"].std() - 0.1) < 0.01
    s0 = W.make_decode_step(cfg, 0, seed=0, batch=4, dim=64)
    s1 = W.make_decode_step(cfg, 1, seed=0, batch=4, dim=64)
    assert not np.array_equal(s0["u"], s1["u"])


def test_bf16_encoding_rounds_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5], dtype=np.float32)
    bits = W.f32_to_bf16_bits(x)
    back = W.bf16_bits_to_f32(bits)
    assert back[0] == 1.0 and back[1] == 1.0           # tie to even
    assert back[2] == 1.0 + 2 ** -6                     # tie to even (up)
    assert back[3] == -2.5


def test_binding_rejects_host_tensors_for_the_device_scan():
    import torch
    from selective_state_space_115_b300 import binding
    u = torch.zeros(1, 2, 8)
    with pytest.raises(binding.SsmError):
        binding.scan_fwd(u, u, torch.zeros(2, 4), torch.zeros(1, 4, 8), torch.zeros(1, 4, 8))


def test_binding_checks_host_scan_arguments_first():
    import torch
    from selective_state_space_115_b300 import binding
    u = torch.zeros(1, 2, 8)
    with pytest.raises(binding.SsmError):  # B has the wrong shape
        binding.scan_fwd_host(u, u, torch.zeros(2, 4), torch.zeros(1, 3, 8),
                              torch.zeros(1, 4, 8))
    with pytest.raises(binding.SsmError):  # A has the wrong dtype
        binding.scan_fwd_host(u, u, torch.zeros(2, 4, dtype=torch.float64),
                              torch.zeros(1, 4, 8), torch.zeros(1, 4, 8))
