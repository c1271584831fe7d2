"""C ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects invalid arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from selective_state_space_115_b300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*SSM_API\s+[^(]*?\b(ssm_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(names) == set(binding.EXPORTED), names


def test_library_exports_every_declared_symbol():
    lib = binding.library()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.ssm_version() == 10000


def test_status_strings():
    for st in range(5):
        s = binding.status_string(st)
        assert s.startswith("SSM_"), s
    assert "unknown" in binding.status_string(99)


def test_workspace_size():
    lib = binding.library()
    assert lib.ssm_scan_fwd_workspace_size(8, 5120, 16, 2048) >= 256
    assert lib.ssm_scan_fwd_workspace_size(8, 5120, 16, 2048) % 16 == 0


def _seg_bytes(chans, n, nseg):
    rnd = lambda x: (x + 255) // 256 * 256  # noqa: E731
    return 256 + rnd(nseg * chans * n * 4) + rnd(nseg * chans * 4)


def test_workspace_size_follows_the_plan():
    """Many channels or short sequences: status words only.  A long sequence over
    few channels: room for each segment's end state and step-size sum, the segments
    sized so one-lane-per-channel CTAs fill the GPU (3 per SM; without a device the
    library assumes 148 SMs)."""
    lib = binding.library()
    ws = lib.ssm_scan_fwd_workspace_size
    # 40960 channels: channel kernel, no split; room for the mixed launch's counters
    assert ws(8, 5120, 16, 2048) == 256 + 1280
    assert ws(8, 5120, 8, 2048) == 256         # the mixed launch is dstate 16 only
    assert ws(2, 1536, 16, 2048) == 256        # few channels, short: lanes over positions
    # 1536 channels x 131072: 12 CTAs of 128 channels -> 444 // 12 = 37 segments
    assert ws(1, 1536, 16, 131072) == _seg_bytes(1536, 16, 37)
    assert ws(1, 1536, 8, 131072) == _seg_bytes(1536, 8, 37)
    # each segment keeps at least 256 positions: 8192 positions -> at most 32 segments
    assert ws(1, 128, 16, 8192) == _seg_bytes(128, 16, 32)
    algo_ws = lib.ssm_scan_fwd_algo_workspace_size
    assert algo_ws(1, 1536, 16, 131072, binding.ALGO_AUTO) == ws(1, 1536, 16, 131072)
    assert algo_ws(1, 1536, 16, 131072, binding.ALGO_CHUNK) == 256
    assert algo_ws(8, 5120, 16, 2048, binding.ALGO_CHANNEL_L2) == 256
    assert algo_ws(2, 64, 16, 2048, binding.ALGO_CHANNEL_MIXED) == 256 + 1280
    # an explicit split asks for at least two segments even when channels are many
    assert algo_ws(8, 5120, 16, 2048, binding.ALGO_SEGMENTED) == _seg_bytes(40960, 16, 2)
    # too short to split (under two 8-position chunks): status words only
    assert algo_ws(1, 4, 4, 8, binding.ALGO_SEGMENTED) == 256


def test_segmented_rejects_a_small_workspace():
    lib = binding.library()
    st = scan(lib, batch=1, dim=256, dstate=16, seqlen=4096, wsb=256,
              algo=binding.ALGO_SEGMENTED)
    assert st == binding.SSM_ERR_INVALID_ARG


# fake device addresses: validation must fail before anything dereferences them
P = 0x7F0000000000
WS = 0x7F0000100000


def scan(lib, batch=2, dim=8, dstate=16, seqlen=64, io=1, u=P, delta=P, bias=None, sp=1, A=P,
         B=P, C=P, D=None, z=None, h0=None, hl=None, y=P, ws=WS, wsb=256, algo=None):
    args = [batch, dim, dstate, seqlen, io, u, delta, bias, sp, A, B, C, D, z, h0, hl, y, ws, wsb]
    args = [ctypes.c_void_p(a) if isinstance(a, int) and i >= 5 and i not in (8, 18) else a
            for i, a in enumerate(args)]
    if algo is None:
        return lib.ssm_scan_fwd(*args, None)
    return lib.ssm_scan_fwd_algo(*args, algo, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(batch=0), binding.SSM_ERR_INVALID_ARG),
    (dict(dim=0), binding.SSM_ERR_INVALID_ARG),
    (dict(seqlen=0), binding.SSM_ERR_INVALID_ARG),
    (dict(seqlen=-5), binding.SSM_ERR_INVALID_ARG),
    (dict(dstate=0), binding.SSM_ERR_INVALID_ARG),
    (dict(dstate=32), binding.SSM_ERR_UNSUPPORTED),
    (dict(dstate=12), binding.SSM_ERR_UNSUPPORTED),
    (dict(io=7), binding.SSM_ERR_UNSUPPORTED),
    (dict(u=None), binding.SSM_ERR_INVALID_ARG),
    (dict(delta=None), binding.SSM_ERR_INVALID_ARG),
    (dict(A=None), binding.SSM_ERR_INVALID_ARG),
    (dict(B=None), binding.SSM_ERR_INVALID_ARG),
    (dict(C=None), binding.SSM_ERR_INVALID_ARG),
    (dict(y=None), binding.SSM_ERR_INVALID_ARG),
    (dict(ws=None), binding.SSM_ERR_INVALID_ARG),
    (dict(wsb=16), binding.SSM_ERR_INVALID_ARG),
    (dict(ws=WS + 8), binding.SSM_ERR_INVALID_ARG),         # workspace not 16-byte aligned
    (dict(u=P + 1), binding.SSM_ERR_INVALID_ARG),           # bf16 pointer not 2-byte aligned
    (dict(io=0, u=P + 2), binding.SSM_ERR_INVALID_ARG),     # fp32 pointer not 4-byte aligned
    (dict(A=P + 2), binding.SSM_ERR_INVALID_ARG),
    (dict(h0=P + 1), binding.SSM_ERR_INVALID_ARG),
    (dict(batch=1 << 40, dim=1 << 20), binding.SSM_ERR_INVALID_ARG),
    (dict(algo=9), binding.SSM_ERR_UNSUPPORTED),
    (dict(algo=-1), binding.SSM_ERR_UNSUPPORTED),
    # a fixed lanes-per-channel split must leave every lane at least 4 states
    (dict(algo=binding.ALGO_CHANNEL_L2, dstate=4), binding.SSM_ERR_UNSUPPORTED),
    (dict(algo=binding.ALGO_CHANNEL_L4, dstate=8), binding.SSM_ERR_UNSUPPORTED),
    (dict(algo=binding.ALGO_CHANNEL_L4, dstate=4), binding.SSM_ERR_UNSUPPORTED),
    # validation still runs first for the fixed splits
    (dict(algo=binding.ALGO_CHANNEL_L4, u=None), binding.SSM_ERR_INVALID_ARG),
])
def test_scan_validation(kw, expect):
    lib = binding.library()
    assert scan(lib, **kw) == expect


def update(lib, batch=4, dim=8, dstate=16, io=1, h=P, u=P, delta=P, bias=None, sp=1, A=P, B=P,
           C=P, D=None, z=None, y=P):
    args = [batch, dim, dstate, io, h, u, delta, bias, sp, A, B, C, D, z, y]
    args = [ctypes.c_void_p(a) if isinstance(a, int) and i >= 4 and i != 8 else a
            for i, a in enumerate(args)]
    return lib.ssm_state_update(*args, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(batch=0), binding.SSM_ERR_INVALID_ARG),
    (dict(dim=-1), binding.SSM_ERR_INVALID_ARG),
    (dict(dstate=2), binding.SSM_ERR_UNSUPPORTED),
    (dict(io=3), binding.SSM_ERR_UNSUPPORTED),
    (dict(h=None), binding.SSM_ERR_INVALID_ARG),
    (dict(u=None), binding.SSM_ERR_INVALID_ARG),
    (dict(B=None), binding.SSM_ERR_INVALID_ARG),
    (dict(y=None), binding.SSM_ERR_INVALID_ARG),
    (dict(h=P + 2), binding.SSM_ERR_INVALID_ARG),
    (dict(u=P + 1), binding.SSM_ERR_INVALID_ARG),
])
def test_update_validation(kw, expect):
    lib = binding.library()
    assert update(lib, **kw) == expect


def test_discretization_is_validated():
    lib = binding.library()
    args = [2, 8, 16, 64, 1] + [ctypes.c_void_p(P)] * 2 + [None, 1] + [ctypes.c_void_p(P)] * 3 + \
        [None] * 4 + [ctypes.c_void_p(P), ctypes.c_void_p(WS), 256]
    assert lib.ssm_scan_fwd_ex(*args, 7, binding.ALGO_AUTO, None) == binding.SSM_ERR_UNSUPPORTED
    assert lib.ssm_scan_fwd_ex(*args, -1, binding.ALGO_AUTO, None) == binding.SSM_ERR_UNSUPPORTED
    up = [4, 8, 16, 1] + [ctypes.c_void_p(P)] * 3 + [None, 1] + [ctypes.c_void_p(P)] * 3 + \
        [None, None, ctypes.c_void_p(P)]
    assert lib.ssm_state_update_ex(*up, 3, None) == binding.SSM_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,expect", [
    (dict(width=0), binding.SSM_ERR_UNSUPPORTED),
    (dict(width=9), binding.SSM_ERR_UNSUPPORTED),
    (dict(seqlen=0), binding.SSM_ERR_INVALID_ARG),
    (dict(batch=0), binding.SSM_ERR_INVALID_ARG),
    (dict(io=5), binding.SSM_ERR_UNSUPPORTED),
    (dict(x=None), binding.SSM_ERR_INVALID_ARG),
    (dict(w=None), binding.SSM_ERR_INVALID_ARG),
    (dict(out=None), binding.SSM_ERR_INVALID_ARG),
    (dict(x=P + 1), binding.SSM_ERR_INVALID_ARG),
    (dict(w=P + 2), binding.SSM_ERR_INVALID_ARG),
])
def test_conv1d_validation(kw, expect):
    lib = binding.library()
    a = dict(batch=2, dim=8, seqlen=64, width=4, io=1, x=P, w=P, bias=None, state=None, silu=1,
             out=P + 4096, state_out=None)
    a.update(kw)
    v = lambda q: None if q is None else ctypes.c_void_p(q)  # noqa: E731
    st = lib.ssm_conv1d_fwd(a["batch"], a["dim"], a["seqlen"], a["width"], a["io"], v(a["x"]),
                            v(a["w"]), v(a["bias"]), v(a["state"]), a["silu"], v(a["out"]),
                            v(a["state_out"]), None)
    assert st == expect
    if "seqlen" not in kw:
        st = lib.ssm_conv1d_update(a["batch"], a["dim"], a["width"], a["io"], v(P + 8192),
                                   v(a["x"]), v(a["w"]), v(a["bias"]), a["silu"], v(a["out"]),
                                   None)
        assert st == expect


def test_read_status_rejects_null():
    lib = binding.library()
    assert lib.ssm_read_device_status(None, None) == binding.SSM_ERR_INVALID_ARG


def _bwd_nseg(batch, dim, seqlen, segments=0, sms=148):
    """The gradient's sequence split: only when the (batch row, 32-channel) CTAs are
    fewer than two per SM, about 16 CTAs per SM, segments of >= 256 positions, a
    multiple of 8 long."""
    nblk = (seqlen + 7) // 8
    ctas = batch * ((dim + 31) // 32)
    nseg = segments
    if segments == 0:
        nseg = 1
        if ctas < 2 * sms:
            nseg = min((sms * 16 + ctas - 1) // ctas, seqlen // 256)
    nseg = max(1, min(nseg, nblk))
    seg_len = -(-seqlen // nseg)
    seg_len = -(-seg_len // 8) * 8
    return -(-seqlen // seg_len)


def _bwd_bytes(batch, dim, n, seqlen, segments=0):
    rnd = lambda x: (x + 255) // 256 * 256  # noqa: E731
    nblk = (seqlen + 7) // 8
    tiles = (dim + 31) // 32
    rows = batch * dim
    nseg = _bwd_nseg(batch, dim, seqlen, segments)
    total = (256 + rnd(nblk * rows * n * 4) + rnd(tiles * batch * 2 * n * seqlen * 4)
             + rnd(nseg * rows * n * 4) + rnd(nseg * rows * 2 * 4))
    if nseg > 1:
        total += 2 * rnd(nseg * rows * n * 4) + rnd(nseg * rows * 4)
    return total + rnd(nseg * batch * tiles)  # one fast/series flag byte per CTA


def test_bwd_workspace_size():
    """Checkpoints every 8 positions, one dB/dC partial per 32-channel CTA, the
    per-(segment, channel) dA / dD / bias sums, with a split each segment's end
    state, own adjoint and step-size sum, and one flag byte per CTA (fast or series
    coefficients); without a device the library assumes 148 SMs."""
    lib = binding.library()
    ws, wsx = lib.ssm_scan_bwd_workspace_size, lib.ssm_scan_bwd_ex_workspace_size
    for shape in ((8, 5120, 16, 2048), (1, 1536, 16, 131072), (2, 37, 8, 69), (1, 1, 4, 1),
                  (1, 64, 4, 4096)):
        assert ws(*shape) == _bwd_bytes(*shape), shape
        assert wsx(*shape, 0) == ws(*shape)
    assert _bwd_nseg(8, 5120, 2048) == 1 and _bwd_nseg(1, 1536, 131072) == 50
    for segs in (1, 2, 3, 7, 1000):
        assert wsx(2, 37, 8, 517, segs) == _bwd_bytes(2, 37, 8, 517, segs), segs
    assert wsx(2, 37, 8, 517, -1) == 256


def _bwd_call(lib, **kw):
    a = dict(batch=2, dim=8, dstate=16, seqlen=64, io=1, u=P, delta=P, bias=None, softplus=1,
             A=P, B=P, C=P, D=None, z=None, h0=None, dy=P, dh_last=None, du=P + 4096,
             ddelta=P + 8192, dA=P + 12288, dB=P + 16384, dC=P + 20480, dD=None, dz=None,
             dbias=None, dh0=None, ws=WS, ws_bytes=1 << 30, disc=0)
    a.update(kw)
    v = lambda q: None if q is None else ctypes.c_void_p(q)  # noqa: E731
    return lib.ssm_scan_bwd(a["batch"], a["dim"], a["dstate"], a["seqlen"], a["io"], v(a["u"]),
                            v(a["delta"]), v(a["bias"]), a["softplus"], v(a["A"]), v(a["B"]),
                            v(a["C"]), v(a["D"]), v(a["z"]), v(a["h0"]), v(a["dy"]),
                            v(a["dh_last"]), v(a["du"]), v(a["ddelta"]), v(a["dA"]), v(a["dB"]),
                            v(a["dC"]), v(a["dD"]), v(a["dz"]), v(a["dbias"]), v(a["dh0"]),
                            v(a["ws"]), a["ws_bytes"], a["disc"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(dstate=12), binding.SSM_ERR_UNSUPPORTED),
    (dict(io=3), binding.SSM_ERR_UNSUPPORTED),
    (dict(seqlen=0), binding.SSM_ERR_INVALID_ARG),
    (dict(batch=0), binding.SSM_ERR_INVALID_ARG),
    (dict(dy=None), binding.SSM_ERR_INVALID_ARG),
    (dict(du=None), binding.SSM_ERR_INVALID_ARG),
    (dict(dA=None), binding.SSM_ERR_INVALID_ARG),
    (dict(dC=None), binding.SSM_ERR_INVALID_ARG),
    (dict(z=P), binding.SSM_ERR_INVALID_ARG),            # z without dz
    (dict(dz=P), binding.SSM_ERR_INVALID_ARG),           # dz without z
    (dict(D=P), binding.SSM_ERR_INVALID_ARG),            # D without dD
    (dict(disc=2), binding.SSM_ERR_INVALID_ARG),
    (dict(ws=None), binding.SSM_ERR_INVALID_ARG),
    (dict(ws=WS + 16), binding.SSM_ERR_INVALID_ARG),     # not 256-byte aligned
    (dict(ws_bytes=1024), binding.SSM_ERR_INVALID_ARG),  # too small
    (dict(u=P + 1), binding.SSM_ERR_INVALID_ARG),        # misaligned bf16
    (dict(dA=P + 2), binding.SSM_ERR_INVALID_ARG),       # misaligned fp32
])
def test_bwd_validation(kw, expect):
    assert _bwd_call(binding.library(), **kw) == expect


def test_bwd_rejects_negative_segments():
    lib = binding.library()
    v = lambda q: None if q is None else ctypes.c_void_p(q)  # noqa: E731
    st = lib.ssm_scan_bwd_ex(2, 8, 16, 64, 1, v(P), v(P), None, 1, v(P), v(P), v(P), None, None,
                             None, v(P), None, v(P + 4096), v(P + 8192), v(P + 12288),
                             v(P + 16384), v(P + 20480), None, None, None, None, v(WS), 1 << 30,
                             0, -2, None)
    assert st == binding.SSM_ERR_INVALID_ARG


@pytest.mark.parametrize("ws,nbytes,limit", [
    (None, 256, 10_000_000),          # no status buffer
    (WS, 8, 10_000_000),              # too small for the status words
    (WS + 4, 256, 10_000_000),        # misaligned
    (WS, 256, 10),                    # limit below 1 us
    (WS, 256, 20_000_000_000),        # limit above 10 s
])
def test_selftest_wait_validation(ws, nbytes, limit):
    lib = binding.library()
    v = None if ws is None else ctypes.c_void_p(ws)
    assert lib.ssm_selftest_wait(v, nbytes, limit, 0, None) == binding.SSM_ERR_INVALID_ARG


def test_host_scan_workspace_size_and_validation():
    lib = binding.library()
    wsz = lib.ssm_scan_fwd_host_workspace_size
    small = wsz(8, 5120, 16, 2048, 1, 1, 0, 0, 0)
    # three staging slots of one batch row (u, delta, z, y + B, C) at least
    assert small >= 3 * (4 * 5120 * 2048 * 2 + 2 * 16 * 2048 * 2)
    assert wsz(8, 5120, 16, 2048, 1, 1, 1, 1, 0) > small  # room for h0 / h_last slices
    v = lambda q: None if q is None else ctypes.c_void_p(q)  # noqa: E731
    args = [8, 64, 16, 256, 1, v(P), v(P), None, 1, v(P), v(P), v(P), None, None, None, None,
            v(P)]
    assert lib.ssm_scan_fwd_host(*args, None, 1 << 30, 0, 0) == binding.SSM_ERR_INVALID_ARG
    assert lib.ssm_scan_fwd_host(*args, v(WS), 256, 0, 0) == binding.SSM_ERR_INVALID_ARG
    assert lib.ssm_scan_fwd_host(*args, v(WS + 16), 1 << 30, 0, 0) == \
        binding.SSM_ERR_INVALID_ARG
    bad = list(args)
    bad[5] = None  # no u
    assert lib.ssm_scan_fwd_host(*bad, v(WS), 1 << 30, 0, 0) == binding.SSM_ERR_INVALID_ARG


def test_ckpt_sizes():
    """Training-step checkpoints: one fp32 state per channel every 8 positions; the
    checkpointed gradient's workspace is the plain one without its own checkpoints."""
    lib = binding.library()
    for b, d, n, L in ((8, 5120, 16, 2048), (2, 37, 8, 69), (1, 1, 4, 1), (1, 1536, 16, 131072)):
        assert lib.ssm_scan_ckpt_bytes(b, d, n, L) == ((L + 7) // 8) * b * d * n * 4
        rnd = ((L + 7) // 8 * b * d * n * 4 + 255) // 256 * 256
        assert (lib.ssm_scan_bwd_ckpt_workspace_size(b, d, n, L, 0)
                == lib.ssm_scan_bwd_ex_workspace_size(b, d, n, L, 0) - rnd), (b, d, n, L)
    assert lib.ssm_scan_ckpt_bytes(0, 8, 16, 64) == 0


def _train_call(lib, ckpt=P + (1 << 24), ckpt_bytes=1 << 20, **kw):
    a = dict(batch=2, dim=8, dstate=16, seqlen=64, io=1, u=P, delta=P, y=P + 8192, ws=WS,
             wsb=4096)
    a.update(kw)
    v = lambda q: None if q is None else ctypes.c_void_p(q)  # noqa: E731
    return lib.ssm_scan_fwd_train(a["batch"], a["dim"], a["dstate"], a["seqlen"], a["io"],
                                  v(a["u"]), v(a["delta"]), None, 1, v(P), v(P), v(P), None,
                                  None, None, None, v(a["y"]), v(ckpt), ckpt_bytes, v(a["ws"]),
                                  a["wsb"], 0, 0, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(ckpt=None), binding.SSM_ERR_INVALID_ARG),
    (dict(ckpt=P + (1 << 24) + 4), binding.SSM_ERR_INVALID_ARG),   # not 16-byte aligned
    (dict(ckpt_bytes=8 * 2 * 8 * 16 * 4 - 4), binding.SSM_ERR_INVALID_ARG),  # one float short
    (dict(batch=0), binding.SSM_ERR_INVALID_ARG),
    (dict(u=None), binding.SSM_ERR_INVALID_ARG),
    (dict(dstate=12), binding.SSM_ERR_UNSUPPORTED),
])
def test_train_forward_validation(kw, expect):
    assert _train_call(binding.library(), **kw) == expect


def test_ckpt_gradient_rejects_null_checkpoints():
    lib = binding.library()
    v = lambda q: None if q is None else ctypes.c_void_p(q)  # noqa: E731
    st = lib.ssm_scan_bwd_ckpt(2, 8, 16, 64, 1, v(P), v(P), None, 1, v(P), v(P), v(P), None, None,
                               None, None, v(P), None, v(P + 4096), v(P + 8192), v(P + 12288),
                               v(P + 16384), v(P + 20480), None, None, None, None, v(WS),
                               1 << 30, 0, 0, None)
    assert st == binding.SSM_ERR_INVALID_ARG
