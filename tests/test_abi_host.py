"""Host-side checks of the C ABI (no GPU needed, nothing is launched).

The library loads, exports every entry point that include/gdn.h declares,
sizes its buffers, and rejects bad arguments with a status before any launch.
"""

import ctypes
import os
import re

import pytest

from gated_delta_rule_06_gb300 import build, ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ops.load_library()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(gdn_\w+)\s*\(", src, re.M))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"gdn_forward", "gdn_backward", "gdn_workspace_bytes", "gdn_saved_bytes"} <= names
    for n in names:
        assert hasattr(lib, n), n


def _shape(B=1, T=130, Hk=2, Hv=4, Dk=64, Dv=32, dtype=1, has_mask=0):
    return ops.GdnShape(B, T, Hk, Hv, Dk, Dv, dtype, has_mask)


def test_sizes(lib):
    s = _shape()
    n = ctypes.c_size_t()
    assert lib.gdn_saved_bytes(ctypes.byref(s), ctypes.byref(n)) == 0
    NC = 3
    assert n.value >= 1 * 4 * NC * 64 * 32 * 4  # fp32 checkpoints
    for p in (0, 1, 2):
        assert lib.gdn_workspace_bytes(ctypes.byref(s), p, ctypes.byref(n)) == 0
        assert n.value > 0 and n.value % 256 == 0
    assert lib.gdn_workspace_bytes(ctypes.byref(s), 3, ctypes.byref(n)) == 1


@pytest.mark.parametrize("kw,code", [
    (dict(Hv=5), 2), (dict(Dk=12), 2), (dict(Dv=264), 2), (dict(T=0), 2), (dict(B=0), 2),
    (dict(dtype=7), 1), (dict(Dk=4), 2)])
def test_bad_shapes(lib, kw, code):
    s = _shape(**kw)
    n = ctypes.c_size_t()
    assert lib.gdn_saved_bytes(ctypes.byref(s), ctypes.byref(n)) == code


def _fwd(lib, s, ptr=0x1000, **over):
    args = dict(q=ptr, k=ptr, v=ptr, a=ptr, b=ptr, A_log=ptr, dt_bias=ptr, state0=None,
                mask=None, o=ptr, state_T=ptr, saved=ptr, saved_bytes=1 << 40, ws=ptr,
                ws_bytes=1 << 40)
    args.update(over)
    vp = ctypes.c_void_p
    return lib.gdn_forward(ctypes.byref(s), *[vp(args[n]) if args[n] else None for n in (
        "q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask", "o", "state_T",
        "saved")], ctypes.c_size_t(args["saved_bytes"]), vp(args["ws"]),
        ctypes.c_size_t(args["ws_bytes"]), None)


def test_forward_rejects_before_launch(lib):
    s = _shape()
    assert _fwd(lib, s, q=None) == 1                       # null input
    assert _fwd(lib, s, v=0x1008) == 4                     # misaligned
    assert _fwd(lib, s, saved_bytes=16) == 3               # saved too small
    assert _fwd(lib, s, ws_bytes=16) == 3                  # workspace too small
    assert _fwd(lib, _shape(has_mask=1)) == 1              # mask promised, not given
    assert _fwd(lib, _shape(Hv=3)) == 2                    # Hv % Hk != 0


def test_backward_rejects_before_launch(lib):
    s = _shape()
    vp = ctypes.c_void_p
    P = vp(0x1000)
    args = [P] * 7 + [None, P, ctypes.c_size_t(1 << 40), P, None] + [P] * 8 + [
        P, ctypes.c_size_t(16), None]
    assert lib.gdn_backward(ctypes.byref(s), *args) == 3   # workspace too small
    args2 = list(args)
    args2[8] = None                                        # no saved buffer
    assert lib.gdn_backward(ctypes.byref(s), *args2) == 1


def test_status_strings(lib):
    for c in range(6):
        assert lib.gdn_status_string(c).startswith(b"GDN_")


def test_lb_entry_points_reject_before_launch(lib):
    """gdn_forward_lb / gdn_backward_lb: the same host checks as the a / b form."""
    s = _shape()
    vp = ctypes.c_void_p
    P = vp(0x1000)
    big = ctypes.c_size_t(1 << 40)
    fwd = [P, P, P, P, P, None, None, P, P, P, big, P, big, None]
    assert lib.gdn_forward_lb(ctypes.byref(s), *fwd[:4], None, *fwd[5:]) == 1      # no beta
    assert lib.gdn_forward_lb(ctypes.byref(s), *fwd[:3], vp(0x1004), *fwd[4:]) == 4  # misaligned
    small = list(fwd)
    small[12] = ctypes.c_size_t(16)
    assert lib.gdn_forward_lb(ctypes.byref(s), *small) == 3                          # ws too small
    assert lib.gdn_forward_lb(ctypes.byref(_shape(Dv=12)), *fwd) == 2               # shape
    bwd = [P] * 5 + [None, P, big, P, None] + [P] * 6 + [P, ctypes.c_size_t(16), None]
    assert lib.gdn_backward_lb(ctypes.byref(s), *bwd) == 3                           # ws too small
    bwd2 = list(bwd)
    bwd2[13] = None                                                                  # no d_log_decay
    assert lib.gdn_backward_lb(ctypes.byref(s), *bwd2) == 1


def test_conv1d_update_rejects_before_launch(lib):
    vp = ctypes.c_void_p
    P = vp(0x1000)
    ok = (2, 64, 1, 4, 1)
    assert lib.gdn_causal_conv1d_update(*ok[:3], 0, ok[4], P, P, P, P, P, None) == 2  # K = 0
    assert lib.gdn_causal_conv1d_update(*ok[:3], 17, ok[4], P, P, P, P, P, None) == 2  # K > 16
    assert lib.gdn_causal_conv1d_update(0, 64, 1, 4, 1, P, P, P, P, P, None) == 2     # B = 0
    assert lib.gdn_causal_conv1d_update(*ok[:4], 9, P, P, P, P, P, None) == 1         # dtype
    assert lib.gdn_causal_conv1d_update(*ok, P, None, P, P, P, None) == 1             # null state
    assert lib.gdn_causal_conv1d_update(*ok, P, P, vp(0x1002), P, P, None) == 4       # misaligned


def test_decode_conv_rejects_before_launch(lib):
    vp = ctypes.c_void_p
    s = _shape(T=1, Dk=64, Dv=64)
    A, B_ = vp(0x100000), vp(0x200000)  # two separate conv-state buffers

    def call(shape=s, gates=1, K=4, conv_state=A, final=B_, hidden=vp(0x1000)):
        return lib.gdn_decode_conv(ctypes.byref(shape), gates, K, hidden, conv_state,
                                   vp(0x3000), final, vp(0x4000), vp(0x5000), None, None, None,
                                   None, vp(0x6000), vp(0x7000), None)

    assert call(shape=_shape(T=2, Dk=64, Dv=64)) == 2   # decode takes T == 1
    assert call(K=0) == 2 and call(K=17) == 2            # kernel length
    assert call(gates=2) == 1                            # gate form
    assert call(gates=0) == 1                            # a / b form needs A_log, dt_bias
    assert call(final=A) == 1                            # final conv state overlaps the input
    assert call(hidden=None) == 1
    assert call(hidden=vp(0x1004)) == 4                  # misaligned


def test_host_session_sizing_and_rejections(lib):
    """gdn_host_session_bytes / _create check everything before any CUDA call."""
    s = _shape()
    n_train, n_inf = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.gdn_host_session_bytes(ctypes.byref(s), 1, ctypes.byref(n_train)) == 0
    assert lib.gdn_host_session_bytes(ctypes.byref(s), 0, ctypes.byref(n_inf)) == 0
    assert n_train.value % 256 == 0 and n_inf.value % 256 == 0
    # three slots of one step's tensors at least: q, k, v and o alone per slot
    per_slot_min = (2 * 130 * 2 * 64 + 2 * 130 * 4 * 32) * 2
    assert n_inf.value >= 3 * per_slot_min
    assert n_train.value > n_inf.value
    assert lib.gdn_host_session_bytes(ctypes.byref(s), 2, ctypes.byref(n_train)) == 1
    assert lib.gdn_host_session_bytes(ctypes.byref(_shape(Hv=5)), 1, ctypes.byref(n_train)) == 2

    vp = ctypes.c_void_p
    h = vp()
    need = n_inf.value

    def create(arena=vp(0x10000000), nbytes=need, gates=0, backward=0, shape=s, out=True):
        return lib.gdn_host_session_create(ctypes.byref(shape), gates, backward, arena,
                                           nbytes, None, ctypes.byref(h) if out else None)

    assert create(arena=None) == 1              # null arena
    assert create(gates=2) == 1                 # gate form
    assert create(backward=3) == 1
    assert create(out=False) == 1               # nowhere to put the session
    assert create(shape=_shape(Dk=12)) == 2
    assert create(arena=vp(0x10000010)) == 4    # not 256-byte aligned
    assert create(nbytes=need - 256) == 3       # arena too small
    assert lib.gdn_host_step(None, None, None) == 1
    assert lib.gdn_host_session_sync(None) == 1
    assert lib.gdn_host_session_destroy(None) == 0


def test_segmented_forward_sizing_and_rejections(lib):
    """gdn_forward_segmented: segment geometry in the extra workspace size, and
    the host checks before any launch."""
    n = ctypes.c_size_t()
    s = _shape(B=2, T=64 * 10, Hk=2, Hv=4, Dk=192, Dv=128)  # NC = 10
    assert lib.gdn_segment_bytes(ctypes.byref(s), 1, ctypes.byref(n)) == 0 and n.value == 0
    # 4 requested: runs of 3 chunks, 4 segments, 3 maps / start states
    wd = 128 + 256
    assert lib.gdn_segment_bytes(ctypes.byref(s), 4, ctypes.byref(n)) == 0
    assert n.value == 3 * 2 * 4 * 192 * (wd + 128) * 4
    # above the chunk count: clamped to one chunk per segment
    assert lib.gdn_segment_bytes(ctypes.byref(s), 100, ctypes.byref(n)) == 0
    assert n.value == 9 * 2 * 4 * 192 * (wd + 128) * 4
    assert lib.gdn_segment_bytes(ctypes.byref(s), -1, ctypes.byref(n)) == 1
    a = ctypes.c_int()
    assert lib.gdn_segments_auto(ctypes.byref(s), ctypes.byref(a)) == 0 and a.value >= 1
    # fp32 has no tensor-core scan: more than one segment is unsupported
    s32 = _shape(B=1, T=64 * 10, Dk=128, Dv=128, dtype=0)
    assert lib.gdn_segment_bytes(ctypes.byref(s32), 4, ctypes.byref(n)) == 2
    vp = ctypes.c_void_p
    P = vp(0x1000)
    big = ctypes.c_size_t(1 << 40)
    fwd = [P] * 7 + [None, None, P, P, P, big, P, big, None]
    assert lib.gdn_forward_segmented(ctypes.byref(s32), 4, *fwd) == 2
    assert lib.gdn_forward_segmented(ctypes.byref(s), -2, *fwd) == 1
    small = list(fwd)
    small[14] = ctypes.c_size_t(16)
    assert lib.gdn_forward_segmented(ctypes.byref(s), 4, *small) == 3
    mis = list(fwd)
    mis[0] = vp(0x1004)
    assert lib.gdn_forward_segmented(ctypes.byref(s), 4, *mis) == 4


def test_segmented_backward_rejections(lib):
    """gdn_backward_segmented: the host checks before any launch."""
    s = _shape(B=2, T=64 * 10, Hk=2, Hv=4, Dk=128, Dv=128)
    s32 = _shape(B=1, T=64 * 10, Dk=128, Dv=128, dtype=0)
    a = ctypes.c_int()
    assert lib.gdn_backward_segments_auto(ctypes.byref(s), ctypes.byref(a)) == 0 and a.value >= 1
    assert lib.gdn_backward_segments_auto(ctypes.byref(s), None) == 1
    vp = ctypes.c_void_p
    P = vp(0x1000)
    big = ctypes.c_size_t(1 << 40)
    bwd = [P] * 9 + [big] + [P] * 10 + [P, big, None]
    assert lib.gdn_backward_segmented(ctypes.byref(s32), 4, *bwd) == 2      # no tensor-core scan
    assert lib.gdn_backward_segmented(ctypes.byref(s), -1, *bwd) == 1       # bad count
    small = list(bwd)
    small[21] = ctypes.c_size_t(16)
    assert lib.gdn_backward_segmented(ctypes.byref(s), 4, *small) == 3      # ws too small
    mis = list(bwd)
    mis[0] = vp(0x1004)
    assert lib.gdn_backward_segmented(ctypes.byref(s), 4, *mis) == 4        # misaligned
    # the backward's workspace covers its automatic count's segment buffers
    n0, n1 = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.gdn_workspace_bytes(ctypes.byref(s), 1, ctypes.byref(n1)) == 0
    assert lib.gdn_segment_bytes(ctypes.byref(s), 4, ctypes.byref(n0)) == 0 and n0.value > 0


def test_compressed_sizes_and_rejections(lib):
    """The compressed-state form (gdn_forward_compressed / _backward_compressed):
    a smaller saved buffer than the plain form at the 9B layer, and shapes or
    ranks outside its range refused."""
    n = [ctypes.c_size_t(0) for _ in range(3)]
    ref = [ctypes.byref(v) for v in n]
    nine = _shape(1, 2048, 16, 64, 192, 128)
    assert lib.gdn_compressed_bytes(ctypes.byref(nine), 16, *ref) == 0
    plain = ctypes.c_size_t()
    assert lib.gdn_saved_bytes(ctypes.byref(nine), ctypes.byref(plain)) == 0
    # the bf16 checkpoint images (64 x 32 x 192 x 128 x 2 bytes) give way to the
    # initial state and rank-16 factors of 31 boundaries (fp32)
    assert plain.value - n[0].value == 64 * 32 * 192 * 128 * 2 - 4 * 64 * (192 * 128 + 32 * 320 * 16)
    for rank in (0, 17):
        assert lib.gdn_compressed_bytes(ctypes.byref(nine), rank, *ref) == 2
    for bad in (_shape(Dk=128, Dv=128, dtype=0), _shape(Dk=128, Dv=64), _shape(Dk=96, Dv=128)):
        assert lib.gdn_compressed_bytes(ctypes.byref(bad), 8, *ref) == 2
    vp = ctypes.c_void_p
    dummy = vp(256)
    ok = _shape(Dk=128, Dv=128)
    lib.gdn_forward_compressed.argtypes = [ctypes.POINTER(ops.GdnShape), ctypes.c_int, ctypes.c_int] + \
        [vp] * 12 + [vp, ctypes.c_size_t, vp, ctypes.c_size_t, vp]
    # no omega -> invalid argument; too small a saved buffer -> workspace too small
    args = [dummy] * 5 + [dummy, dummy, None, None, dummy, dummy]
    assert lib.gdn_forward_compressed(ctypes.byref(ok), 8, 3, None, *args, dummy, 1 << 40,
                                      dummy, 1 << 40, None) == 1
    assert lib.gdn_forward_compressed(ctypes.byref(ok), 8, 3, dummy, *args, dummy, 16,
                                      dummy, 1 << 40, None) == 3
    assert lib.gdn_forward_compressed(ctypes.byref(ok), 8, 17, dummy, *args, dummy, 1 << 40,
                                      dummy, 1 << 40, None) == 2
