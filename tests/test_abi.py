"""The C-ABI library builds, loads and exports every declared entry point; host-side
validation rejects bad arguments before anything is launched (no GPU needed)."""
import ctypes
import os
import re

import pytest

from dropless_mixture_experts_top_gb300 import _build, moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return moe.lib()


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", txt)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n
    assert set(moe.EXPORTED) <= set(names)


def cfg(T=512, H=128, I=64, E=8, k=2, prec=0):
    return moe.Config(T, H, I, E, k, prec)


def test_query_workspace_sizes(L):
    rs, sv, fs, bs = moe.query_workspace(cfg())
    M = 512 * 2
    assert sv >= M * (128 * 2 * 2 + 64 * 3 * 2)   # x_perm, Y, G, U, A
    assert bs >= 256 + M * (128 * 2 * 2 + 64 * 2 * 2)  # dyw, dX, dG, dU
    assert rs >= 256 + M + (512 // 64) * 8 * 4  # status, a rank byte per slot, the per-block histograms
    offs = moe.saved_offsets(cfg())
    assert offs["x_perm"] == 0 and all(v % 256 == 0 for v in offs.values())
    assert offs["Y"] + M * 128 * 2 <= sv


@pytest.mark.parametrize("bad", [dict(H=100), dict(I=32), dict(E=0), dict(E=257), dict(k=0), dict(k=17),
                                 dict(E=4, k=5), dict(T=-1), dict(prec=7)])
def test_bad_shapes_rejected(L, bad):
    c = cfg(**bad)
    sz = ctypes.c_size_t()
    assert L.moe_query_workspace(ctypes.byref(c), ctypes.byref(sz), None, None, None) == -1


# The validation checks below pass made-up device addresses on purpose.  They run
# in a child process that sees no GPU (CUDA_VISIBLE_DEVICES=""), so even a
# validation bug could never hand those addresses to a kernel.
_VALIDATION_SCRIPT = r"""
import ctypes, sys
sys.path.insert(0, sys.argv[1])
from dropless_mixture_experts_top_gb300 import moe
L = moe.lib()
P = ctypes.c_void_p
res = {}
c = moe.Config(512, 128, 64, 8, 2, 0)
rs, sv, fs, bs = moe.query_workspace(c)
good = [0x1000 * (i + 1) for i in range(7)]
r = moe.Routing(*good)
r0 = moe.Routing(*([0] + good[1:]))
res["route_null_member"] = L.moe_route(ctypes.byref(c), P(0x10000), ctypes.byref(r0), P(0x20000), rs, None)
res["route_misaligned"] = L.moe_route(ctypes.byref(c), P(0x10004), ctypes.byref(r), P(0x20000), rs, None)
res["route_small_scratch"] = L.moe_route(ctypes.byref(c), P(0x10000), ctypes.byref(r), P(0x20000), rs - 1, None)
a = [P(0x100000 * (i + 1)) for i in range(12)]
res["fwd_small_saved"] = L.moe_forward(ctypes.byref(c), a[0], ctypes.byref(r), a[1], a[2], a[3], a[4], a[5],
                                       sv - 16, a[6], fs, None)
res["fwd_misaligned"] = L.moe_forward(ctypes.byref(c), P(0x100008), ctypes.byref(r), a[1], a[2], a[3], a[4],
                                      a[5], sv, a[6], fs, None)
res["nosave_null_out"] = L.moe_forward_nosave(ctypes.byref(c), a[0], ctypes.byref(r), a[1], a[2], a[3], None,
                                              a[5], sv, a[6], fs, None)
res["recompute_misaligned"] = L.moe_forward_recompute(ctypes.byref(c), P(0x100008), ctypes.byref(r), a[1], a[2],
                                                      a[3], a[5], sv, a[6], fs, None)
res["recompute_small_scratch"] = L.moe_forward_recompute(ctypes.byref(c), a[0], ctypes.byref(r), a[1], a[2],
                                                         a[3], a[5], sv, a[6], fs - 16, None)
res["bwd_null_dlogits"] = L.moe_backward(ctypes.byref(c), a[0], a[1], ctypes.byref(r), a[2], a[3], a[4], a[5],
                                         sv, a[6], a[7], a[8], a[9], None, None, a[10], bs, None)
res["bwd_small_scratch"] = L.moe_backward(ctypes.byref(c), a[0], a[1], ctypes.byref(r), a[2], a[3], a[4], a[5],
                                          sv, a[6], a[7], a[8], a[9], a[11], None, a[10], bs - 256, None)
print(repr(res))
"""

EXPECTED = {"route_null_member": -1, "route_misaligned": -2, "route_small_scratch": -3,
            "fwd_small_saved": -3, "fwd_misaligned": -2, "nosave_null_out": -1, "recompute_misaligned": -2,
            "recompute_small_scratch": -3, "bwd_null_dlogits": -1, "bwd_small_scratch": -3}


def test_validation_rejects_before_launch(L):
    import ast
    import subprocess
    import sys
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "-c", _VALIDATION_SCRIPT, ROOT], env=env, capture_output=True,
                         text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert ast.literal_eval(out.stdout.strip().splitlines()[-1]) == EXPECTED


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert len(moe.status_string(code)) >= 2
    assert moe.status_string(-99) == "unknown status"
    assert L.moe_timing_count() == 0


def test_fp8_shapes_and_layout(L):
    # fp8_bwd stages K in 128-byte blocks: H and I multiples of 128
    sz = ctypes.c_size_t()
    for H, I in ((192, 128), (128, 192)):
        assert L.moe_query_workspace(ctypes.byref(cfg(H=H, I=I, prec=1)), ctypes.byref(sz), None, None,
                                     None) == -1
    lay = moe.Fp8Layout()
    assert L.moe_fp8_scratch_offsets(ctypes.byref(cfg(I=128)), ctypes.byref(lay)) == -1  # bf16 config
    c = cfg(T=300, H=256, I=128, E=8, k=2, prec=1)
    q = moe.fp8_scratch_offsets(c)
    M, E, H, I = 600, 8, 256, 128
    from dropless_mixture_experts_top_gb300.synth import MoEShape
    moe_shape = MoEShape(T=300, H=H, I=I, E=E, k=2)
    Mp = q["m_pad"]
    assert Mp % 128 == 0 and Mp >= M + 127 * E
    sizes = {"pad_offsets": 4 * (E + 1), "dy_q": Mp * H, "dg_q": Mp * I, "du_q": Mp * I,
             "dy_t": H * Mp, "dg_t": I * Mp, "du_t": I * Mp}
    for n in list(sizes):
        if n != "pad_offsets":
            R, K = {"dy_q": (Mp, H), "wd_q": (E * I, H), "dg_q": (Mp, I), "du_q": (Mp, I), "wg_q": (E * H, I),
                    "wu_q": (E * H, I), "aw_t": (I, Mp), "dy_t": (H, Mp), "x_t": (H, Mp), "dg_t": (I, Mp),
                    "du_t": (I, Mp)}[n]
            seg, group = moe.sf_grouping(n, moe_shape, Mp)
            sizes[(n[:-2] if n.endswith("_q") else n) + "_sf"] = moe.sf_layout_bytes(R, K, seg, group)
            assert sizes[(n[:-2] if n.endswith("_q") else n) + "_sf"] >= R * K // 32
    spans = sorted((q[n], q[n] + b, n) for n, b in sizes.items())
    for (a0, a1, n0), (b0, b1, n1) in zip(spans, spans[1:]):
        assert a1 <= b0, (n0, n1)  # disjoint
    assert all(q[n] % 256 == 0 for n in sizes)
    _, _, _, bs = moe.query_workspace(c)
    _, _, _, bs16 = moe.query_workspace(cfg(T=300, H=256, I=128, E=8, k=2, prec=0))
    # after the status header, dX and the router gradient's partials (the bf16 backward's dy_perm,
    # dG and dU are not allocated: fp8_bwd quantises dy straight from dy and keeps dG and dU only
    # quantised)
    assert spans[0][0] >= 256 + M * H * 2 + M * 4 * 4 and spans[-1][1] <= bs
    assert bs < bs16 + sum(sizes.values()) + 256 * len(sizes)
    # w * A and x along tokens and the weights' codes live in `saved` (the forward writes
    # them), after the bf16 activations
    _, sv, _, _ = moe.query_workspace(c)
    so = moe.saved_offsets(c)
    ssz = {"aw_t": I * Mp, "aw_t_sf": moe.sf_layout_bytes(I, Mp, I, 128),
           "x_t": H * Mp, "x_t_sf": moe.sf_layout_bytes(H, Mp, H, 128),
           "wd_q": E * I * H, "wg_q": E * H * I, "wu_q": E * H * I}
    for n, (R, K, seg) in {"wd_q": (E * I, H, I), "wg_q": (E * H, I, H), "wu_q": (E * H, I, H)}.items():
        ssz[n[:-2] + "_sf"] = moe.sf_layout_bytes(R, K, seg, moe.MX_BN)
    sspans = sorted((q[n], q[n] + b, n) for n, b in ssz.items())
    for (a0, a1, n0), (b0, b1, n1) in zip(sspans, sspans[1:]):
        assert a1 <= b0, (n0, n1)
    assert all(q[n] % 256 == 0 for n in ssz)
    assert sspans[0][0] >= so["A_w"] + M * I * 2 and sspans[-1][1] <= sv


def test_router_workspace_and_shapes(L):
    f, b = moe.router_workspace(moe.Config(300, 256, 64, 16, 2, 0))
    assert f >= 512 and b >= f + 300 * 16 * 2
    # the weight gradient of a long batch is split over token segments: its fp32
    # partials are part of the backward workspace (9 of [H,E] at the 30B shape,
    # filling the 76 CTA pairs with 8 tiles each; none below 2048 tokens)
    T, H, E = 16384, 2048, 128
    _, b_split = moe.router_workspace(moe.Config(T, H, 64, E, 8, 0))
    assert b_split >= 9 * H * E * 4 + T * E * 2
    _, b_short = moe.router_workspace(moe.Config(2047, H, 64, E, 8, 0))
    assert b_short < H * E * 4 + 2047 * E * 2 + 16384
    for bad in (dict(E=12), dict(E=4), dict(H=96)):  # E % 8, E >= 8, H % 64
        c = moe.Config(300, bad.get("H", 256), 64, bad.get("E", 16), 2, 0)
        assert L.moe_router_workspace(ctypes.byref(c), None, None) == -1


def test_mxfp8_shapes_and_forward_layout(L):
    sz = ctypes.c_size_t()
    for H, I in ((192, 128), (128, 192)):  # K staged in 128-byte blocks
        assert L.moe_query_workspace(ctypes.byref(cfg(H=H, I=I, prec=2)), ctypes.byref(sz), None, None,
                                     None) == -1
    lay = moe.Mx8FwdLayout()
    for prec in (0, 1):
        assert L.moe_mxfp8_forward_offsets(ctypes.byref(cfg(I=128, prec=prec)), ctypes.byref(lay)) == -1
    T, H, I, E, k = 300, 256, 128, 8, 2
    c = cfg(T=T, H=H, I=I, E=E, k=k, prec=2)
    f = moe.mxfp8_forward_offsets(c)
    M = T * k
    Mp = f["m_pad"]
    assert Mp % 128 == 0 and Mp >= M + 127 * E
    from dropless_mixture_experts_top_gb300.synth import MoEShape
    shape = MoEShape(T=T, H=H, I=I, E=E, k=k)
    sizes = {"pad_offsets": 4 * (E + 1), "x_q": Mp * H, "a_q": Mp * I, "wgu_q": E * 2 * I * H, "wdt_q": E * H * I}
    for n, (R, K) in {"x_q": (Mp, H), "a_q": (Mp, I), "wgu_q": (E * 2 * I, H), "wdt_q": (E * H, I)}.items():
        seg, group = moe.sf_grouping(n, shape, Mp)
        sizes[n[:-2] + "_sf"] = moe.sf_layout_bytes(R, K, seg, group)
        assert sizes[n[:-2] + "_sf"] >= R * K // 32
    spans = sorted((f[n], f[n] + b, n) for n, b in sizes.items())
    for (a0, a1, n0), (b0, b1, n1) in zip(spans, spans[1:]):
        assert a1 <= b0, (n0, n1)
    assert all(f[n] % 256 == 0 for n in sizes)
    _, _, fs, bs = moe.query_workspace(c)
    assert spans[0][0] >= 256 and spans[-1][1] <= fs  # after the status header, inside the forward scratch
    # the backward's weight codes are written by the forward into `saved`, after the activations
    rs, sv, _, _ = moe.query_workspace(c)
    so = moe.saved_offsets(c)
    wsz = {"bwd_wd_q": E * I * H, "bwd_wg_q": E * H * I, "bwd_wu_q": E * H * I}
    for n, (R, K, seg) in {"bwd_wd_q": (E * I, H, I), "bwd_wg_q": (E * H, I, H), "bwd_wu_q": (E * H, I, H)}.items():
        wsz[n[:-2] + "_sf"] = moe.sf_layout_bytes(R, K, seg, moe.MX_BN)
    wspans = sorted((f[n], f[n] + b, n) for n, b in wsz.items())
    for (a0, a1, n0), (b0, b1, n1) in zip(wspans, wspans[1:]):
        assert a1 <= b0, (n0, n1)
    assert wspans[0][0] >= so["A_w"] + M * I * 2 and wspans[-1][1] <= sv
    # the backward is fp8_bwd's, reading the same weight codes from `saved`
    q = moe.fp8_scratch_offsets(c)
    assert all(q[n] == f["bwd_" + n] for n in ("wd_q", "wd_sf", "wg_q", "wg_sf", "wu_q", "wu_sf"))
    c1 = cfg(T=T, H=H, I=I, E=E, k=k, prec=1)
    assert bs == moe.query_workspace(c1)[3]
