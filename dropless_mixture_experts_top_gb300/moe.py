"""Thin ctypes binding of libmoe_gb300.so (include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  There is no fallback:
if the library is missing or the GPU is not an sm_103a part, calls raise.

Low-level functions mirror the C names (query_workspace, route, forward,
backward, get_device_status, status_string, timing_*).  `MoELayer` bundles the
buffers one configuration needs.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

MOE_OK = 0
PRECISIONS = {"bf16": 0, "fp8_bwd": 1, "mxfp8": 2}
DEV_NONFINITE_LOGIT = 0x1
DEV_WAIT_TIMEOUT = 0x2

_lib = None

EXPORTED = [
    "moe_query_workspace", "moe_saved_offsets", "moe_fp8_scratch_offsets", "moe_mxfp8_forward_offsets",
    "moe_route",
    "moe_route_static_scratch", "moe_forward", "moe_forward_nosave", "moe_forward_recompute", "moe_backward",
    "moe_get_device_status",
    "moe_status_string", "moe_timing_attach", "moe_timing_count", "moe_timing_label",
    "moe_selftest_wait_timeout", "moe_router_workspace", "moe_router_forward", "moe_router_backward",
]


class Config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("precision", ctypes.c_int32)]


class Routing(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("topk_idx", "topk_w", "counts", "offsets", "row_of_slot", "slot_of_row", "w_row")]


class SavedLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("x_perm", "G", "U", "A", "Y", "A_w")]


class Fp8Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "m_pad", "pad_offsets", "dy_q", "dy_sf", "wd_q", "wd_sf", "dg_q", "dg_sf", "du_q", "du_sf",
        "wg_q", "wg_sf", "wu_q", "wu_sf", "aw_t", "aw_t_sf", "dy_t", "dy_t_sf", "x_t", "x_t_sf",
        "dg_t", "dg_t_sf", "du_t", "du_t_sf")]


class Mx8FwdLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "m_pad", "pad_offsets", "x_q", "x_sf", "a_q", "a_sf", "wgu_q", "wgu_sf", "wdt_q", "wdt_sf",
        "bwd_wd_q", "bwd_wd_sf", "bwd_wg_q", "bwd_wg_sf", "bwd_wu_q", "bwd_wu_sf")]


class MoEError(RuntimeError):
    def __init__(self, what, code):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


def library_path() -> str:
    return _build.LIB


def lib():
    """Load the in-tree library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(path)
        P, sz = ctypes.c_void_p, ctypes.c_size_t
        L.moe_query_workspace.argtypes = [P, P, P, P, P]
        L.moe_saved_offsets.argtypes = [P, P]
        L.moe_fp8_scratch_offsets.argtypes = [P, P]
        L.moe_mxfp8_forward_offsets.argtypes = [P, P]
        L.moe_route.argtypes = [P, P, P, P, sz, P]
        L.moe_forward.argtypes = [P, P, P, P, P, P, P, P, sz, P, sz, P]
        L.moe_forward_nosave.argtypes = [P, P, P, P, P, P, P, P, sz, P, sz, P]
        L.moe_forward_recompute.argtypes = [P, P, P, P, P, P, P, sz, P, sz, P]
        L.moe_backward.argtypes = [P, P, P, P, P, P, P, P, sz, P, P, P, P, P, P, P, sz, P]
        L.moe_get_device_status.argtypes = [P, P, P]
        L.moe_selftest_wait_timeout.argtypes = [P, P]
        L.moe_selftest_wait_timeout.restype = ctypes.c_int
        L.moe_router_workspace.argtypes = [P, P, P]
        L.moe_router_forward.argtypes = [P, P, P, P, P, sz, P]
        L.moe_router_backward.argtypes = [P, P, P, P, P, P, P, sz, P]
        for f in ("moe_router_workspace", "moe_router_forward", "moe_router_backward"):
            getattr(L, f).restype = ctypes.c_int
        L.moe_status_string.argtypes = [ctypes.c_int]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_timing_attach.argtypes = [P, ctypes.c_int32]
        L.moe_timing_count.argtypes = []
        L.moe_timing_count.restype = ctypes.c_int32
        L.moe_timing_label.argtypes = [ctypes.c_int32]
        L.moe_timing_label.restype = ctypes.c_char_p
        for f in ("moe_query_workspace", "moe_saved_offsets", "moe_fp8_scratch_offsets",
                  "moe_mxfp8_forward_offsets", "moe_route", "moe_forward", "moe_backward",
                  "moe_get_device_status", "moe_timing_attach"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def _check(code, what):
    if code != MOE_OK:
        raise MoEError(what, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_config(shape, precision="bf16") -> Config:
    return Config(int(shape.T), int(shape.H), int(shape.I), int(shape.E), int(shape.k),
                  PRECISIONS[precision] if isinstance(precision, str) else int(precision))


def query_workspace(cfg: Config):
    out = [ctypes.c_size_t() for _ in range(4)]
    _check(lib().moe_query_workspace(ctypes.byref(cfg), *[ctypes.byref(o) for o in out]),
           "moe_query_workspace")
    return tuple(int(o.value) for o in out)


def saved_offsets(cfg: Config) -> dict:
    lay = SavedLayout()
    _check(lib().moe_saved_offsets(ctypes.byref(cfg), ctypes.byref(lay)), "moe_saved_offsets")
    return {n: int(getattr(lay, n)) for n, _ in SavedLayout._fields_}


def fp8_scratch_offsets(cfg: Config) -> dict:
    lay = Fp8Layout()
    _check(lib().moe_fp8_scratch_offsets(ctypes.byref(cfg), ctypes.byref(lay)),
           "moe_fp8_scratch_offsets")
    return {n: int(getattr(lay, n)) for n, _ in Fp8Layout._fields_}


def mxfp8_forward_offsets(cfg: Config) -> dict:
    lay = Mx8FwdLayout()
    _check(lib().moe_mxfp8_forward_offsets(ctypes.byref(cfg), ctypes.byref(lay)),
           "moe_mxfp8_forward_offsets")
    return {n: int(getattr(lay, n)) for n, _ in Mx8FwdLayout._fields_}


MX_BN = 192  # N extent of an MXFP8 GEMM tile: B-operand scales are grouped by it


def sf_grouping(base: str, shape, m_pad: int):
    """(segment rows, group rows) of a quantised operand's scale atoms."""
    if base in ("wd_q",):
        return shape.I, MX_BN
    if base in ("wg_q", "wu_q"):
        return shape.H, MX_BN
    if base == "dy_t":
        return shape.H, MX_BN
    if base in ("dg_t", "du_t"):
        return shape.I, MX_BN
    if base == "wgu_q":
        return 2 * shape.I, MX_BN
    if base == "wdt_q":
        return shape.H, MX_BN
    rows = {"dy_q": m_pad, "dg_q": m_pad, "du_q": m_pad, "aw_t": shape.I, "x_t": shape.H,
            "x_q": m_pad, "a_q": m_pad}[base]
    return rows, 128


def sf_layout_bytes(rows: int, K: int, seg: int, group: int) -> int:
    nseg, gps, apg = -(-rows // seg), -(-seg // group), -(-group // 128)
    return nseg * gps * apg * (K // 128) * 512


def make_routing(r: dict) -> Routing:
    return Routing(*[r[n].data_ptr() for n, _ in Routing._fields_])


def route(cfg, logits, routing: dict, scratch, stream=None):
    rt = make_routing(routing)
    _check(lib().moe_route(ctypes.byref(cfg), _ptr(logits), ctypes.byref(rt), _ptr(scratch),
                           scratch.numel(), _stream(stream)), "moe_route")


def forward(cfg, x, routing: dict, W_gate, W_up, W_down, out, saved, scratch, stream=None, save=True):
    """moe_forward, or moe_forward_nosave when save is False (out only)."""
    rt = make_routing(routing)
    fn, name = (lib().moe_forward, "moe_forward") if save else (lib().moe_forward_nosave, "moe_forward_nosave")
    _check(fn(ctypes.byref(cfg), _ptr(x), ctypes.byref(rt), _ptr(W_gate), _ptr(W_up), _ptr(W_down), _ptr(out),
              _ptr(saved), saved.numel(), _ptr(scratch), scratch.numel(), _stream(stream)), name)


def forward_recompute(cfg, x, routing: dict, W_gate, W_up, W_down, saved, scratch, stream=None):
    rt = make_routing(routing)
    _check(lib().moe_forward_recompute(ctypes.byref(cfg), _ptr(x), ctypes.byref(rt), _ptr(W_gate), _ptr(W_up),
                                       _ptr(W_down), _ptr(saved), saved.numel(), _ptr(scratch), scratch.numel(),
                                       _stream(stream)), "moe_forward_recompute")


def backward(cfg, dy, x, routing: dict, W_gate, W_up, W_down, saved, dx, dW_gate, dW_up, dW_down,
             d_logits, d_topk_w, scratch, stream=None):
    rt = make_routing(routing)
    _check(lib().moe_backward(ctypes.byref(cfg), _ptr(dy), _ptr(x), ctypes.byref(rt), _ptr(W_gate),
                              _ptr(W_up), _ptr(W_down), _ptr(saved), saved.numel(), _ptr(dx),
                              _ptr(dW_gate), _ptr(dW_up), _ptr(dW_down), _ptr(d_logits),
                              _ptr(d_topk_w), _ptr(scratch), scratch.numel(), _stream(stream)),
           "moe_backward")


def get_device_status(scratch, stream=None) -> int:
    code = ctypes.c_int32()
    rc = lib().moe_get_device_status(_ptr(scratch), _stream(stream), ctypes.byref(code))
    if rc not in (MOE_OK, -6):
        _check(rc, "moe_get_device_status")
    return int(code.value)


def router_workspace(cfg: Config):
    f, b = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().moe_router_workspace(ctypes.byref(cfg), ctypes.byref(f), ctypes.byref(b)),
           "moe_router_workspace")
    return int(f.value), int(b.value)


class Router:
    """The router projection logits = x . W_r (bf16 in, fp32 logits) and its
    backward, over scratch buffers sized for one configuration."""

    def __init__(self, shape, device="cuda"):
        self.shape = shape
        self.cfg = make_config(shape)
        fs, bs = router_workspace(self.cfg)
        self.fwd_scratch = torch.empty(fs, dtype=torch.uint8, device=device)
        self.bwd_scratch = torch.empty(bs, dtype=torch.uint8, device=device)
        self.device = device

    def forward(self, x, W_r, logits=None, stream=None):
        if logits is None:
            logits = torch.empty((self.shape.T, self.shape.E), dtype=torch.float32, device=self.device)
        _check(lib().moe_router_forward(ctypes.byref(self.cfg), _ptr(x), _ptr(W_r), _ptr(logits),
                                        _ptr(self.fwd_scratch), self.fwd_scratch.numel(), _stream(stream)),
               "moe_router_forward")
        return logits

    def backward(self, x, W_r, d_logits, dx, dW_r=None, stream=None):
        """dx (bf16 [T,H]) is updated in place; returns dW_r (fp32 [H,E])."""
        if dW_r is None:
            dW_r = torch.empty((self.shape.H, self.shape.E), dtype=torch.float32, device=self.device)
        _check(lib().moe_router_backward(ctypes.byref(self.cfg), _ptr(x), _ptr(W_r), _ptr(d_logits), _ptr(dx),
                                         _ptr(dW_r), _ptr(self.bwd_scratch), self.bwd_scratch.numel(),
                                         _stream(stream)), "moe_router_backward")
        return dW_r

    def status(self, stream=None) -> dict:
        return {n: get_device_status(b, stream) for n, b in (("forward", self.fwd_scratch),
                                                             ("backward", self.bwd_scratch))}


def selftest_wait_timeout(status, stream=None):
    """Launch the bounded-wait diagnostic; `status` is a device int32 tensor."""
    _check(lib().moe_selftest_wait_timeout(_ptr(status), _stream(stream)), "moe_selftest_wait_timeout")


def timing_attach(events):
    """events: list of torch.cuda.Event (enable_timing=True), two per kernel.
    torch creates the CUDA event object lazily, so each one is recorded once here
    to make its handle valid."""
    global _timing_keep
    if events is None:
        _check(lib().moe_timing_attach(None, 0), "moe_timing_attach")
        _timing_keep = None
        return
    for e in events:
        e.record()
    torch.cuda.synchronize()
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _timing_keep = arr
    _check(lib().moe_timing_attach(arr, len(events) // 2), "moe_timing_attach")


_timing_keep = None


def timing_count() -> int:
    return int(lib().moe_timing_count())


def timing_label(i: int) -> str:
    s = lib().moe_timing_label(int(i))
    return s.decode() if s else ""


def bf16_view(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.bfloat16)


class MoELayer:
    """Device buffers for one configuration, and the three calls over them."""

    def __init__(self, shape, precision="bf16", device="cuda"):
        self.shape = shape
        self.cfg = make_config(shape, precision)
        self.device = torch.device(device)
        T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
        rs, sv, fs, bs = query_workspace(self.cfg)
        dev = self.device
        i32, f32, u8 = torch.int32, torch.float32, torch.uint8
        self.routing = {
            "topk_idx": torch.empty((T, k), dtype=i32, device=dev),
            "topk_w": torch.empty((T, k), dtype=f32, device=dev),
            "counts": torch.empty((E,), dtype=i32, device=dev),
            "offsets": torch.empty((E + 1,), dtype=i32, device=dev),
            "row_of_slot": torch.empty((T, k), dtype=i32, device=dev),
            "slot_of_row": torch.empty((T * k,), dtype=i32, device=dev),
            "w_row": torch.empty((T * k,), dtype=f32, device=dev),
        }
        self.route_scratch = torch.empty(rs, dtype=u8, device=dev)
        self.saved = torch.empty(sv, dtype=u8, device=dev)
        self.fwd_scratch = torch.empty(fs, dtype=u8, device=dev)
        self.bwd_scratch = torch.empty(bs, dtype=u8, device=dev)
        self.saved_offsets = saved_offsets(self.cfg)

    def saved_tensor(self, name):
        T, H, I, k = self.shape.T, self.shape.H, self.shape.I, self.shape.k
        cols = H if name in ("x_perm", "Y") else I
        off = self.saved_offsets[name]
        n = T * k * cols
        return self.saved[off:off + 2 * n].view(torch.int16).view(T * k, cols)

    def fp8_tensor(self, name):
        """A quantised operand left in the backward scratch (the fp8 modes), or for
        aw_t (w * A along tokens), x_t (x along tokens) and the weights' wd_q, wg_q,
        wu_q (all written by the forward) in `saved`: uint8 codes [rows, K] for *_q and *_t, the raw
        scale-atom bytes for *_sf, int32 [E+1] for pad_offsets."""
        lay = fp8_scratch_offsets(self.cfg)
        s = self.shape
        Mp = lay["m_pad"]
        rows_k = {"dy_q": (Mp, s.H), "wd_q": (s.E * s.I, s.H), "dg_q": (Mp, s.I), "du_q": (Mp, s.I),
                  "wg_q": (s.E * s.H, s.I), "wu_q": (s.E * s.H, s.I), "aw_t": (s.I, Mp),
                  "dy_t": (s.H, Mp), "x_t": (s.H, Mp), "dg_t": (s.I, Mp), "du_t": (s.I, Mp)}
        off = lay[name]
        in_saved = name.startswith(("aw_t", "x_t", "wd_", "wg_", "wu_"))  # written by the forward
        buf = self.saved if in_saved else self.bwd_scratch
        if name == "pad_offsets":
            return buf[off:off + 4 * (s.E + 1)].view(torch.int32)
        if name.endswith("_sf"):
            base = name[:-3] + "_q" if name[:-3] + "_q" in rows_k else name[:-3]
            R, K = rows_k[base]
            seg, group = sf_grouping(base, s, Mp)
            return buf[off:off + sf_layout_bytes(R, K, seg, group)]
        R, K = rows_k[name]
        return buf[off:off + R * K].view(R, K)

    def fwd_fp8_tensor(self, name):
        """A quantised operand of the mxfp8 forward: in the forward scratch, or for
        bwd_* (the backward's weight operands) in `saved`.  uint8 codes [rows, K]
        for *_q, raw scale-atom bytes for *_sf, int32 [E+1] for pad_offsets."""
        lay = mxfp8_forward_offsets(self.cfg)
        s = self.shape
        Mp = lay["m_pad"]
        rows_k = {"x_q": (Mp, s.H), "a_q": (Mp, s.I), "wgu_q": (s.E * 2 * s.I, s.H), "wdt_q": (s.E * s.H, s.I),
                  "bwd_wd_q": (s.E * s.I, s.H), "bwd_wg_q": (s.E * s.H, s.I), "bwd_wu_q": (s.E * s.H, s.I)}
        buf = self.saved if name.startswith("bwd_") else self.fwd_scratch
        off = lay[name]
        if name == "pad_offsets":
            return buf[off:off + 4 * (s.E + 1)].view(torch.int32)
        if name.endswith("_sf"):
            base = name[:-3] + "_q"
            R, K = rows_k[base]
            seg, group = sf_grouping(base[4:] if base.startswith("bwd_") else base, s, Mp)
            return buf[off:off + sf_layout_bytes(R, K, seg, group)]
        R, K = rows_k[name]
        return buf[off:off + R * K].view(R, K)

    def route(self, logits, stream=None):
        route(self.cfg, logits, self.routing, self.route_scratch, stream)

    def forward(self, x, W_gate, W_up, W_down, out=None, stream=None, save=True):
        """save=False: a checkpointed layer's first pass (out only; call recompute
        before backward)."""
        if out is None:
            out = torch.empty((self.shape.T, self.shape.H), dtype=torch.int16, device=self.device)
        forward(self.cfg, x, self.routing, W_gate, W_up, W_down, out, self.saved, self.fwd_scratch, stream,
                save=save)
        return out

    def recompute(self, x, W_gate, W_up, W_down, stream=None):
        """What backward reads, rebuilt from the same inputs (no out)."""
        forward_recompute(self.cfg, x, self.routing, W_gate, W_up, W_down, self.saved, self.fwd_scratch, stream)

    def backward(self, dy, x, W_gate, W_up, W_down, grads=None, stream=None):
        s = self.shape
        dev = self.device
        if grads is None:
            grads = {
                "dx": torch.empty((s.T, s.H), dtype=torch.int16, device=dev),
                "dW_gate": torch.empty((s.E, s.H, s.I), dtype=torch.int16, device=dev),
                "dW_up": torch.empty((s.E, s.H, s.I), dtype=torch.int16, device=dev),
                "dW_down": torch.empty((s.E, s.I, s.H), dtype=torch.int16, device=dev),
                "d_logits": torch.empty((s.T, s.E), dtype=torch.float32, device=dev),
                "d_topk_w": torch.empty((s.T, s.k), dtype=torch.float32, device=dev),
            }
        backward(self.cfg, dy, x, self.routing, W_gate, W_up, W_down, self.saved, grads["dx"],
                 grads["dW_gate"], grads["dW_up"], grads["dW_down"], grads["d_logits"],
                 grads.get("d_topk_w"), self.bwd_scratch, stream)
        return grads

    def status(self, stream=None) -> dict:
        return {n: get_device_status(b, stream) for n, b in
                (("route", self.route_scratch), ("forward", self.fwd_scratch), ("backward", self.bwd_scratch))}
