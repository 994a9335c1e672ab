"""moe_route_static_scratch: routing for callers that cannot allocate device memory
(for example code running under CUDA-graph capture, or inside a framework whose
allocator owns the GPU).  It must give the same results as moe_route with a
caller-provided scratch buffer, call after call, while allocating nothing itself.

Named so that pytest collects it last."""
import ctypes

import pytest
import torch

from dropless_mixture_experts_top_gb300 import _build, moe, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    _build.build()
    L = moe.lib()
    L.moe_route_static_scratch.argtypes = [ctypes.c_void_p] * 5
    L.moe_route_static_scratch.restype = ctypes.c_int
    return L


def routing_buffers(shape):
    T, E, k = shape.T, shape.E, shape.k
    i32, f32 = torch.int32, torch.float32
    return {
        "topk_idx": torch.full((T, k), -7, dtype=i32, device="cuda"),
        "topk_w": torch.full((T, k), -7.0, dtype=f32, device="cuda"),
        "counts": torch.full((E,), -7, dtype=i32, device="cuda"),
        "offsets": torch.full((E + 1,), -7, dtype=i32, device="cuda"),
        "row_of_slot": torch.full((T, k), -7, dtype=i32, device="cuda"),
        "slot_of_row": torch.full((T * k,), -7, dtype=i32, device="cuda"),
        "w_row": torch.full((T * k,), -7.0, dtype=f32, device="cuda"),
    }


def test_static_scratch_route_matches_moe_route(L):
    shape = synth.MoEShape(T=3000, H=128, I=64, E=64, k=6)
    cfg = moe.make_config(shape)
    stream = torch.cuda.current_stream()
    scratch = torch.empty(moe.query_workspace(cfg)[0], dtype=torch.uint8, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call, seed in enumerate((101, 202)):  # two calls in a row, different routing
        logits = torch.from_numpy(synth.make_inputs_shape(shape, seed, parts=("logits",))["logits"]).cuda()
        if call == 1:
            logits[:, 5] += 4.0  # a hot expert: loads differ from the first call
        ref = routing_buffers(shape)
        moe.route(cfg, logits, ref, scratch, stream)
        got = routing_buffers(shape)
        rt = moe.make_routing(got)
        rc = L.moe_route_static_scratch(ctypes.byref(cfg), ctypes.c_void_p(logits.data_ptr()),
                                        ctypes.byref(rt), ctypes.c_void_p(status.data_ptr()),
                                        ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, moe.status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for n in ("topk_idx", "counts", "offsets", "row_of_slot", "slot_of_row"):
            assert torch.equal(got[n], ref[n]), (call, n)
        for n in ("topk_w", "w_row"):  # the same kernels on the same logits: bit for bit
            assert torch.equal(got[n], ref[n]), (call, n)
        assert int(got["counts"].sum()) == shape.T * shape.k


def test_static_scratch_allocates_nothing(L):
    shape = synth.MoEShape(T=2048, H=128, I=64, E=32, k=4)
    cfg = moe.make_config(shape)
    stream = torch.cuda.current_stream()
    logits = torch.from_numpy(synth.make_inputs_shape(shape, 7, parts=("logits",))["logits"]).cuda()
    got = routing_buffers(shape)
    rt = moe.make_routing(got)
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    args = (ctypes.byref(cfg), ctypes.c_void_p(logits.data_ptr()), ctypes.byref(rt),
            ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    assert L.moe_route_static_scratch(*args) == 0  # first call on the device: the address lookup
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        assert L.moe_route_static_scratch(*args) == 0
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == torch_before
    assert torch.cuda.mem_get_info()[0] == free_before
    assert int(status.item()) == 0


def test_static_scratch_reports_nonfinite_logits(L):
    shape = synth.MoEShape(T=512, H=128, I=64, E=16, k=2)
    cfg = moe.make_config(shape)
    stream = torch.cuda.current_stream()
    logits = torch.from_numpy(synth.make_inputs_shape(shape, 9, parts=("logits",))["logits"]).cuda()
    logits[17, 3] = float("nan")
    got = routing_buffers(shape)
    rt = moe.make_routing(got)
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    rc = L.moe_route_static_scratch(ctypes.byref(cfg), ctypes.c_void_p(logits.data_ptr()), ctypes.byref(rt),
                                    ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) & moe.DEV_NONFINITE_LOGIT
    idx = got["topk_idx"]
    assert int(idx.min()) >= 0 and int(idx.max()) < shape.E  # indices stay in range


def test_static_scratch_rejects_oversized_configuration(L):
    # route scratch needed: one rank byte per slot and the per-block expert histograms, 3.2 MB >
    # the 2.5 MiB array.  Real device buffers throughout, so nothing could fault even if the
    # check were missing.
    shape = synth.MoEShape(T=100000, H=128, I=64, E=256, k=16)
    cfg = moe.make_config(shape)
    assert moe.query_workspace(cfg)[0] > (5 << 19) + 4096
    logits = torch.zeros((shape.T, shape.E), dtype=torch.float32, device="cuda")
    bufs = routing_buffers(shape)
    rt = moe.make_routing(bufs)
    rc = L.moe_route_static_scratch(ctypes.byref(cfg), ctypes.c_void_p(logits.data_ptr()), ctypes.byref(rt),
                                    None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == -3  # MOE_ERR_WORKSPACE
    assert int(bufs["counts"].min()) == -7 and int(bufs["topk_idx"].max()) == -7  # nothing launched
