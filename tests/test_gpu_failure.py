"""Failure detection without a GPU fault: a pipeline wait that is never
satisfied gives up after its bound, reports MOE_DEV_WAIT_TIMEOUT through the
status word, and leaves the CUDA context usable (a full layer call afterwards
still matches the oracle)."""
import time

import pytest
import torch

from dropless_mixture_experts_top_gb300 import moe, synth
from dropless_mixture_experts_top_gb300.synth import MoEShape
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from dropless_mixture_experts_top_gb300 import _build as B
    B.build()


def test_bounded_wait_reports_timeout_and_context_survives():
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    moe.selftest_wait_timeout(status)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert int(status.item()) == moe.DEV_WAIT_TIMEOUT
    assert elapsed < 30.0, elapsed  # the bound is about two seconds of SM clock
    # the context is still usable: a full layer call matches the oracle
    shape = MoEShape(T=256, H=128, I=128, E=8, k=2)
    inp = synth.make_inputs_shape(shape, 71)
    layer, out, grads = G.run_layer(shape, inp)
    assert layer.status() == {"route": 0, "forward": 0, "backward": 0}
    G.check_full(shape, inp, layer, out, grads)
