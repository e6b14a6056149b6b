"""Failure detection without a GPU fault: a bounded wait that runs out
reports MOE_DEV_ERR_TIMEOUT and the context stays usable; a bad expert id and
an unbound slot are reported through the device status word."""
import time

import numpy as np
import pytest
import torch

import edge_moe_serving_gb300 as moe
from moe_inputs import CONFIGS
from moe_inputs.device import DeviceCache, DeviceLayer, x_dev
from gpu_helpers import DEV, status, status_bits
from gpu_helpers import run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def test_bounded_wait_runs_out_and_reports_timeout():
    st = status()
    t0 = time.perf_counter()
    moe.moe_check_bounded_wait(st)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert status_bits(st) & moe.MOE_DEV_ERR_TIMEOUT
    assert 0.5 < elapsed < 10.0
    # the context is still usable: a whole layer runs and reports no error
    cfg = CONFIGS["tiny"]
    dc = DeviceCache(cfg, DEV)
    dl = DeviceLayer(cfg, 0, DEV)
    got = run_layer(dc, dl, x_dev(cfg, 0, 0), cfg.T, 0, 1, 0)
    assert got["status"] == 0 and torch.isfinite(got["out"].float()).all()


def test_bad_expert_id_reported_by_bind():
    cfg = CONFIGS["tiny"]
    dc = DeviceCache(cfg, DEV)
    ids = torch.tensor([[0, 1], [2, 99]], dtype=torch.int32, device=DEV)
    nb = moe.moe_cache_bind_workspace_size(dc.struct, 2, 2)
    st = status()
    moe.moe_cache_bind_slots(dc.struct, 0, ids, 2, 2, 0, 1, 0, 0, None, None,
                             torch.empty(nb, dtype=torch.uint8, device=DEV), nb, st)
    torch.cuda.synchronize()
    assert status_bits(st) & moe.MOE_DEV_ERR_BAD_ID
