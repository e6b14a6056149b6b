"""moe_expert_ffn_grouped_noalloc: the expert FFN for callers that cannot
allocate device memory (a host framework that owns all device memory, a fixed
memory budget, a loop that must not call cudaMalloc/cudaFree).  Its scratch
is a static array inside the library.  Two calls in a row, through the C ABI,
must give the outputs of the ordinary entry point with a caller workspace.
This file is collected last on purpose; it also passes when run on its own.
"""
import numpy as np
import pytest
import torch

import edge_moe_serving_gb300 as moe
from moe_inputs import CONFIGS
from moe_inputs.device import DeviceCache, x_dev
from gpu_helpers import DEV, ExpertCache, assert_close, oracle_layer, status, status_bits, token_major, ws

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _inputs(cfg, ref, x):
    R = cfg.T * cfg.k
    counts = torch.from_numpy(ref["counts"].astype(np.int32)).to(DEV)
    offsets = torch.from_numpy(ref["offsets"].astype(np.int32)).to(DEV)
    perm = torch.from_numpy(ref["perm"].astype(np.int32)).to(DEV)
    ids = torch.from_numpy(ref["ids"].astype(np.int32)).to(DEV)
    xp = torch.empty((R, cfg.H), dtype=torch.bfloat16, device=DEV)
    c2 = torch.empty(cfg.E, dtype=torch.int32, device=DEV)
    o2 = torch.empty(cfg.E + 1, dtype=torch.int32, device=DEV)
    p2 = torch.empty(R, dtype=torch.int32, device=DEV)
    inv = torch.empty(R, dtype=torch.int32, device=DEV)
    nb = moe.moe_dispatch_workspace_size(cfg.T, cfg.k, cfg.E)
    moe.moe_dispatch(ids, cfg.T, cfg.k, cfg.E, c2, o2, p2, inv, x, cfg.H, xp, ws(nb), nb, status())
    return counts, offsets, perm, xp


def test_noalloc_matches_workspace_entry_point_twice():
    cfg = CONFIGS["batched_decode"]
    dc = DeviceCache(cfg, DEV)
    wc = ExpertCache(cfg, cap=64)
    R = cfg.T * cfg.k
    mode = moe.MOE_FFN_AUTO
    for step in (0, 1):                      # two calls in a row, different tokens
        ref = oracle_layer(cfg, 0, step, wc)
        x = x_dev(cfg, 0, step)
        counts, offsets, perm, xp = _inputs(cfg, ref, x)
        y_ws = torch.full((R, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
        nb = moe.moe_expert_ffn_workspace_size(cfg.T, cfg.k, cfg.E, cfg.H, cfg.I, mode)
        st1 = status()
        moe.moe_expert_ffn_grouped(dc.struct, 0, counts, offsets, perm, x, xp, cfg.T, cfg.k, None, mode, y_ws,
                                   ws(nb), nb, st1)
        y_na = torch.full((R, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
        st2 = status()
        moe.moe_expert_ffn_grouped_noalloc(dc.struct, 0, counts, offsets, perm, x, xp, cfg.T, cfg.k, None, mode,
                                           y_na, st2)
        torch.cuda.synchronize()
        assert status_bits(st1) == 0 and status_bits(st2) == 0
        a, b = y_na.cpu().numpy(), y_ws.cpu().numpy()
        assert np.isfinite(a).all()
        assert_close(a, b, what=f"no-alloc vs workspace entry point, call {step}")
        assert_close(a, token_major(ref), what=f"no-alloc vs oracle, call {step}")


def test_noalloc_rejects_calls_beyond_its_scratch():
    cfg = CONFIGS["batched_decode"]
    dc = DeviceCache(cfg, DEV)
    T = 4096                                  # h would need 4096*8*768*2 bytes > 4 MiB
    assert moe.moe_expert_ffn_workspace_size(T, cfg.k, cfg.E, cfg.H, cfg.I, moe.MOE_FFN_AUTO) > \
        moe.MOE_NOALLOC_FFN_SCRATCH_BYTES
    R = T * cfg.k
    i32 = torch.zeros(R + cfg.E + 1, dtype=torch.int32, device=DEV)
    x = torch.zeros((T, cfg.H), dtype=torch.bfloat16, device=DEV)
    y = torch.zeros((R, cfg.H), dtype=torch.float32, device=DEV)
    st = status()
    rc = moe.lib().moe_expert_ffn_grouped_noalloc(dc.struct, 0, i32.data_ptr(), i32.data_ptr(), i32.data_ptr(),
                                                  x.data_ptr(), None, T, cfg.k, None, moe.MOE_FFN_AUTO,
                                                  y.data_ptr(), st.data_ptr(), None)
    assert rc == moe.MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert status_bits(st) == 0 and not y.any()   # nothing was launched
