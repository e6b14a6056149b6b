"""Host-side plumbing of the block-scaled FP4 inputs: the seeded generators
draw what the recipe states, and the device-pool builder lays the banks out
as include/moe.h documents (built here on the CPU)."""
import numpy as np
import torch

import edge_moe_serving_gb300 as moe
from moe_inputs import gen
from moe_inputs.device import MxPool
from oracle import moe_oracle as O


def test_mx_generator_draws_the_recipe():
    gq, gs, uq, us, dq, ds = gen.mx_expert(5, 1, 7, 256, 160)
    assert gq.shape == uq.shape == (160, 128) and dq.shape == (256, 80)
    assert gs.shape == us.shape == (160, 8) and ds.shape == (256, 5)
    for s in (gs, us, ds):
        assert s.min() >= gen.MX_SCALE_EXPONENTS[0] and s.max() <= gen.MX_SCALE_EXPONENTS[1]
    nibbles = np.concatenate([gq & 15, gq >> 4]).ravel()
    assert set(np.unique(nibbles)) == set(range(16))               # every E2M1 code occurs
    # seeded: same key, same bytes; another expert, other bytes
    assert np.array_equal(gen.mx_expert(5, 1, 7, 256, 160)[0], gq)
    assert not np.array_equal(gen.mx_expert(5, 1, 8, 256, 160)[0], gq)
    W = O.mx_expert_weights(gq, gs, uq, us, dq, ds)
    assert all(0.014 < w.std() < 0.022 for w in W)                  # near the bf16 experts' 0.02


def test_nvfp4_generator_draws_the_recipe():
    c, s, ts = gen.nvfp4_bank(2, 0, 3, 1, 64, 96)
    assert c.shape == (64, 48) and s.shape == (64, 6) and ts == np.float32(2.0 ** -9)
    assert s.min() >= gen.NV_SCALE_BYTES[0] and s.max() <= gen.NV_SCALE_BYTES[1]
    assert 0.012 < O.nvfp4_dequant(c, s, ts).std() < 0.022


def test_mx_pool_layout_matches_the_header():
    H, I, n = 64, 96, 3
    experts = {1: gen.mx_expert(0, 0, 4, H, I)}
    pool = MxPool(n, H, I, experts, device="cpu")
    shapes = [tuple(b.shape) for b in pool.banks]
    assert shapes == [(n, I, H // 2), (n, I, H // 32), (n, I, H // 2), (n, I, H // 32), (n, H, I // 2),
                      (n, H, I // 32)]
    assert all(b.dtype == torch.uint8 for b in pool.banks)
    st = pool.struct
    assert [st.gate_q, st.gate_s, st.up_q, st.up_s, st.down_q, st.down_s] == [b.data_ptr() for b in pool.banks]
    assert st.n_slots == n and st.reserved == 0
    for bank, a in zip(pool.banks, experts[1]):
        assert np.array_equal(bank[1].numpy(), a) and not bank[0].any() and not bank[2].any()
    assert isinstance(st, moe.moe_pool_mxfp4)
