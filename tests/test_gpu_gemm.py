"""GPU parity of the expert-FFN kernel variants: the tcgen05 grouped GEMM
(forced and automatic) and the general-shape GEMV, against the fp64 oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import edge_moe_serving_gb300 as moe
from moe_inputs import CONFIGS, gen
from moe_inputs.device import DeviceCache, to_dev_bf16, x_dev
from oracle import moe_oracle as O
from gpu_helpers import DEV, ExpertCache, assert_close, oracle_layer, status, status_bits, token_major, ws

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _ffn(cfg, dc, ref, x, mode, mask=None):
    R = cfg.T * cfg.k
    counts = torch.from_numpy(ref["counts"].astype(np.int32)).to(DEV)
    offsets = torch.from_numpy(ref["offsets"].astype(np.int32)).to(DEV)
    perm = torch.from_numpy(ref["perm"].astype(np.int32)).to(DEV)
    inv = torch.empty(R, dtype=torch.int32, device=DEV)
    ids = torch.from_numpy(ref["ids"].astype(np.int32)).to(DEV)
    xp = torch.empty((R, cfg.H), dtype=torch.bfloat16, device=DEV)
    c2 = torch.empty(cfg.E, dtype=torch.int32, device=DEV)
    o2 = torch.empty(cfg.E + 1, dtype=torch.int32, device=DEV)
    p2 = torch.empty(R, dtype=torch.int32, device=DEV)
    nb = moe.moe_dispatch_workspace_size(cfg.T, cfg.k, cfg.E)
    moe.moe_dispatch(ids, cfg.T, cfg.k, cfg.E, c2, o2, p2, inv, x, cfg.H, xp, ws(nb), nb, status())
    y = torch.full((R, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
    nb = moe.moe_expert_ffn_workspace_size(cfg.T, cfg.k, cfg.E, cfg.H, cfg.I, mode)
    st = status()
    moe.moe_expert_ffn_grouped(dc.struct, 0, counts, offsets, perm, x, xp, cfg.T, cfg.k, mask, mode, y, ws(nb), nb, st)
    torch.cuda.synchronize()
    return y.cpu().numpy(), status_bits(st)


def test_gemm_forced_tiny():
    cfg = CONFIGS["tiny"]
    dc = DeviceCache(cfg, DEV)
    ref = oracle_layer(cfg, 0, 0, ExpertCache(cfg))
    y, st = _ffn(cfg, dc, ref, x_dev(cfg, 0, 0), moe.MOE_FFN_GEMM)
    assert st == 0
    assert_close(y, token_major(ref), what="tiny GEMM y_rows")


@pytest.mark.parametrize("T", [300, 1000])
def test_gemm_auto_mixed_groups(T):
    """Groups of a few rows and of over 256 rows, ragged tails, and experts
    served from both pools, in every FFN mode."""
    cfg = dataclasses.replace(CONFIGS["batched_decode"], name="mixed", T=T, bias="none", cache_slots=40)
    dc = DeviceCache(cfg, DEV)
    xb = gen.f32_to_bf16_bits(np.random.default_rng(T).standard_normal((T, cfg.H)).astype(np.float32))
    wc = ExpertCache(cfg, cap=128)
    x = gen.bf16_bits_to_f64(xb)
    wr = gen.w_router(cfg)
    b = np.zeros(cfg.E, np.float32)
    b[:5] = 3.0                        # a few experts with hundreds of rows
    ref = O.layer_forward(x, wr, b, cfg.k, lambda e: wc(0, e), E=cfg.E)
    assert ref["counts"].max() > 256
    if T == 300:
        assert (ref["counts"][ref["counts"] > 0] <= 8).any()
    for mode in (moe.MOE_FFN_AUTO, moe.MOE_FFN_GEMM, moe.MOE_FFN_GEMV):
        y, st = _ffn(cfg, dc, ref, to_dev_bf16(xb, DEV), mode)
        assert st == 0
        assert_close(y, token_major(ref), what=f"T={T} mode {mode}")


@pytest.mark.parametrize("T,concentrated", [(32, True), (32, False), (7, False), (19, True)])
def test_gemm_thin_tiles(T, concentrated):
    """Calls of at most 32 tokens run the GEMM with 32-row chunks and a deeper
    pipeline: full 32-row groups (every token routed to the same k experts),
    ragged groups of 1..T rows, and both pools."""
    cfg = dataclasses.replace(CONFIGS["batched_decode"], name="thin", T=T, bias="none", cache_slots=40)
    dc = DeviceCache(cfg, DEV)
    xb = gen.f32_to_bf16_bits(np.random.default_rng(100 + T).standard_normal((T, cfg.H)).astype(np.float32))
    wc = ExpertCache(cfg, cap=128)
    x = gen.bf16_bits_to_f64(xb)
    b = np.zeros(cfg.E, np.float32)
    if concentrated:
        b[40:40 + cfg.k] = 50.0            # every token takes the same k experts
    ref = O.layer_forward(x, gen.w_router(cfg), b, cfg.k, lambda e: wc(0, e), E=cfg.E)
    if concentrated:
        assert (ref["counts"][40:40 + cfg.k] == T).all()
    y, st = _ffn(cfg, dc, ref, to_dev_bf16(xb, DEV), moe.MOE_FFN_GEMM)
    assert st == 0
    assert_close(y, token_major(ref), what=f"thin GEMM T={T}")


def test_gemm_mask_split_is_bitwise():
    cfg = dataclasses.replace(CONFIGS["batched_decode"], name="mixed", T=400, bias="none")
    dc = DeviceCache(cfg, DEV)
    xb = gen.f32_to_bf16_bits(np.random.default_rng(1).standard_normal((cfg.T, cfg.H)).astype(np.float32))
    x = gen.bf16_bits_to_f64(xb)
    ref = O.layer_forward(x, gen.w_router(cfg), None, cfg.k, lambda e: gen.expert_f64(cfg, 0, e), E=cfg.E)
    xd = to_dev_bf16(xb, DEV)
    full, _ = _ffn(cfg, dc, ref, xd, moe.MOE_FFN_GEMM)
    mask = (np.arange(cfg.E) % 3 == 0).astype(np.uint8)
    y1, _ = _ffn(cfg, dc, ref, xd, moe.MOE_FFN_GEMM, torch.from_numpy(mask).to(DEV))
    y2, _ = _ffn(cfg, dc, ref, xd, moe.MOE_FFN_GEMM, torch.from_numpy(1 - mask).to(DEV))
    rows_m = mask[ref["ids"].reshape(-1)].astype(bool)        # token-major rows
    assert np.array_equal(np.where(rows_m[:, None], y1, y2), full)


def test_gemv_general_shape():
    """H, I not multiples of 256: the general GEMV kernel."""
    cfg = dataclasses.replace(CONFIGS["tiny"], name="odd", H=200, I=136, T=20, E=6, k=3)
    dc = DeviceCache(cfg, DEV)
    xb = gen.f32_to_bf16_bits(np.random.default_rng(2).standard_normal((cfg.T, cfg.H)).astype(np.float32))
    x = gen.bf16_bits_to_f64(xb)
    ref = O.layer_forward(x, gen.w_router(cfg), None, cfg.k, lambda e: gen.expert_f64(cfg, 0, e), E=cfg.E)
    for mode in (moe.MOE_FFN_AUTO, moe.MOE_FFN_GEMV):
        y, st = _ffn(cfg, dc, ref, to_dev_bf16(xb, DEV), mode)
        assert st == 0
        assert_close(y, token_major(ref), what=f"odd shape mode {mode}")
