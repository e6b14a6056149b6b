"""GPU parity of every step of the routed MoE layer against the fp64 oracle.

All calls go through the C ABI (ctypes binding).  Routing ids and dispatch
permutations must be bit-exact; residency state after every bind call must
equal the oracle's; expert outputs and layer outputs must meet relative
Frobenius error <= 1e-2 and max-abs error <= 2e-2.
"""
import dataclasses

import numpy as np
import pytest
import torch

import edge_moe_serving_gb300 as moe
from moe_inputs import CONFIGS, gen
from moe_inputs.device import DeviceCache, DeviceLayer, to_dev, to_dev_bf16, x_dev
from oracle import moe_oracle as O
from gpu_helpers import (DEV, ExpertCache, assert_close, bf16_to_f64, oracle_layer, run_layer, status,
                         status_bits, token_major, ws)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _route(cfg, layer, step, x_bits=None, want_logits=True):
    xb = gen.x_bits(cfg, layer, step) if x_bits is None else x_bits
    T = xb.shape[0]
    x = to_dev_bf16(xb, DEV)
    wr = to_dev(gen.w_router(cfg, layer), DEV)
    b = gen.bias(cfg, layer, step)
    bd = None if b is None else to_dev(b, DEV)
    ids = torch.empty((T, cfg.k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, cfg.k), dtype=torch.float32, device=DEV)
    lg = torch.empty((T, cfg.E), dtype=torch.float32, device=DEV) if want_logits else None
    nb = moe.moe_route_topk_workspace_size(T, cfg.H, cfg.E)
    st = status()
    moe.moe_route_topk(x, T, cfg.H, wr, bd, cfg.E, cfg.k, ids, w, lg, ws(nb), nb, st)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), (lg.cpu().numpy() if want_logits else None), status_bits(st)


# ------------------------------------------------------------------ router + top-k
@pytest.mark.parametrize("name,steps", [("tiny", [0]), ("decode", [0, 1, 7, 31]), ("batched_decode", [0, 5, 31]),
                                        ("prefill", [0]), ("long_prefill", [0])])
def test_route_topk_bit_exact(name, steps):
    cfg = CONFIGS[name]
    for layer in range(min(cfg.n_layers, 2)):
        for step in steps:
            ids, w, lg, st = _route(cfg, layer, step)
            x = gen.bf16_bits_to_f64(gen.x_bits(cfg, layer, step))
            ref_lg = O.router_logits(x, gen.w_router(cfg, layer), gen.bias(cfg, layer, step))
            ref_ids, ref_w = O.select_topk(ref_lg, cfg.k)
            assert st == 0
            assert np.array_equal(ids, ref_ids), (name, layer, step)
            assert np.abs(lg - ref_lg).max() < 1e-4
            assert np.abs(w - ref_w).max() < 1e-5


def test_route_topk_small_shapes_and_ties():
    """Ragged E and T, all-equal logits (ties go to the lower id)."""
    rng = np.random.default_rng(0)
    # (T > 32, H % 64 == 0) runs on the tensor cores: ragged expert tiles
    # (E = 100, 130), ragged token tiles (T = 200, 129, 300), E = 512, tiny E.
    for T, H, E, k in ((1, 8, 3, 1), (5, 24, 33, 4), (33, 64, 100, 7), (70, 40, 512, 16), (31, 16, 64, 16),
                       (32, 128, 512, 16), (17, 64, 256, 8),
                       (200, 128, 130, 6), (129, 192, 512, 16), (300, 64, 8, 2)):
        xb = gen.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
        wr = (rng.standard_normal((E, H)) * 0.1).astype(np.float32)
        b = (rng.standard_normal(E) * 0.05).astype(np.float32)
        x = to_dev_bf16(xb, DEV)
        ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
        w = torch.empty((T, k), dtype=torch.float32, device=DEV)
        lg = torch.empty((T, E), dtype=torch.float32, device=DEV)
        nb = moe.moe_route_topk_workspace_size(T, H, E)
        st = status()
        moe.moe_route_topk(x, T, H, to_dev(wr, DEV), to_dev(b, DEV), E, k, ids, w, lg, ws(nb), nb, st)
        ref_lg = O.router_logits(gen.bf16_bits_to_f64(xb), wr, b)
        gaps = O.topk_gap(ref_lg, k) if k < E else np.full(T, np.inf)
        ref_ids, ref_w = O.select_topk(ref_lg, k)
        ok = gaps >= 1e-3
        assert status_bits(st) == 0
        assert np.abs(lg.cpu().numpy() - ref_lg).max() < 1e-4, (T, H, E)
        assert np.array_equal(ids.cpu().numpy()[ok], ref_ids[ok]), (T, H, E)
        assert np.abs(w.cpu().numpy()[ok] - ref_w[ok]).max() < 1e-5, (T, H, E)
    # ties: zero router weights -> every logit equal -> ids 0..k-1, weights 1/k
    for T, H in ((1, 16), (3, 16), (20, 16), (32, 32), (40, 16), (40, 64), (257, 128)):
        x = to_dev_bf16(np.zeros((T, H), np.uint16), DEV)
        wr = torch.zeros((10, H), dtype=torch.float32, device=DEV)
        ids = torch.empty((T, 3), dtype=torch.int32, device=DEV)
        w = torch.empty((T, 3), dtype=torch.float32, device=DEV)
        nb = moe.moe_route_topk_workspace_size(T, H, 10)
        moe.moe_route_topk(x, T, H, wr, None, 10, 3, ids, w, None, ws(nb), nb, status())
        assert (ids.cpu().numpy() == np.array([0, 1, 2])).all()
        assert np.allclose(w.cpu().numpy(), 1.0 / 3, atol=1e-7)


# ------------------------------------------------------------------ dispatch
def _dispatch(ids_np, E, x=None, H=0):
    T, k = ids_np.shape
    R = T * k
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, np.int32)).to(DEV)
    counts = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
    perm = torch.full((max(R, 1),), -7, dtype=torch.int32, device=DEV)
    inv = torch.full((max(R, 1),), -7, dtype=torch.int32, device=DEV)
    xp = torch.empty((max(R, 1), H), dtype=torch.bfloat16, device=DEV) if x is not None else None
    nb = moe.moe_dispatch_workspace_size(T, k, E)
    st = status()
    moe.moe_dispatch(ids, T, k, E, counts, offsets, perm, inv, x, H, xp, ws(nb), nb, st)
    torch.cuda.synchronize()
    return (counts.cpu().numpy(), offsets.cpu().numpy(), perm.cpu().numpy()[:R], inv.cpu().numpy()[:R],
            xp, status_bits(st))


@pytest.mark.parametrize("T,k,E", [(1, 6, 256), (64, 2, 8), (32, 8, 128), (700, 6, 256), (8192, 6, 256),
                                   (16384, 6, 256), (5000, 3, 1000), (1111, 7, 13), (0, 6, 256)])
def test_dispatch_bit_exact(T, k, E):
    rng = np.random.default_rng(T + E)
    p = rng.zipf(1.3, size=E).astype(np.float64)
    p /= p.sum()
    ids = np.stack([np.sort(rng.choice(E, k, replace=False, p=p)) for _ in range(T)]).reshape(T, k) \
        if T else np.zeros((0, k), np.int32)
    counts, offsets, perm, inv, _, st = _dispatch(ids, E)
    rc, ro, rp, ri = O.dispatch(ids, E)
    assert st == 0
    assert np.array_equal(counts, rc) and np.array_equal(offsets, ro)
    assert np.array_equal(perm, rp) and np.array_equal(inv, ri)


def test_dispatch_gather_and_bad_ids():
    rng = np.random.default_rng(5)
    T, k, E, H = 300, 4, 16, 64
    ids = np.stack([np.sort(rng.choice(E, k, replace=False)) for _ in range(T)])
    xb = gen.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    x = to_dev_bf16(xb, DEV)
    counts, offsets, perm, inv, xp, st = _dispatch(ids, E, x, H)
    ref = xb[perm // k]
    assert np.array_equal(xp.cpu().view(torch.int16).numpy().view(np.uint16), ref)
    bad = ids.copy()
    bad[3, 1] = E + 5
    bad[7, 0] = -1
    counts, offsets, perm, inv, _, st = _dispatch(bad, E)
    assert st & moe.MOE_DEV_ERR_BAD_ID
    assert counts.sum() == T * k - 2 and offsets[-1] == T * k - 2


# ------------------------------------------------------------------ bind (residency)
def _bind_trace(name, steps, layers=None):
    cfg = CONFIGS[name]
    dc = DeviceCache(cfg, DEV)
    ref = gen.initial_cache(cfg)
    layers = list(range(cfg.n_layers)) if layers is None else layers
    nb = moe.moe_cache_bind_workspace_size(dc.struct, cfg.T, cfg.k)
    w = ws(nb)
    kmax = min(cfg.T * cfg.k, cfg.E)
    n_fills = 0
    for step in range(steps):
        for layer in layers:
            x = gen.bf16_bits_to_f64(gen.x_bits(cfg, layer, step))
            ids, _ = O.select_topk(O.router_logits(x, gen.w_router(cfg, layer), gen.bias(cfg, layer, step)), cfg.k)
            seed = 1234 + step
            ref, res = O.bind(ref, layer, ids, cfg.E, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, seed)
            st = status()
            stats = torch.zeros(8, dtype=torch.int32, device=DEV)
            fills = torch.full((kmax, 2), -1, dtype=torch.int32, device=DEV)
            moe.moe_cache_bind_slots(dc.struct, layer, torch.from_numpy(ids).to(DEV), cfg.T, cfg.k, cfg.phi_q16,
                                     cfg.min_fill, cfg.fill_policy, seed, stats, fills, w, nb, st)
            torch.cuda.synchronize()
            got = dc.state()
            for key in ("table", "owner", "stamp"):
                assert np.array_equal(got[key], np.asarray(ref[key])), (name, step, layer, key)
            assert got["clock"] == ref["clock"]
            s = dict(zip(moe.BIND_STATS_FIELDS, stats.cpu().numpy().tolist()))
            for kk, v in res["stats"].items():
                assert s[kk] == v, (name, step, layer, kk)
            nf = res["stats"]["n_fill"]
            assert [tuple(r) for r in fills.cpu().numpy()[:nf].tolist()] == res["fills"]
            assert status_bits(st) == 0
            n_fills += nf
    return dc, n_fills


def test_bind_decode_trace():
    dc, n_fills = _bind_trace("decode", 32)
    assert n_fills > 0
    # every cache slot holds the weights of the pair it claims (the fused fill copy)
    owner = dc.owner.cpu().numpy()
    for b in range(3):
        assert torch.equal(dc.cache[b], dc.staging[b].index_select(0, torch.from_numpy(owner.astype(np.int64)).to(DEV)))


def test_bind_batched_decode_trace_random_policy():
    dc, n_fills = _bind_trace("batched_decode", 32)
    assert n_fills > 0
    owner = dc.owner.cpu().numpy()
    for b in range(3):
        assert torch.equal(dc.cache[b], dc.staging[b].index_select(0, torch.from_numpy(owner.astype(np.int64)).to(DEV)))


def test_bind_long_prefill_layers():
    _bind_trace("long_prefill", 1)


def test_bind_edge_cases():
    """Overflow (all slots hit), empty call, floor of one fill, phi = 0."""
    cfg = CONFIGS["tiny"]
    import dataclasses
    small = dataclasses.replace(cfg, cache_slots=2)
    dc = DeviceCache(small, DEV)
    ref = gen.initial_cache(small)
    nb = moe.moe_cache_bind_workspace_size(dc.struct, 4, 2)
    w = ws(nb)
    cases = [(np.array([[int(ref["owner"][0]), int(ref["owner"][1])], [3, 5]]), moe.Q16 if hasattr(moe, "Q16") else 65536, 1),
             (np.zeros((0, 2), np.int32), 65536, 1),
             (np.array([[0, 1], [2, 3]]), 1000, 1),
             (np.array([[4, 6]]), 0, 1),
             (np.array([[7, 6]]), 1000, 0)]
    for ids, phi, mf in cases:
        ids = np.asarray(ids, np.int32)
        T = ids.shape[0]
        ref, res = O.bind(ref, 0, ids, small.E, phi, mf, 0, 0)
        stats = torch.zeros(8, dtype=torch.int32, device=DEV)
        moe.moe_cache_bind_slots(dc.struct, 0, torch.from_numpy(ids).to(DEV) if T else None, T, 2, phi, mf, 0, 0,
                                 stats, None, w, nb, status())
        torch.cuda.synchronize()
        got = dc.state()
        for key in ("table", "owner", "stamp"):
            assert np.array_equal(got[key], np.asarray(ref[key])), (ids.tolist(), key)
        s = dict(zip(moe.BIND_STATS_FIELDS, stats.cpu().numpy().tolist()))
        for kk, v in res["stats"].items():
            assert s[kk] == v


# ------------------------------------------------------------------ expert FFN
@pytest.mark.parametrize("name,steps", [("tiny", [0]), ("decode", [0, 3]), ("batched_decode", [0, 9])])
def test_expert_ffn_gemv_rows(name, steps):
    cfg = CONFIGS[name]
    dc = DeviceCache(cfg, DEV)
    wc = ExpertCache(cfg)
    for step in steps:
        ref = oracle_layer(cfg, 0, step, wc)
        R = cfg.T * cfg.k
        counts = torch.from_numpy(ref["counts"].astype(np.int32)).to(DEV)
        offsets = torch.from_numpy(ref["offsets"].astype(np.int32)).to(DEV)
        perm = torch.from_numpy(ref["perm"].astype(np.int32)).to(DEV)
        x = x_dev(cfg, 0, step)
        y = torch.full((R, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
        nb = moe.moe_expert_ffn_workspace_size(cfg.T, cfg.k, cfg.E, cfg.H, cfg.I, moe.MOE_FFN_GEMV)
        st = status()
        # the slot table of the initial state binds every expert (cache or staging pool)
        moe.moe_expert_ffn_grouped(dc.struct, 0, counts, offsets, perm, x, None, cfg.T, cfg.k, None,
                                   moe.MOE_FFN_GEMV, y, ws(nb), nb, st)
        torch.cuda.synchronize()
        assert status_bits(st) == 0
        assert_close(y.cpu().numpy(), token_major(ref), what=f"{name} step {step} y_rows")


def test_expert_ffn_mask_split_is_bitwise():
    """F and C evaluated in separate launches give the same bits as one launch."""
    cfg = CONFIGS["batched_decode"]
    dc = DeviceCache(cfg, DEV)
    wc = ExpertCache(cfg)
    ref = oracle_layer(cfg, 0, 2, wc)
    R = cfg.T * cfg.k
    counts = torch.from_numpy(ref["counts"].astype(np.int32)).to(DEV)
    offsets = torch.from_numpy(ref["offsets"].astype(np.int32)).to(DEV)
    perm = torch.from_numpy(ref["perm"].astype(np.int32)).to(DEV)
    x = x_dev(cfg, 0, 2)
    nb = moe.moe_expert_ffn_workspace_size(cfg.T, cfg.k, cfg.E, cfg.H, cfg.I, moe.MOE_FFN_GEMV)
    w = ws(nb)
    y_full = torch.zeros((R, cfg.H), dtype=torch.float32, device=DEV)
    moe.moe_expert_ffn_grouped(dc.struct, 0, counts, offsets, perm, x, None, cfg.T, cfg.k, None,
                               moe.MOE_FFN_GEMV, y_full, w, nb, status())
    rng = np.random.default_rng(9)
    for _ in range(5):
        mask = (rng.random(cfg.E) < 0.5).astype(np.uint8)
        m1 = torch.from_numpy(mask).to(DEV)
        m2 = torch.from_numpy(1 - mask).to(DEV)
        y = torch.zeros((R, cfg.H), dtype=torch.float32, device=DEV)
        moe.moe_expert_ffn_grouped(dc.struct, 0, counts, offsets, perm, x, None, cfg.T, cfg.k, m1,
                                   moe.MOE_FFN_GEMV, y, w, nb, status())
        moe.moe_expert_ffn_grouped(dc.struct, 0, counts, offsets, perm, x, None, cfg.T, cfg.k, m2,
                                   moe.MOE_FFN_GEMV, y, w, nb, status())
        torch.cuda.synchronize()
        assert torch.equal(y, y_full)


def test_expert_ffn_unbound_slot_is_reported():
    """A -1 table entry: the expert's rows stay unwritten and the status bit is set."""
    cfg = CONFIGS["tiny"]
    dc = DeviceCache(cfg, DEV)
    wc = ExpertCache(cfg)
    ref = oracle_layer(cfg, 0, 0, wc)
    e_bad = int(np.nonzero(ref["counts"])[0][1])
    dc.table[e_bad] = -1
    R = cfg.T * cfg.k
    y = torch.full((R, cfg.H), 123.0, dtype=torch.float32, device=DEV)
    nb = moe.moe_expert_ffn_workspace_size(cfg.T, cfg.k, cfg.E, cfg.H, cfg.I, moe.MOE_FFN_GEMV)
    st = status()
    moe.moe_expert_ffn_grouped(dc.struct, 0, torch.from_numpy(ref["counts"].astype(np.int32)).to(DEV),
                               torch.from_numpy(ref["offsets"].astype(np.int32)).to(DEV),
                               torch.from_numpy(ref["perm"].astype(np.int32)).to(DEV), x_dev(cfg, 0, 0), None,
                               cfg.T, cfg.k, None, moe.MOE_FFN_GEMV, y, ws(nb), nb, st)
    torch.cuda.synchronize()
    assert status_bits(st) & moe.MOE_DEV_ERR_UNBOUND
    yc = y.cpu().numpy()
    bad_rows = ref["ids"].reshape(-1) == e_bad            # token-major rows of the unbound expert
    assert bad_rows.sum() == ref["counts"][e_bad] > 0
    assert np.all(yc[bad_rows] == 123.0)
    assert_close(yc[~bad_rows], token_major(ref)[~bad_rows], what="other experts")


# ------------------------------------------------------------------ combine
def test_combine_matches_oracle_definition():
    rng = np.random.default_rng(3)
    for T, k, H in ((1, 6, 4096), (37, 3, 64), (513, 8, 2048)):
        R = T * k
        y = rng.standard_normal((R, H)).astype(np.float32)        # token-major rows
        w = rng.random((T, k)).astype(np.float32)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        o32 = torch.empty((T, H), dtype=torch.float32, device=DEV)
        moe.moe_combine(to_dev(y, DEV), to_dev(w, DEV), T, k, H, out, o32, status())
        torch.cuda.synchronize()
        ref = O.combine(y.astype(np.float64), np.arange(R), w.astype(np.float64), k)
        got32 = o32.cpu().numpy()
        assert np.abs(got32 - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())
        # the bf16 output is the fp32 result rounded to nearest even
        bits = out.cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(bits, gen.f32_to_bf16_bits(got32))


# ------------------------------------------------------------------ whole layer
def test_layer_tiny():
    cfg = CONFIGS["tiny"]
    dc = DeviceCache(cfg, DEV)
    dl = DeviceLayer(cfg, 0, DEV)
    wc = ExpertCache(cfg)
    ref = oracle_layer(cfg, 0, 0, wc)
    for mode in (moe.MOE_FFN_AUTO, moe.MOE_FFN_GEMV):
        got = run_layer(dc, dl, x_dev(cfg, 0, 0), cfg.T, 0, 1, 0, ffn_mode=mode)
        assert got["status"] == 0
        assert np.array_equal(got["topk_ids"].cpu().numpy().reshape(cfg.T, cfg.k), ref["ids"])
        assert np.array_equal(got["perm"].cpu().numpy(), ref["perm"])
        assert_close(bf16_to_f64(got["out"]), ref["out"], what=f"tiny out mode {mode}")


def _layer_without_buffers(dc, dl, x, T, mode):
    """moe_layer_forward with no caller buffers: calls whose groups all run on
    the GEMM keep the expert rows internally in bf16."""
    cfg = dc.cfg
    nbytes = moe.moe_layer_workspace_size(dl.struct, dc.struct, T, mode)
    out = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=DEV)
    st = status()
    moe.moe_layer_forward(dl.struct, dc.struct, x, T, out, 0, 1, 0, 0, mode, None, ws(nbytes), nbytes, st, None)
    torch.cuda.synchronize()
    return out, status_bits(st)


@pytest.mark.parametrize("name", ["tiny", "batched_decode"])
def test_layer_bf16_expert_rows(name):
    """Without caller buffers the GEMM path keeps the expert rows in bf16; the
    output stays within the tolerance of the oracle and of the fp32-rows path."""
    cfg = CONFIGS[name]
    dc = DeviceCache(cfg, DEV)
    dl = DeviceLayer(cfg, 0, DEV)
    ref = oracle_layer(cfg, 0, 0, ExpertCache(cfg, cap=64))
    for mode in (moe.MOE_FFN_AUTO, moe.MOE_FFN_GEMM):
        dc.reset()
        out, st = _layer_without_buffers(dc, dl, x_dev(cfg, 0, 0), cfg.T, mode)
        assert st == 0
        assert_close(bf16_to_f64(out), ref["out"], what=f"{name} mode {mode} bf16 rows")
        dc.reset()
        got = run_layer(dc, dl, x_dev(cfg, 0, 0), cfg.T, 0, 1, 0, ffn_mode=mode)
        assert_close(bf16_to_f64(out), bf16_to_f64(got["out"]), what=f"{name} bf16 rows vs fp32 rows")


def _decode_trace(name, out_steps):
    cfg = CONFIGS[name]
    dc = DeviceCache(cfg, DEV)
    dl = DeviceLayer(cfg, 0, DEV)
    wc = ExpertCache(cfg, cap=48)
    ref_state = gen.initial_cache(cfg)
    outs = []
    for step in range(cfg.steps):
        dl.set_bias(step)
        seed = 77 + step
        got = run_layer(dc, dl, x_dev(cfg, 0, step), cfg.T, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, seed)
        ids = got["topk_ids"].cpu().numpy().reshape(cfg.T, cfg.k)
        x = gen.bf16_bits_to_f64(gen.x_bits(cfg, 0, step))
        ref_ids, _ = O.select_topk(O.router_logits(x, gen.w_router(cfg, 0), gen.bias(cfg, 0, step)), cfg.k)
        assert np.array_equal(ids, ref_ids), step
        ref_state, res = O.bind(ref_state, 0, ref_ids, cfg.E, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, seed)
        st = dc.state()
        for key in ("table", "owner", "stamp"):
            assert np.array_equal(st[key], np.asarray(ref_state[key])), (step, key)
        for kk, v in res["stats"].items():
            assert got["stats"][kk] == v, (step, kk)
        assert got["status"] == 0
        if step in out_steps:
            ref = oracle_layer(cfg, 0, step, wc)
            assert np.array_equal(got["perm"].cpu().numpy(), ref["perm"])
            assert_close(bf16_to_f64(got["out"]), ref["out"], what=f"{name} step {step}")
        outs.append(got["out"].clone())
    return outs


def _gap_safe_x_bits(cfg, step):
    """x of (layer 0, step) with every token's k-th/(k+1)-th logit gap >= 1e-3
    (rows redrawn from the seeded stream until they are), for configurations
    that have no stored redraw map."""
    xb = gen.x_bits(cfg, 0, step, redraws={})
    wr, b = gen.w_router(cfg, 0), gen.bias(cfg, 0, step)
    for t in range(cfg.T):
        r = 0
        while O.topk_gap(O.router_logits(gen.bf16_bits_to_f64(xb[t:t + 1]), wr, b), cfg.k)[0] < 1e-3:
            xb[t] = gen.x_row_redraw(cfg, 0, step, t, r)
            r += 1
    return xb


@pytest.mark.parametrize("base,T,mode", [("decode", 2, moe.MOE_FFN_AUTO), ("decode", 3, moe.MOE_FFN_GEMV),
                                         ("decode", 5, moe.MOE_FFN_GEMV), ("batched_decode", 4, moe.MOE_FFN_GEMV)])
def test_layer_one_launch_multi_token(base, T, mode):
    """The one-launch decode layer for 2..5 tokens (instances of 2, 4 and 8
    rows): ids and residency state bit-exact over a short trace with fills,
    outputs within tolerance."""
    cfg = dataclasses.replace(CONFIGS[base], name=f"{base}_t{T}", T=T, steps=6)
    assert cfg.T * cfg.k <= 32
    dc = DeviceCache(cfg, DEV)
    dl = DeviceLayer(cfg, 0, DEV)
    wc = ExpertCache(cfg, cap=32)
    ref_state = gen.initial_cache(cfg)
    for step in range(cfg.steps):
        dl.set_bias(step)
        seed = 300 + step
        xb = _gap_safe_x_bits(cfg, step)
        got = run_layer(dc, dl, to_dev_bf16(xb, DEV), cfg.T, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, seed,
                        ffn_mode=mode)
        assert got["status"] == 0
        ref = oracle_layer(cfg, 0, step, wc, x_bits=xb)
        assert np.array_equal(got["topk_ids"].cpu().numpy().reshape(cfg.T, cfg.k), ref["ids"]), step
        assert np.array_equal(got["perm"].cpu().numpy(), ref["perm"]), step
        ref_state, res = O.bind(ref_state, 0, ref["ids"], cfg.E, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, seed)
        st = dc.state()
        for key in ("table", "owner", "stamp"):
            assert np.array_equal(st[key], np.asarray(ref_state[key])), (step, key)
        for kk, v in res["stats"].items():
            assert got["stats"][kk] == v, (step, kk)
        assert_close(bf16_to_f64(got["out"]), ref["out"], what=f"{cfg.name} step {step}")
        assert_close(got["y_rows"].cpu().numpy(), token_major(ref), what=f"{cfg.name} step {step} y_rows")


def test_layer_one_launch_max_shape():
    """The one-launch decode layer at its limits: 512 experts (four router rows
    per CTA), top-8 of 4 tokens (32 routed rows, instances of 4 rows), 1024
    cache slots shared by 3 layers (the largest state copy, a full 32-word
    hitmap, victims scanned 32 slots per lane), pure fill: ids, residency
    state and stats bit-exact over a trace with fills, outputs within
    tolerance."""
    from moe_inputs.configs import LayerConfig, Q16
    cfg = LayerConfig("decode_max", T=4, H=256, E=512, k=8, I=512, seed=41, n_layers=3, steps=6,
                      cache_slots=1024, phi_q16=Q16, bias="zipf")
    dc = DeviceCache(cfg, DEV)
    dl = DeviceLayer(cfg, 0, DEV)
    wc = ExpertCache(cfg, cap=64)
    ref_state = gen.initial_cache(cfg)
    fills = 0
    for step in range(cfg.steps):
        dl.set_bias(step)
        seed = 700 + step
        xb = _gap_safe_x_bits(cfg, step)
        got = run_layer(dc, dl, to_dev_bf16(xb, DEV), cfg.T, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, seed,
                        ffn_mode=moe.MOE_FFN_GEMV)   # GEMV mode: no gathered rows, the one-launch path
        assert got["status"] == 0
        ref = oracle_layer(cfg, 0, step, wc, x_bits=xb)
        assert np.array_equal(got["topk_ids"].cpu().numpy().reshape(cfg.T, cfg.k), ref["ids"]), step
        assert np.array_equal(got["perm"].cpu().numpy(), ref["perm"]), step
        ref_state, res = O.bind(ref_state, 0, ref["ids"], cfg.E, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, seed)
        st = dc.state()
        for key in ("table", "owner", "stamp"):
            assert np.array_equal(st[key], np.asarray(ref_state[key])), (step, key)
        for kk, v in res["stats"].items():
            assert got["stats"][kk] == v, (step, kk)
        fills += res["stats"]["n_fill"]
        assert_close(bf16_to_f64(got["out"]), ref["out"], what=f"{cfg.name} step {step}")
    assert fills > 0


@pytest.mark.parametrize("T,n_layers,slots,mode", [(16, 1, None, moe.MOE_FFN_GEMV), (1, 256, 1536, moe.MOE_FFN_AUTO),
                                                   (3, 256, 1536, moe.MOE_FFN_GEMV)])
def test_layer_front_small_fused_combine(T, n_layers, slots, mode):
    """Calls the one-launch kernel does not take (16 tokens; or a pool of more
    than 1024 slots) but with at most 32 routed rows: the one-warp front end,
    then the fused GEMV launch whose CTAs combine their own output rows.  ids,
    residency state and stats bit-exact over a trace, outputs within
    tolerance."""
    from moe_inputs.configs import Q16
    cfg = dataclasses.replace(CONFIGS["tiny"], name=f"front_t{T}_s{slots}", T=T, n_layers=n_layers, steps=4,
                              cache_slots=slots, phi_q16=Q16 if slots else 0, bias="zipf")
    assert cfg.T * cfg.k <= 32
    dc = DeviceCache(cfg, DEV)
    dl = DeviceLayer(cfg, 0, DEV)
    wc = ExpertCache(cfg, cap=16)
    ref_state = gen.initial_cache(cfg)
    for step in range(cfg.steps):
        dl.set_bias(step)
        seed = 900 + step
        xb = _gap_safe_x_bits(cfg, step)
        got = run_layer(dc, dl, to_dev_bf16(xb, DEV), cfg.T, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, seed,
                        ffn_mode=mode)
        assert got["status"] == 0
        ref = oracle_layer(cfg, 0, step, wc, x_bits=xb)
        assert np.array_equal(got["topk_ids"].cpu().numpy().reshape(cfg.T, cfg.k), ref["ids"]), step
        assert np.array_equal(got["perm"].cpu().numpy(), ref["perm"]), step
        ref_state, res = O.bind(ref_state, 0, ref["ids"], cfg.E, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, seed)
        st = dc.state()
        for key in ("table", "owner", "stamp"):
            assert np.array_equal(st[key], np.asarray(ref_state[key])), (step, key)
        for kk, v in res["stats"].items():
            assert got["stats"][kk] == v, (step, kk)
        assert_close(bf16_to_f64(got["out"]), ref["out"], what=f"{cfg.name} step {step}")


def test_layer_decode_trace():
    _decode_trace("decode", set(range(32)))


def test_layer_batched_decode_trace():
    _decode_trace("batched_decode", {0, 1, 2, 5, 11, 17, 23, 31})


def test_layer_output_independent_of_split():
    """The same decode trace under different F/C splits gives bitwise identical
    outputs (the merge is exact): phi = 1 (all fills), 0.25, and 0 (no fills)."""
    cfg = CONFIGS["decode"]
    results = []
    for phi, mf in ((65536, 1), (16384, 1), (0, 0)):
        dc = DeviceCache(cfg, DEV)
        dl = DeviceLayer(cfg, 0, DEV)
        outs, fills = [], 0
        for step in range(12):
            got = run_layer(dc, dl, x_dev(cfg, 0, step), cfg.T, phi, mf, cfg.fill_policy, 5,
                            ffn_mode=moe.MOE_FFN_GEMV)
            outs.append(got["out"].clone())
            fills += got["stats"]["n_fill"]
        results.append((outs, fills))
    assert results[0][1] > results[1][1] > results[2][1] == 0
    for outs, _ in results[1:]:
        for a, b in zip(results[0][0], outs):
            assert torch.equal(a, b)


def test_layer_deterministic():
    cfg = CONFIGS["batched_decode"]
    outs = []
    for _ in range(2):
        dc = DeviceCache(cfg, DEV)
        dl = DeviceLayer(cfg, 0, DEV)
        got = run_layer(dc, dl, x_dev(cfg, 0, 0), cfg.T, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, 1)
        outs.append((got["out"].clone(), got["y_rows"].clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_empty_calls():
    cfg = CONFIGS["tiny"]
    dc = DeviceCache(cfg, DEV)
    dl = DeviceLayer(cfg, 0, DEV)
    nb = moe.moe_layer_workspace_size(dl.struct, dc.struct, 0, moe.MOE_FFN_AUTO)
    assert moe.moe_layer_forward(dl.struct, dc.struct, None, 0, None, 0, 1, 0, 0, moe.MOE_FFN_AUTO, None,
                                 ws(nb), nb, status(), None) == moe.MOE_OK
