"""The whole layer over an FP4 expert cache (moe_layer_forward_fp4), on the
GPU, against the oracle (FreeToken paper, section 5.1: MXFP4 and NVFP4
expert banks; section 4.1: device-side cache control and a fill copy that
moves every bank of an admitted expert; section 3.2: the decode order).

Decode traces over two layers of one cache: after every call the residency
state (table, owner, stamps, clock) and the bind statistics equal the
oracle's bind on the oracle's routing, bit for bit; every cache slot's code
bytes, scale bytes and tensor scales equal those of the pair that owns it
(the fill copy is byte work); and the layer output matches the oracle's
fp64 layer on the dequantised experts within the output tolerance.  Phi = 1
(every miss filled), 0.25 with the random fill policy (fills and staged
experts in one call) and 0 (no fills); one-token calls (the one-launch
kernel, also checked bitwise against the public per-step calls) and batched
calls (the ring kernel up to 64 routed rows, the tensor-core GEMM above
it)."""
import dataclasses

import numpy as np
import pytest
import torch

import edge_moe_serving_gb300 as moe
from moe_inputs import CONFIGS, gen
from moe_inputs.configs import FILL_RANDOM, LayerConfig
from moe_inputs.device import DeviceLayer, Fp4Cache, x_dev
from oracle import moe_oracle as O
from gpu_helpers import DEV, assert_close, bf16_to_f64, status, status_bits, ws

pytestmark = pytest.mark.gpu

SEED = 71
Q16 = 65536
FP4 = LayerConfig("fp4_layer", T=1, H=2048, E=32, k=6, I=1024, seed=31, n_layers=2, steps=10, cache_slots=10,
                  phi_q16=Q16, min_fill=1, bias="zipf")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


class Weights:
    """fp64 dequantised experts (the oracle's dequantisers), memoised."""

    def __init__(self, cfg, fmt):
        self.cfg, self.fmt, self.d = cfg, fmt, {}

    def __call__(self, layer, e):
        key = (layer, e)
        if key not in self.d:
            H, I = self.cfg.H, self.cfg.I
            if self.fmt == moe.MOE_FP4_MXFP4:
                self.d[key] = O.mx_expert_weights(*gen.mx_expert(SEED, layer, e, H, I))
            else:
                self.d[key] = tuple(O.nvfp4_dequant(*b) for b in gen.nvfp4_expert(SEED, layer, e, H, I))
        return self.d[key]


def _trace(cfg, fmt, T, phi_q16, policy, steps, check_every=1):
    fc = Fp4Cache(cfg, fmt, SEED, DEV)
    layers = [DeviceLayer(cfg, l, DEV) for l in range(cfg.n_layers)]
    weights = Weights(cfg, fmt)
    ref = gen.initial_cache(cfg)
    nb = moe.moe_layer_fp4_workspace_size(layers[0].struct, fc.struct, T)
    w = ws(nb)
    totals = {"n_fill": 0, "n_staged": 0}
    for step in range(steps):
        l = step % cfg.n_layers
        dl = layers[l]
        dl.set_bias(step)
        x = x_dev(cfg, l, step)[:T].contiguous()
        out = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=DEV)
        st = status()
        stats = torch.zeros(8, dtype=torch.int32, device=DEV)
        moe.moe_layer_forward_fp4(dl.struct, fc.struct, x, T, out, phi_q16, cfg.min_fill, policy, 500 + step, w, nb,
                                  st, stats)
        torch.cuda.synchronize()
        assert status_bits(st) == 0, step
        xf = gen.bf16_bits_to_f64(gen.x_bits(cfg, l, step)[:T])
        wr, bias = gen.w_router(cfg, l), gen.bias(cfg, l, step)
        ids = O.select_topk(O.router_logits(xf, wr, bias), cfg.k)[0]
        ref, res = O.bind(ref, l, ids, cfg.E, phi_q16, cfg.min_fill, policy, 500 + step)
        state = fc.state()
        for key in ("table", "owner", "stamp"):
            assert np.array_equal(state[key], np.asarray(ref[key])), (step, key)
        assert state["clock"] == ref["clock"]
        got_stats = dict(zip(moe.BIND_STATS_FIELDS, stats.cpu().numpy().tolist()))
        for key in ("n_unique", "n_hit", "n_miss", "q", "n_fill", "n_overflow", "n_staged"):
            assert got_stats[key] == res["stats"][key], (step, key)
        assert fc.cache_matches_owners(), step
        if step % check_every == 0:
            r = O.layer_forward(xf, wr, bias, cfg.k, lambda e: weights(l, e), E=cfg.E)
            assert_close(bf16_to_f64(out), r["out"], what=f"fmt {fmt} T {T} phi {phi_q16} step {step}")
        for key in totals:
            totals[key] += res["stats"][key]
    return totals


@pytest.mark.parametrize("fmt", [moe.MOE_FP4_MXFP4, moe.MOE_FP4_NVFP4])
def test_fp4_layer_decode_every_miss_filled(fmt):
    t = _trace(FP4, fmt, 1, Q16, 0, 10)
    assert t["n_fill"] > 0 and t["n_staged"] == 0


@pytest.mark.parametrize("fmt", [moe.MOE_FP4_MXFP4, moe.MOE_FP4_NVFP4])
def test_fp4_layer_decode_split_fills_and_staged(fmt):
    t = _trace(FP4, fmt, 1, Q16 // 4, FILL_RANDOM, 10)
    assert t["n_fill"] > 0 and t["n_staged"] > 0


def test_fp4_layer_no_fills_reads_staged_in_place():
    t = _trace(FP4, moe.MOE_FP4_MXFP4, 1, 0, 0, 4)
    assert t["n_fill"] == 0 and t["n_staged"] > 0


@pytest.mark.parametrize("fmt,T", [(moe.MOE_FP4_MXFP4, 8), (moe.MOE_FP4_NVFP4, 8), (moe.MOE_FP4_MXFP4, 16),
                                   (moe.MOE_FP4_NVFP4, 16)])
def test_fp4_layer_batched_calls(fmt, T):
    """48 routed rows (one ring launch) and 96 routed rows (the tensor-core
    GEMM)."""
    cfg = dataclasses.replace(FP4, T=T)
    t = _trace(cfg, fmt, T, Q16 // 4, FILL_RANDOM, 4, check_every=1)
    assert t["n_fill"] > 0


def test_fp4_layer_nvfp4_rejects_calls_that_fit_neither_kernel_before_the_bind():
    """An NVFP4 call whose shape neither FFN kernel takes (rows of 1040
    inputs) is refused before any launch: the residency state is unchanged."""
    cfg = dataclasses.replace(FP4, H=1040, I=1040, E=8, cache_slots=4)
    fc = Fp4Cache(cfg, moe.MOE_FP4_NVFP4, SEED, DEV)
    dl = DeviceLayer(cfg, 0, DEV)
    before = fc.state()
    x = x_dev(cfg, 0, 0)[:1].contiguous()
    out = torch.empty((1, cfg.H), dtype=torch.bfloat16, device=DEV)
    nb = moe.moe_layer_fp4_workspace_size(dl.struct, fc.struct, 1)
    n0 = moe.moe_kernel_launch_count()
    rc = moe.lib().moe_layer_forward_fp4(dl.struct, fc.struct, x.data_ptr(), 1, out.data_ptr(), Q16, 1, 0, 0,
                                         ws(nb).data_ptr(), nb, None, None, None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_kernel_launch_count() == n0
    after = fc.state()
    for key in ("table", "owner", "stamp"):
        assert np.array_equal(before[key], after[key])


@pytest.mark.parametrize("fmt", [moe.MOE_FP4_MXFP4, moe.MOE_FP4_NVFP4])
def test_fp4_layer_one_token_is_one_launch_matching_the_per_step_calls(fmt):
    """A one-token call runs as one kernel and matches the public calls
    chained on the same cache: router + top-k, dispatch, the FP4 expert FFN,
    the combine (phi = 0: the call changes no binding, so both read the same
    slot table).  The two routers sum the logits in different orders, so
    the gate weights may differ in their last bits: every output is within 2
    bf16 units in the last place of the chained one (other experts would
    differ by whole units), and almost all are equal."""
    cfg = FP4
    fc = Fp4Cache(cfg, fmt, SEED, DEV)
    E, H, I, k = cfg.E, cfg.H, cfg.I, cfg.k
    for step in range(3):
        l = step % cfg.n_layers
        dl = DeviceLayer(cfg, l, DEV, step)
        x = x_dev(cfg, l, step)[:1].contiguous()
        # the public calls
        i32 = lambda n: torch.empty(n, dtype=torch.int32, device=DEV)
        ids, counts, offsets, perm, inv = i32(k), i32(E), i32(E + 1), i32(k), i32(k)
        w = torch.empty(k, dtype=torch.float32, device=DEV)
        y = torch.empty((k, H), dtype=torch.float32, device=DEV)
        ref = torch.empty((1, H), dtype=torch.bfloat16, device=DEV)
        st = status()
        nr, nd = moe.moe_route_topk_workspace_size(1, H, E), moe.moe_dispatch_workspace_size(1, k, E)
        moe.moe_route_topk(x, 1, H, dl.w_router, dl.bias, E, k, ids, w, None, ws(nr), nr, st)
        moe.moe_dispatch(ids, 1, k, E, counts, offsets, perm, inv, None, H, None, ws(nd), nd, st)
        c = fc.struct
        if fmt == moe.MOE_FP4_MXFP4:
            pools = [moe.moe_pool_mxfp4(q.gate_q, q.gate_s, q.up_q, q.up_s, q.down_q, q.down_s, q.n_slots, 0)
                     for q in (c.cache, c.staging)]
            nf = moe.moe_expert_ffn_mxfp4_workspace_size(1, k, H, I)
            moe.moe_expert_ffn_mxfp4(pools[0], pools[1], fc.table, cfg.n_layers, l, E, H, I, counts, offsets, perm, x,
                                     1, k, y, ws(nf), nf, st)
        else:
            nf = moe.moe_expert_ffn_nvfp4_workspace_size(1, k, H, I)
            moe.moe_expert_ffn_nvfp4(c.cache, c.staging, fc.table, cfg.n_layers, l, E, H, I, counts, offsets, perm,
                                     x, 1, k, y, ws(nf), nf, st)
        moe.moe_combine(y, w, 1, k, H, ref, None, st)
        torch.cuda.synchronize()
        assert status_bits(st) == 0
        # the layer call
        out = torch.empty((1, H), dtype=torch.bfloat16, device=DEV)
        nb = moe.moe_layer_fp4_workspace_size(dl.struct, fc.struct, 1)
        st2 = status()
        before = moe.moe_kernel_launch_count()
        w2 = ws(nb)
        moe.moe_layer_forward_fp4(dl.struct, fc.struct, x, 1, out, 0, 1, 0, 0, w2, nb, st2, None)
        torch.cuda.synchronize()
        assert moe.moe_kernel_launch_count() - before == 1
        assert status_bits(st2) == 0
        a, b = out.float(), ref.float()
        assert torch.all((a - b).abs() <= 2.0 ** -7 * b.abs() + 1e-30), (fmt, step)
        assert (a == b).float().mean().item() >= 0.95, (fmt, step)


@pytest.mark.parametrize("fmt", [moe.MOE_FP4_MXFP4, moe.MOE_FP4_NVFP4])
def test_fp4_layer_one_launch_at_the_decode_shape(fmt):
    """The one-launch kernel at the decode layer's shape (256 experts, so
    CTAs score two router rows; hidden 4096, intermediate 2048; 95 cache
    slots, every miss filled): three steps, state and stats bit-exact against
    the oracle's bind, cache bytes (and NVFP4 tensor scales) equal to the
    owners', outputs within the tolerance of the oracle's fp64 layer."""
    cfg = dataclasses.replace(CONFIGS["decode"], n_layers=1)
    t = _trace(cfg, fmt, 1, Q16, 0, 3)
    assert t["n_fill"] > 0


@pytest.mark.parametrize("fmt", [moe.MOE_FP4_MXFP4, moe.MOE_FP4_NVFP4])
def test_fp4_layer_one_token_outside_the_one_launch_shapes(fmt):
    """One-token calls whose rows the ring kernel does not take (hidden 1536)
    run the per-step launches: router, bind with the FP4 fill copy, dispatch,
    the tensor-core GEMM on 32-row chunks, combine.  Traces at phi = 1 and
    0.25 (random fills): state, stats and cache bytes bit-exact, outputs
    within tolerance."""
    cfg = dataclasses.replace(FP4, H=1536, I=1024, E=16, cache_slots=6)
    t1 = _trace(cfg, fmt, 1, Q16, 0, 4)
    t2 = _trace(cfg, fmt, 1, Q16 // 4, FILL_RANDOM, 4)
    assert t1["n_fill"] > 0 and t2["n_staged"] > 0
