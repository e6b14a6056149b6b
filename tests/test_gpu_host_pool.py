"""The source-of-truth expert pool in host memory, on the GPU.

* Decode with a host-resident staging pool (FreeToken paper, section 3: the
  two-level expert hierarchy; section 3.2, Eq. 1-4): the GPU copies the fill
  set F into its HBM cache slots and reads the in-place set C from host
  memory over NVLink-C2C, with plain loads only (the fill copy, and a
  weight-streaming GEMV pass over the experts bound to the host pool).  Over
  traces at phi = 0, 0.25 and 1, every layer output matches the oracle within
  the output tolerance and the residency state after every step equals the
  oracle's bind; the outputs also match the same trace with the staging pool
  in HBM within the tolerance (not bitwise: the experts read in place run on
  a different kernel, with another fp32 summation order).  One-token calls
  and 32-token calls (whose cache-pool experts run on the tensor-core GEMM).
* Full-layer double-buffered prefill (section 3.1, Figure 2 (1)): a stack of
  layers whose experts stream from a host pool into two HBM layer buffers
  while the previous layer computes; the outputs equal the layer-by-layer
  calls on an all-HBM cache bitwise, with overlap and on demand, and the
  oracle's on the tokens whose routing is decided by a gap of at least 1e-3.
"""
import dataclasses

import numpy as np
import pytest
import torch

import edge_moe_serving_gb300 as moe
from moe_inputs import CONFIGS, gen
from moe_inputs.configs import LayerConfig
from moe_inputs.device import DeviceCache, DeviceLayer, x_dev
from oracle import moe_oracle as O
from gpu_helpers import DEV, ExpertCache, assert_close, bf16_to_f64, oracle_layer, run_layer, status, status_bits, ws

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _trace(cfg, staging_host, steps, phi_q16, T, wc=None):
    """Runs the trace; checks the state against the oracle's bind after every
    step and, when an expert cache is given, the output against the oracle."""
    dc = DeviceCache(cfg, DEV, staging_host=staging_host)
    dl = DeviceLayer(cfg, 0, DEV)
    ref = gen.initial_cache(cfg)
    outs, fills, staged = [], 0, 0
    for step in range(steps):
        dl.set_bias(step)
        xb = gen.x_bits(cfg, 0, step)[:T]
        got = run_layer(dc, dl, x_dev(cfg, 0, step)[:T].contiguous(), T, phi_q16, cfg.min_fill, cfg.fill_policy,
                        100 + step, want_y_rows=False)
        assert got["status"] == 0
        x = gen.bf16_bits_to_f64(xb)
        lr = oracle_layer(cfg, 0, step, wc, x_bits=xb) if wc is not None else None
        ids = lr["ids"] if lr is not None else O.select_topk(
            O.router_logits(x, gen.w_router(cfg, 0), gen.bias(cfg, 0, step)), cfg.k)[0]
        ref, res = O.bind(ref, 0, ids, cfg.E, phi_q16, cfg.min_fill, cfg.fill_policy, 100 + step)
        state = dc.state()
        for key in ("table", "owner", "stamp"):
            assert np.array_equal(state[key], np.asarray(ref[key])), (step, key)
        if lr is not None:
            assert_close(bf16_to_f64(got["out"]), lr["out"], what=f"{cfg.name} step {step} phi_q16 {phi_q16}")
        fills += res["stats"]["n_fill"]
        staged += res["stats"]["n_staged"]
        outs.append(got["out"].clone())
    return outs, fills, staged


def _check_against_hbm(host, hbm, what):
    for step, (a, b) in enumerate(zip(host, hbm)):
        assert_close(bf16_to_f64(a), bf16_to_f64(b), what=f"{what} step {step}: host pool vs HBM pool")


def test_host_pool_tiny_one_token_calls():
    """Smallest case first: the tiny layer with 3 cache slots, one token per
    call; phi = 0 (every miss read in place), 0.25 (fills and in-place reads
    in the same call) and 1 (every miss filled)."""
    cfg = dataclasses.replace(CONFIGS["tiny"], cache_slots=3, steps=8)
    wc = ExpertCache(cfg)
    for phi in (0, 16384, 65536):
        host, fills, staged = _trace(cfg, True, 8, phi, 1, wc)
        hbm, _, _ = _trace(cfg, False, 8, phi, 1)
        assert (fills > 0) == (phi > 0) and (staged > 0) == (phi < 65536)
        _check_against_hbm(host, hbm, f"tiny phi_q16 {phi}")


def test_host_pool_decode_one_token_calls():
    """The decode layer shape (32 experts, 12 cache slots) at phi = 0.25."""
    cfg = CONFIGS["decode_profile"]
    host, fills, staged = _trace(cfg, True, 6, 16384, 1, ExpertCache(cfg, cap=8))
    hbm, _, _ = _trace(cfg, False, 6, 16384, 1)
    assert fills > 0 and staged > 0
    _check_against_hbm(host, hbm, "decode shape")


def test_host_pool_batched_decode_gemm_calls():
    cfg = CONFIGS["batched_decode"]
    host, fills, staged = _trace(cfg, True, 3, cfg.phi_q16, cfg.T, ExpertCache(cfg, cap=64))
    hbm, _, _ = _trace(cfg, False, 3, cfg.phi_q16, cfg.T)
    assert fills > 0 and staged > 0
    _check_against_hbm(host, hbm, "batched decode")


STACK = LayerConfig("stack_small", T=256, H=1024, E=16, k=4, I=1024, seed=21, n_layers=3)


def _stack_state(cfg):
    """Residency arrays of the double-buffered call: every expert of layer l
    is slot e of its layer buffer."""
    E, L = cfg.E, cfg.n_layers
    c = moe.moe_cache()
    table = torch.from_numpy(np.tile(np.arange(E, dtype=np.int32), L)).to(DEV)
    owner = torch.arange(E, dtype=torch.int32, device=DEV)
    stamp = torch.zeros(E, dtype=torch.int32, device=DEV)
    clock = torch.zeros(1, dtype=torch.int32, device=DEV)
    c.slot_table, c.owner, c.stamp, c.clock = table.data_ptr(), owner.data_ptr(), stamp.data_ptr(), clock.data_ptr()
    c.n_layers, c.E, c.H, c.I = L, E, cfg.H, cfg.I
    return c, (table, owner, stamp, clock)


@pytest.mark.parametrize("overlap", [1, 0])
def test_prefill_double_buffered_stack(overlap):
    cfg = STACK
    L, E, T, H = cfg.n_layers, cfg.E, cfg.T, cfg.H
    src = DeviceCache(cfg, DEV, staging_host=True)        # the source pool: every (layer, expert) in host memory
    bufs = [[torch.empty((E,) + gen.bank_shape(cfg, b), dtype=torch.bfloat16, device=DEV) for b in range(3)]
            for _ in range(2)]
    source = moe.moe_pool(*[t.data_ptr() for t in src.staging], L * E, 1)
    layer_buf = [moe.moe_pool(*[t.data_ptr() for t in bb], E) for bb in bufs]
    state, keep = _stack_state(cfg)
    layers = [DeviceLayer(cfg, l, DEV) for l in range(L)]
    xs = [x_dev(cfg, l, 0) for l in range(L)]
    outs = [torch.empty((T, H), dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    nbytes = moe.moe_layer_workspace_size(layers[0].struct, src.struct, T, moe.MOE_FFN_AUTO)
    w = ws(nbytes)
    st = status()
    main, copy = torch.cuda.Stream(), torch.cuda.Stream()
    moe.moe_prefill_double_buffered([dl.struct for dl in layers], source, layer_buf, state, xs, T, outs,
                                    moe.MOE_FFN_AUTO, overlap, w, nbytes, st, main, copy)
    torch.cuda.synchronize()
    assert status_bits(st) == 0
    # the same layers on an all-HBM cache, layer by layer
    hbm = DeviceCache(dataclasses.replace(cfg, cache_slots=None), DEV)
    for l in range(L):
        got = run_layer(hbm, layers[l], xs[l], T, 0, 0, 0, 0, want_y_rows=False)
        assert got["status"] == 0
        assert torch.equal(got["out"], outs[l]), (overlap, l)
        # the oracle on the tokens whose routing has a gap of at least 1e-3
        x = gen.bf16_bits_to_f64(gen.x_bits(cfg, l, 0))
        lg = O.router_logits(x, gen.w_router(cfg, l), gen.bias(cfg, l, 0))
        toks = np.nonzero(O.topk_gap(lg, cfg.k) >= 1e-3)[0][:64]
        ref = O.layer_forward(x[toks], gen.w_router(cfg, l), gen.bias(cfg, l, 0), cfg.k,
                              lambda e: gen.expert_f64(cfg, l, e), E=E)["out"]
        assert_close(bf16_to_f64(outs[l])[toks], ref, what=f"double-buffered layer {l}")
    del keep


def test_prefill_double_buffered_argument_checks():
    cfg = STACK
    L, E = cfg.n_layers, cfg.E
    layers = (moe.moe_layer * L)(*[moe.moe_layer(16, None, l, E, cfg.k, cfg.H, cfg.I) for l in range(L)])
    state, keep = _stack_state(cfg)
    src = moe.moe_pool(256, 256, 256, L * E)
    bufs = (moe.moe_pool * 2)(moe.moe_pool(256, 256, 256, E), moe.moe_pool())
    fn = moe.lib().moe_prefill_double_buffered
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    xs = (moe.c_void_p * L)(*([256] * L))
    assert fn(layers, L, src, bufs, state, xs, 0, xs, 0, 1, None, 0, None, s1.cuda_stream,
              s2.cuda_stream) == moe.MOE_OK                                    # T = 0
    short = moe.moe_pool(256, 256, 256, L * E - 1)
    assert fn(layers, L, short, bufs, state, xs, 8, xs, 0, 1, None, 0, None, s1.cuda_stream,
              s2.cuda_stream) == moe.MOE_ERR_INVALID_ARG                       # source too small
    assert fn(layers, L, src, bufs, state, xs, 8, xs, 0, 1, None, 0, None, s1.cuda_stream,
              s1.cuda_stream) == moe.MOE_ERR_INVALID_ARG                       # one stream for both
    layers[1].layer = 2
    assert fn(layers, L, src, bufs, state, xs, 8, xs, 0, 1, None, 0, None, s1.cuda_stream,
              s2.cuda_stream) == moe.MOE_ERR_INVALID_ARG                       # layer index out of place
    del keep
