"""GPU parity of the prefill-sized layer calls against the fp64 oracle, at
full size and in the configuration the benchmark times.

* The 8192-token prefill block (every expert resident): routing ids and the
  dispatch of all tokens bit-exact; the layer output of 1024 seeded tokens
  within the output tolerance, once as the benchmark calls the layer (expert
  rows kept inside the library, bf16 on the GEMM path) and once with the
  fp32 expert rows returned to the caller, whose rows are then compared in
  full for the smallest group, two random groups and a sample of the largest.
* The long-prefill stack: the four 16384-token layers run back to back on one
  cache of 113 resident (layer, expert) pairs with no fills (phi = 0), as in
  the benchmark.  After every layer: ids and dispatch of all tokens, the
  residency state and the bind statistics bit-exact against the oracle's
  bind, and the output of 1024 seeded tokens within the tolerance.

The oracle evaluates only the sampled tokens (every step of the layer acts
per token, so that is the full block's output restricted to them).
"""
import numpy as np
import pytest
import torch

import edge_moe_serving_gb300 as moe
from moe_inputs import CONFIGS, gen
from moe_inputs.device import DeviceCache, DeviceLayer, x_dev
from oracle import moe_oracle as O
from gpu_helpers import DEV, assert_close, bf16_to_f64, oracle_tokens, run_layer

pytestmark = pytest.mark.gpu

N_TOKENS = 1024          # sampled tokens per layer whose whole output row is compared
LARGEST_ROWS = 256       # rows of the largest expert group compared one by one


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _full_routing(cfg, layer):
    x = gen.bf16_bits_to_f64(gen.x_bits(cfg, layer, 0))
    ids, _ = O.select_topk(O.router_logits(x, gen.w_router(cfg, layer), gen.bias(cfg, layer, 0)), cfg.k)
    return x, ids


def _check_routing(got, ids_ref, cfg, what):
    ids = got["topk_ids"].cpu().numpy().reshape(cfg.T, cfg.k)
    assert np.array_equal(ids, ids_ref), what
    counts, offsets, perm, inv = O.dispatch(ids_ref, cfg.E)
    assert np.array_equal(got["counts"].cpu().numpy(), counts), what
    assert np.array_equal(got["offsets"].cpu().numpy(), offsets), what
    assert np.array_equal(got["perm"].cpu().numpy(), perm), what
    assert np.array_equal(got["inv_perm"].cpu().numpy(), inv), what
    return counts, offsets, perm


def _check_tokens(got, cfg, layer, toks, what):
    ref, ids = oracle_tokens(cfg, layer, 0, toks)
    assert np.array_equal(got["topk_ids"].cpu().numpy().reshape(cfg.T, cfg.k)[toks], ids), what
    assert_close(bf16_to_f64(got["out"])[toks], ref, what=f"{what}: output of {len(toks)} tokens")


def test_prefill_layer_1024_tokens():
    cfg = CONFIGS["prefill"]
    dc = DeviceCache(cfg, DEV)
    dl = DeviceLayer(cfg, 0, DEV)
    x, ids_ref = _full_routing(cfg, 0)
    toks = np.sort(np.random.default_rng(8192).choice(cfg.T, N_TOKENS, replace=False))
    # as the benchmark calls it: no caller buffer for the expert rows
    got = run_layer(dc, dl, x_dev(cfg, 0, 0), cfg.T, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, 1000,
                    want_y_rows=False)
    assert got["status"] == 0
    _check_routing(got, ids_ref, cfg, "prefill (benchmark path)")
    _check_tokens(got, cfg, 0, toks, "prefill (benchmark path)")
    # fp32 expert rows returned to the caller
    got = run_layer(dc, dl, x_dev(cfg, 0, 0), cfg.T, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, 1000)
    assert got["status"] == 0
    counts, offsets, perm = _check_routing(got, ids_ref, cfg, "prefill (fp32 rows)")
    _check_tokens(got, cfg, 0, toks, "prefill (fp32 rows)")
    y = got["y_rows"].cpu().numpy()
    rng = np.random.default_rng(3)
    active = np.nonzero(counts)[0]
    big = int(active[np.argmax(counts[active])])
    small = int(active[np.argmin(counts[active])])
    picks = {small: None, big: None}
    for e in rng.choice(active, 2, replace=False):
        picks.setdefault(int(e), None)
    for e in picks:
        rows = perm[offsets[e]:offsets[e + 1]]
        if e == big and rows.size > LARGEST_ROWS:
            rows = np.sort(rng.choice(rows, LARGEST_ROWS, replace=False))
        wg, wu, wd = gen.expert_f64(cfg, 0, e)
        ref = O.swiglu_expert(x[rows // cfg.k], wg, wu, wd)
        assert_close(y[rows], ref, what=f"prefill expert {e} ({counts[e]} rows)")


def test_long_prefill_stack_one_cache():
    cfg = CONFIGS["long_prefill"]
    dc = DeviceCache(cfg, DEV)
    layers = [DeviceLayer(cfg, l, DEV) for l in range(cfg.n_layers)]
    ref_state = gen.initial_cache(cfg)
    rng = np.random.default_rng(16384)
    for l in range(cfg.n_layers):
        got = run_layer(dc, layers[l], x_dev(cfg, l, 0), cfg.T, cfg.phi_q16, cfg.min_fill, cfg.fill_policy,
                        1000 + l, want_y_rows=False)
        what = f"long prefill layer {l} of the stack"
        assert got["status"] == 0, what
        _, ids_ref = _full_routing(cfg, l)
        _check_routing(got, ids_ref, cfg, what)
        ref_state, res = O.bind(ref_state, l, ids_ref, cfg.E, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, 1000 + l)
        state = dc.state()
        for key in ("table", "owner", "stamp"):
            assert np.array_equal(state[key], np.asarray(ref_state[key])), (what, key)
        assert state["clock"] == ref_state["clock"], what
        for key, v in res["stats"].items():
            assert got["stats"][key] == v, (what, key)
        # the layer reads some experts from the cache pool and the rest in place from the staging pool
        assert 0 < res["stats"]["n_hit"] < res["stats"]["n_unique"], what
        toks = np.sort(rng.choice(cfg.T, N_TOKENS, replace=False))
        _check_tokens(got, cfg, l, toks, what)
