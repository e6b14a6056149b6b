"""GPU parity of the MXFP4 expert FFN (moe_expert_ffn_mxfp4) against the
oracle: the same SwiGLU experts on the fp64 dequantised banks (FP4 E2M1
elements, E8M0 scales per 32 inputs), through the slot table into both pools,
on ragged groups, every row-chunk width, the decode and batched-decode shapes,
and the unbound / out-of-range slot errors."""
import numpy as np
import pytest
import torch

import edge_moe_serving_gb300 as moe
from moe_inputs import gen
from moe_inputs.device import MxPool
from oracle import moe_oracle as O
from gpu_helpers import DEV, assert_close, status, status_bits, ws

pytestmark = pytest.mark.gpu

SEED = 41


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _route(rng, T, k, experts):
    return np.stack([np.sort(rng.choice(experts, k, replace=False)) for _ in range(T)]).astype(np.int32)


def _run(T, k, E, H, I, n_layers, layer, cached, staged, seed, unbound=(), bad=(), active=None):
    """cached: experts placed in cache-pool slots (in a seeded order); staged:
    experts bound to the staging pool; unbound: entry -1; bad: a cache slot
    past the pool.  Returns (y from the GPU, oracle rows, status bits, ids)."""
    rng = np.random.default_rng(seed)
    ids = _route(rng, T, k, np.arange(E) if active is None else np.asarray(active))
    x_bits = gen.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    n_cache = max(len(cached), 1)
    slots = rng.permutation(n_cache)
    table = np.full(n_layers * E, -1, np.int32)
    base = layer * E
    cache_experts, staging_experts = {}, {}
    for s, e in zip(slots, cached):
        table[base + e] = s
        cache_experts[int(s)] = gen.mx_expert(SEED, layer, int(e), H, I)
    for e in staged:
        table[base + e] = gen.STAGING_TAG | (base + e)
        staging_experts[base + int(e)] = gen.mx_expert(SEED, layer, int(e), H, I)
    for e in unbound:
        table[base + e] = -1
    for e in bad:
        table[base + e] = n_cache + 3
    pool_a = MxPool(n_cache, H, I, cache_experts, DEV)
    pool_b = MxPool(n_layers * E, H, I, staging_experts, DEV) if len(staged) else None

    counts, offsets, perm, inv = O.dispatch(ids, E)
    dev_i32 = lambda a: torch.from_numpy(np.asarray(a, np.int32)).to(DEV)
    x = torch.from_numpy(x_bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    R = T * k
    y = torch.full((R, H), 7.0, dtype=torch.float32, device=DEV)
    nb = moe.moe_expert_ffn_mxfp4_workspace_size(T, k, H, I)
    st = status()
    moe.moe_expert_ffn_mxfp4(pool_a.struct, pool_b.struct if pool_b else None, dev_i32(table), n_layers, layer, E,
                             H, I, dev_i32(counts), dev_i32(offsets), dev_i32(perm), x, T, k, y, ws(nb), nb, st)
    torch.cuda.synchronize()

    xf = gen.bf16_bits_to_f64(x_bits)
    ref = np.full((R, H), np.nan)
    weights = {}
    for i, e in enumerate(ids.reshape(-1)):
        e = int(e)
        if e in unbound or e in bad:
            continue
        if e not in weights:
            weights[e] = O.mx_expert_weights(*gen.mx_expert(SEED, layer, e, H, I))
        ref[i] = O.swiglu_expert(xf[i // k][None, :], *weights[e])[0]
    return y.cpu().numpy().astype(np.float64), ref, status_bits(st), ids


def _check(y, ref, what):
    ok = ~np.isnan(ref[:, 0])
    assert ok.any()
    assert_close(y[ok], ref[ok], what=what)


@pytest.mark.parametrize("T,k,E,H,I", [(5, 3, 12, 256, 160), (2, 4, 16, 512, 256), (1, 2, 6, 64, 96),
                                       (9, 5, 7, 128, 64)])
def test_mxfp4_ffn_small_shapes_both_pools(T, k, E, H, I):
    """Groups of 1..T rows (row chunks of 1, 2 and 4 plus ragged tails),
    experts in the cache pool and in the staging pool, layer 1 of 2."""
    experts = list(range(E))
    cached, staged = experts[: E // 2 + 1], experts[E // 2 + 1:]
    y, ref, st, _ = _run(T, k, E, H, I, 2, 1, cached, staged, seed=T * 100 + E)
    assert st == 0
    _check(y, ref, f"mxfp4 T={T} k={k} E={E} H={H} I={I}")


def test_mxfp4_ffn_decode_shape():
    """One token, 6 of 256 experts, hidden 4096, intermediate 2048."""
    rng = np.random.default_rng(5)
    active = np.sort(rng.choice(256, 6, replace=False))
    y, ref, st, ids = _run(1, 6, 256, 4096, 2048, 1, 0, list(active[:5]), list(active[5:]), seed=6,
                           active=active)
    assert st == 0 and sorted(ids[0].tolist()) == active.tolist()
    _check(y, ref, "mxfp4 decode shape")


def test_mxfp4_ffn_batched_decode_shape():
    """32 tokens, top-8 of 128 experts routed over 24 of them (groups of ~10
    rows: several row chunks each), hidden 2048, intermediate 768."""
    rng = np.random.default_rng(8)
    active = np.sort(rng.choice(128, 24, replace=False))
    y, ref, st, _ = _run(32, 8, 128, 2048, 768, 1, 0, list(active[:18]), list(active[18:]), seed=9,
                         active=active)
    assert st == 0
    _check(y, ref, "mxfp4 batched decode shape")


def test_mxfp4_ffn_unbound_and_bad_slot_rows_left_unwritten():
    T, k, E, H, I = 4, 3, 8, 64, 64
    y, ref, st, ids = _run(T, k, E, H, I, 1, 0, [0, 1, 2, 3, 4], [], seed=3, active=np.arange(8),
                           unbound=(5,), bad=(6,))
    flat = ids.reshape(-1)
    skipped = np.isin(flat, [5, 6, 7])
    if np.isin(flat, 5).any():
        assert st & moe.MOE_DEV_ERR_UNBOUND
    if np.isin(flat, 6).any():
        assert st & moe.MOE_DEV_ERR_BAD_SLOT
    assert np.all(y[skipped] == 7.0)            # sentinel kept: nothing written for those experts
    keep = ~skipped
    _check(y[keep], ref[keep], "mxfp4 rows of bound experts")


def test_mxfp4_ffn_empty_call_launches_nothing():
    pool = MxPool(1, 64, 64, {}, DEV)
    before = moe.moe_kernel_launch_count()
    moe.moe_expert_ffn_mxfp4(pool.struct, None, torch.zeros(8, dtype=torch.int32, device=DEV), 1, 0, 8, 64, 64,
                             None, None, None, None, 0, 2, None, None, 0, None)
    assert moe.moe_kernel_launch_count() == before


@pytest.mark.parametrize("T,H,I,k", [(1, 1024, 1024, 4), (1, 2048, 4096, 6), (1, 4096, 1024, 5), (3, 1024, 2048, 4),
                                     (8, 1024, 1024, 8)])
def test_mxfp4_ffn_ring_kernel(T, H, I, k):
    """Calls of up to 64 routed rows run on the weight-streaming ring kernel
    (one launch): experts in both pools, layer 1 of 2, every row width it
    takes, one token and several."""
    E = 16
    experts = list(range(E))
    before = moe.moe_kernel_launch_count()
    y, ref, st, _ = _run(T, k, E, H, I, 2, 1, experts[:9], experts[9:], seed=T * 1000 + H + I + k)
    assert moe.moe_kernel_launch_count() - before == 1
    assert st == 0
    _check(y, ref, f"mxfp4 ring kernel T={T} H={H} I={I} k={k}")


def test_mxfp4_ffn_one_token_unbound_and_bad_slot():
    T, k, E, H, I = 1, 4, 8, 1024, 2048
    y, ref, st, ids = _run(T, k, E, H, I, 1, 0, [0, 1, 3, 4], [], seed=12, active=np.array([0, 2, 3, 5]),
                           unbound=(2,), bad=(5,))
    assert sorted(ids[0].tolist()) == [0, 2, 3, 5]
    assert st & moe.MOE_DEV_ERR_UNBOUND and st & moe.MOE_DEV_ERR_BAD_SLOT
    skipped = np.isin(ids.reshape(-1), [2, 5])
    assert np.all(y[skipped] == 7.0)
    _check(y[~skipped], ref[~skipped], "mxfp4 ring kernel rows of bound experts")


@pytest.mark.parametrize("T,k,H,I", [(2, 1, 128, 64), (1, 2, 1024, 1024)])
def test_mxfp4_ffn_special_block_scales(T, k, H, I):
    """E8M0 scales 0 (2^-127), 254 (2^127) and 255 (NaN) of the OCP MX
    encoding.  Inputs 0..31 of the token rows are about 2^120 and inputs
    32..63 about 2^-132, and every gate and up row scales those blocks by
    2^-127 and 2^127, so both contribute order-one terms; the other blocks
    are ordinary.  One gate row of expert 0 has a NaN block scale, which makes
    every output of its routed row NaN; one down row of expert 1 has a NaN
    scale, which makes one output element of the other routed row NaN.
    Everything else matches the oracle's fp64 dequantisation.  Two tokens of
    one expert each run on the table kernel, one token routed to both experts
    on the ring kernel."""
    E = 2
    rng = np.random.default_rng(77)
    experts = {}
    for e in range(E):
        gq, gs, uq, us, dq, ds = (np.array(a) for a in gen.mx_expert(SEED, 0, e, H, I))
        for s in (gs, us):
            s[:, 0] = 0          # 2^-127 on inputs 0..31
            s[:, 1] = 254        # 2^127 on inputs 32..63
        if e == 0:
            gs[3, 2] = 255       # NaN: gate row 3 of expert 0
        else:
            ds[5, 0] = 255       # NaN: down row 5 of expert 1
        experts[e] = (gq, gs, uq, us, dq, ds)
    xf = rng.standard_normal((T, H)).astype(np.float32)
    xf[:, :32] *= np.float32(2.0 ** 120)
    xf[:, 32:64] *= np.float32(2.0 ** -132)
    x_bits = gen.f32_to_bf16_bits(xf)
    # two tokens with one expert each (table kernel), or one token routed to both (ring kernel)
    ids = np.array([[0], [1]] if T == 2 else [[0, 1]], np.int32)
    counts, offsets, perm, _ = O.dispatch(ids, E)
    pool = MxPool(E, H, I, experts, DEV)
    dev_i32 = lambda a: torch.from_numpy(np.asarray(a, np.int32)).to(DEV)
    x = torch.from_numpy(x_bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    y = torch.zeros((T * k, H), dtype=torch.float32, device=DEV)
    nb = moe.moe_expert_ffn_mxfp4_workspace_size(T, k, H, I)
    st = status()
    moe.moe_expert_ffn_mxfp4(pool.struct, None, dev_i32(np.arange(E)), 1, 0, E, H, I, dev_i32(counts),
                             dev_i32(offsets), dev_i32(perm), x, T, k, y, ws(nb), nb, st)
    torch.cuda.synchronize()
    assert status_bits(st) == 0
    got = y.cpu().numpy().astype(np.float64)
    xd = gen.bf16_bits_to_f64(x_bits)
    ref = np.stack([O.swiglu_expert(xd[r // k][None, :], *O.mx_expert_weights(*experts[int(ids.reshape(-1)[r])]))[0]
                    for r in range(T * k)])
    assert np.isnan(ref[0]).all() and np.isnan(got[0]).all()
    nan1 = np.isnan(ref[1])
    assert nan1.tolist() == [c == 5 for c in range(H)]
    assert np.array_equal(np.isnan(got[1]), nan1)
    # the rescaled blocks carry real terms: dropping the 2^-127 block moves the reference by 16% (26% at
    # hidden 1024; relative Frobenius), the 2^127 block by 98% (83%), far beyond the tolerance
    assert np.abs(ref[1][~nan1]).max() > 0.05
    assert_close(got[1][~nan1], ref[1][~nan1], what="mxfp4 rows with block scales 0 and 254")


@pytest.mark.parametrize("T,k,E,H,I", [(64, 4, 8, 1024, 512), (320, 4, 4, 512, 512), (24, 6, 12, 1024, 768),
                                       (40, 3, 6, 2048, 256)])
def test_mxfp4_ffn_tensor_core_gemm(T, k, E, H, I):
    """Calls beyond the ring kernel whose shapes the tensor-core GEMM takes:
    the token rows gathered in dispatch order, then the gate/up and down
    launches (three launches in all).  Groups of a few rows to several
    256-row chunks (320 tokens over 4 experts), the thin 32-row chunks of
    calls of at most 32 tokens (24 tokens), scale rows of 24 bytes
    (intermediate 768), experts in both pools, layer 1 of 2."""
    experts = list(range(E))
    before = moe.moe_kernel_launch_count()
    y, ref, st, _ = _run(T, k, E, H, I, 2, 1, experts[: E // 2 + 1], experts[E // 2 + 1:], seed=T * 7 + E + H)
    assert moe.moe_kernel_launch_count() - before == 3
    assert st == 0
    _check(y, ref, f"mxfp4 tensor-core GEMM T={T} k={k} E={E} H={H} I={I}")


def test_mxfp4_ffn_tensor_core_gemm_special_block_scales():
    """The tensor-core GEMM's exact expansion at the ends of its range: gate
    and up rows scale inputs 0..31 by 2^-127 (E8M0 byte 0: bf16 subnormal
    weights) and inputs 32..63 by 2^125 (byte 252, the largest scale every
    code fits in bf16 with).  Each token has one nonzero input in each of
    those blocks, about 2^125 at input 0 and in [2^-126, 2^-125) at input 32,
    so that both blocks carry one order-one term and the outputs stay near
    unit scale.  A NaN block scale (255) in gate row 3 of expert 0 makes every
    output of its rows NaN; one in down row 5 of expert 1 makes element 5 of
    its rows NaN."""
    T, k, E, H, I = 40, 1, 2, 512, 256
    rng = np.random.default_rng(78)
    experts = {}
    for e in range(E):
        gq, gs, uq, us, dq, ds = (np.array(a) for a in gen.mx_expert(SEED, 0, e, H, I))
        for s in (gs, us):
            s[:, 0] = 0          # 2^-127 on inputs 0..31
            s[:, 1] = 252        # 2^125 on inputs 32..63
        if e == 0:
            gs[3, 2] = 255
        else:
            ds[5, 0] = 255
        experts[e] = (gq, gs, uq, us, dq, ds)
    xf = rng.standard_normal((T, H)).astype(np.float32)
    xf[:, 0] *= np.float32(2.0 ** 125)
    mag = (1.0 + 0.9 * rng.random(T)) * 2.0 ** -126                  # normal bf16 values in [2^-126, 2^-125)
    xf[:, 32] = (np.sign(xf[:, 32]) * mag).astype(np.float32)
    xf[:, 1:32] = 0.0
    xf[:, 33:64] = 0.0
    x_bits = gen.f32_to_bf16_bits(xf)
    ids = (np.arange(T) % 2).astype(np.int32)[:, None]
    counts, offsets, perm, _ = O.dispatch(ids, E)
    pool = MxPool(E, H, I, experts, DEV)
    dev_i32 = lambda a: torch.from_numpy(np.asarray(a, np.int32)).to(DEV)
    x = torch.from_numpy(x_bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    y = torch.zeros((T * k, H), dtype=torch.float32, device=DEV)
    nb = moe.moe_expert_ffn_mxfp4_workspace_size(T, k, H, I)
    st = status()
    before = moe.moe_kernel_launch_count()
    moe.moe_expert_ffn_mxfp4(pool.struct, None, dev_i32(np.arange(E)), 1, 0, E, H, I, dev_i32(counts),
                             dev_i32(offsets), dev_i32(perm), x, T, k, y, ws(nb), nb, st)
    torch.cuda.synchronize()
    assert moe.moe_kernel_launch_count() - before == 3          # gather + the two GEMM launches
    assert status_bits(st) == 0
    got = y.cpu().numpy().astype(np.float64)
    xd = gen.bf16_bits_to_f64(x_bits)
    w = {e: O.mx_expert_weights(*experts[e]) for e in range(E)}
    ref = np.stack([O.swiglu_expert(xd[t][None, :], *w[int(ids[t, 0])])[0] for t in range(T)])
    rows0, rows1 = ids[:, 0] == 0, ids[:, 0] == 1
    assert np.isnan(ref[rows0]).all() and np.isnan(got[rows0]).all()
    nan1 = np.isnan(ref[rows1])
    assert nan1[:, 5].all() and nan1.sum() == rows1.sum()
    assert np.array_equal(np.isnan(got[rows1]), nan1)
    keep = ~nan1
    assert np.abs(ref[rows1][keep]).max() > 0.05
    assert_close(got[rows1][keep], ref[rows1][keep], what="mxfp4 GEMM rows with block scales 0 and 252")
