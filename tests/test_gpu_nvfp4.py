"""GPU parity of the NVFP4 expert FFN (moe_expert_ffn_nvfp4) against the
oracle: the same SwiGLU experts on the fp64 dequantised banks (FP4 E2M1
elements, an E4M3 scale per 16 inputs, an fp32 scale per bank), through the
slot table into both pools, for one and several tokens, with distinct tensor
scales per bank, the E4M3 special values, unbound and out-of-range slots, and
the calls the decode-sized kernel does not take."""
import numpy as np
import pytest
import torch

import edge_moe_serving_gb300 as moe
from moe_inputs import gen
from moe_inputs.device import NvPool
from oracle import moe_oracle as O
from gpu_helpers import DEV, assert_close, status, status_bits, ws

pytestmark = pytest.mark.gpu

SEED = 43
BANK_TS = (2.0 ** -9, 2.0 ** -8, 3.0 * 2.0 ** -11)   # distinct tensor scales for gate, up, down


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _expert(layer, e, H, I, edit=None):
    banks = [list(b) for b in gen.nvfp4_expert(SEED, layer, e, H, I)]
    for b, ts in enumerate(BANK_TS):
        banks[b][2] = np.float32(ts)
        banks[b][1] = np.array(banks[b][1])
    if edit is not None:
        edit(e, banks)
    return [tuple(b) for b in banks]


def _run(T, k, E, H, I, n_layers, layer, cached, staged, seed, unbound=(), bad=(), active=None, edit=None):
    rng = np.random.default_rng(seed)
    experts_ids = np.arange(E) if active is None else np.asarray(active)
    ids = np.stack([np.sort(rng.choice(experts_ids, k, replace=False)) for _ in range(T)]).astype(np.int32)
    x_bits = gen.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    n_cache = max(len(cached), 1)
    slots = rng.permutation(n_cache)
    table = np.full(n_layers * E, -1, np.int32)
    base = layer * E
    weights, cache_experts, staging_experts = {}, {}, {}
    for s, e in zip(slots, cached):
        table[base + e] = s
        cache_experts[int(s)] = weights.setdefault(int(e), _expert(layer, int(e), H, I, edit))
    for e in staged:
        table[base + e] = gen.STAGING_TAG | (base + e)
        staging_experts[base + int(e)] = weights.setdefault(int(e), _expert(layer, int(e), H, I, edit))
    for e in unbound:
        table[base + e] = -1
    for e in bad:
        table[base + e] = n_cache + 3
    pool_a = NvPool(n_cache, H, I, cache_experts, DEV)
    pool_b = NvPool(n_layers * E, H, I, staging_experts, DEV) if len(staged) else None
    counts, offsets, perm, _ = O.dispatch(ids, E)
    dev_i32 = lambda a: torch.from_numpy(np.asarray(a, np.int32)).to(DEV)
    x = torch.from_numpy(x_bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    R = T * k
    y = torch.full((R, H), 7.0, dtype=torch.float32, device=DEV)
    nb = moe.moe_expert_ffn_nvfp4_workspace_size(T, k, H, I)
    st = status()
    before = moe.moe_kernel_launch_count()
    moe.moe_expert_ffn_nvfp4(pool_a.struct, pool_b.struct if pool_b else None, dev_i32(table), n_layers, layer, E,
                             H, I, dev_i32(counts), dev_i32(offsets), dev_i32(perm), x, T, k, y, ws(nb), nb, st)
    torch.cuda.synchronize()
    launches = moe.moe_kernel_launch_count() - before
    xf = gen.bf16_bits_to_f64(x_bits)
    ref = np.full((R, H), np.nan)
    dense = {}
    for i, e in enumerate(ids.reshape(-1)):
        e = int(e)
        if e in unbound or e in bad:
            continue
        if e not in dense:
            dense[e] = tuple(O.nvfp4_dequant(q, s, ts) for q, s, ts in weights[e])
        ref[i] = O.swiglu_expert(xf[i // k][None, :], *dense[e])[0]
    return y.cpu().numpy().astype(np.float64), ref, status_bits(st), ids, launches


def _check(y, ref, what):
    ok = ~np.isnan(ref[:, 0])
    assert ok.any()
    assert_close(y[ok], ref[ok], what=what)


@pytest.mark.parametrize("T,k,H,I", [(1, 6, 4096, 2048), (1, 4, 1024, 1024), (1, 5, 2048, 4096), (3, 4, 1024, 2048),
                                     (8, 8, 1024, 1024)])
def test_nvfp4_ffn_both_pools(T, k, H, I):
    """One token (the decode shape among them) and several tokens (up to the
    64 routed rows the kernel takes), experts in both pools, layer 1 of 2, a
    distinct tensor scale per bank; one launch."""
    E = 16
    experts = list(range(E))
    y, ref, st, _, launches = _run(T, k, E, H, I, 2, 1, experts[:9], experts[9:], seed=T * 1000 + H + I + k)
    assert st == 0 and launches == 1
    _check(y, ref, f"nvfp4 T={T} k={k} H={H} I={I}")


def test_nvfp4_ffn_e4m3_special_scales():
    """E4M3 scale bytes 0x00 (zero), 0x01 (the smallest subnormal, 2^-9),
    0x7E (448, the largest) and 0x7F (NaN): expert 0's gate row 3 has a NaN
    block, so its routed row is NaN everywhere; expert 1's down row 5 has
    one, so one element of the other row is NaN; zero, subnormal and largest
    scales elsewhere match the oracle."""
    def edit(e, banks):
        gate_s, up_s, down_s = banks[0][1], banks[1][1], banks[2][1]
        gate_s[:, 0] = 0x00
        up_s[:, 1] = 0x01
        gate_s[:, 2] = 0x7E
        if e == 0:
            gate_s[3, 5] = 0x7F
        else:
            down_s[5, 0] = 0x7F
    T, k, E, H, I = 1, 2, 2, 1024, 1024
    y, ref, st, ids, _ = _run(T, k, E, H, I, 1, 0, [0, 1], [], seed=5, active=np.arange(2), edit=edit)
    assert st == 0 and ids.tolist() == [[0, 1]]
    assert np.isnan(ref[0]).all() and np.isnan(y[0]).all()
    nan1 = np.isnan(ref[1])
    assert nan1.tolist() == [c == 5 for c in range(H)]
    assert np.array_equal(np.isnan(y[1]), nan1)
    assert_close(y[1][~nan1], ref[1][~nan1], what="nvfp4 row with zero, subnormal and largest E4M3 scales")


def test_nvfp4_ffn_unbound_and_bad_slot_rows_left_unwritten():
    T, k, E, H, I = 2, 3, 8, 1024, 1024
    y, ref, st, ids, _ = _run(T, k, E, H, I, 1, 0, [0, 1, 2, 3, 4], [], seed=7, active=np.arange(8),
                              unbound=(5, 7), bad=(6,))
    flat = ids.reshape(-1)
    if np.isin(flat, [5, 7]).any():
        assert st & moe.MOE_DEV_ERR_UNBOUND
    if np.isin(flat, 6).any():
        assert st & moe.MOE_DEV_ERR_BAD_SLOT
    skipped = np.isin(flat, [5, 6, 7])
    assert np.all(y[skipped] == 7.0)
    _check(y[~skipped], ref[~skipped], "nvfp4 rows of bound experts")


def test_nvfp4_ffn_rejects_calls_that_fit_neither_kernel():
    """More than 64 routed rows with rows the tensor-core GEMM does not take,
    or rows of other widths: MOE_ERR_UNSUPPORTED before any launch."""
    L = moe.lib()
    pool = NvPool(2, 1024, 1024, {}, DEV)
    i32 = torch.zeros(1024, dtype=torch.int32, device=DEV)
    x = torch.zeros((16, 1024), dtype=torch.bfloat16, device=DEV)
    y = torch.zeros((16 * 8, 1024), dtype=torch.float32, device=DEV)
    w = ws(moe.moe_expert_ffn_nvfp4_workspace_size(16, 8, 1024, 1024))
    before = moe.moe_kernel_launch_count()
    args = lambda T, k, H, I: (pool.struct, None, i32.data_ptr(), 1, 0, 8, H, I, i32.data_ptr(), i32.data_ptr(),
                               i32.data_ptr(), x.data_ptr(), T, k, y.data_ptr(), w.data_ptr(), w.numel(), None, None)
    assert L.moe_expert_ffn_nvfp4(*args(9, 8, 1040, 1040)) == moe.MOE_ERR_UNSUPPORTED    # 72 rows of 1040 inputs
    assert L.moe_expert_ffn_nvfp4(*args(1, 2, 1024, 1040)) == moe.MOE_ERR_UNSUPPORTED    # I not 1024/2048/4096
    assert moe.moe_kernel_launch_count() == before


@pytest.mark.parametrize("T,k,E,H,I", [(64, 4, 8, 1024, 512), (320, 4, 4, 512, 256), (24, 6, 12, 1024, 768)])
def test_nvfp4_ffn_tensor_core_gemm(T, k, E, H, I):
    """Calls beyond the ring kernel on the tensor-core GEMM (gather + gate/up
    + down: three launches): groups of a few rows to several 256-row chunks,
    the thin 32-row chunks of calls of at most 32 tokens, experts in both
    pools, layer 1 of 2, a distinct tensor scale per bank."""
    experts = list(range(E))
    y, ref, st, _, launches = _run(T, k, E, H, I, 2, 1, experts[: E // 2 + 1], experts[E // 2 + 1:],
                                   seed=T * 11 + E + H)
    assert launches == 3
    assert st == 0
    _check(y, ref, f"nvfp4 tensor-core GEMM T={T} k={k} E={E} H={H} I={I}")
