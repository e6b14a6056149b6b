"""Pins of the CPU fp64 oracle against what the pages and mathematics fix.

None of these tests need a GPU.  Each pin is chosen so that a plausible slip
in the oracle (a dropped term, a wrong sign or index, a transposed operand,
a wrong tie rule) fails at least one of them.
"""
import collections
import os

import numpy as np
import pytest
import scipy.special

from moe_inputs import CONFIGS, gen
from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out.append(line.split())
    return out


def _rand_layer(rng, T, H, E, k, I, bias=True):
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) * 0.3
    b = rng.standard_normal(E) * 0.5 if bias else None
    W = [(rng.standard_normal((I, H)) * 0.2, rng.standard_normal((I, H)) * 0.2,
          rng.standard_normal((H, I)) * 0.2) for _ in range(E)]
    return x, wr, b, W


# ------------------------------------------------------------------ q* rule
def test_qrule_printed_values():
    """Every count the write-up prints or asserts (shipped rule, no floor)."""
    rows = _rows("qrule_writeup.txt")
    assert len(rows) >= 17
    for m, bp, bh, q, *_ in rows:
        fq = min(O.Q16, round(float(bp) / float(bh) * O.Q16))
        assert O.fill_count(int(m), fq, min_fill=0) == int(q), (m, bp, bh)


def test_qrule_table1_ratios():
    for name, bp, bh, ratio in _rows("table1_bandwidths.txt"):
        assert round(float(bh) / float(bp), 2) == float(ratio), name


def test_qrule_is_integer_argmin_and_tracks_eq4():
    """q minimises the Eq. 3 makespan over all integers 0..m and |q - phi m| <= 1."""
    for phi in (0.1, 0.2484, 0.3972, 0.415, 0.5, 0.6817, 0.9108, 1.0, 1 / 3, 0.999):
        fq = O.phi_to_q16(phi)
        for m in range(0, 97):
            q = O.fill_count(m, fq, min_fill=0)
            assert 0 <= q <= m
            cost = [max(f * (O.Q16 - fq), (m - f) * fq) for f in range(m + 1)]
            assert cost[q] == min(cost), (phi, m, q)
            assert abs(q - fq / O.Q16 * m) <= 1.0
            # ties resolve to the smaller count
            assert q == min(f for f in range(m + 1) if cost[f] == min(cost)) or q == (m * fq) // O.Q16


def test_qrule_endpoints_and_floor():
    for m in range(0, 40):
        assert O.fill_count(m, O.Q16, 0) == m          # B_P >= B_H: pure on-demand fill (Eq. 4)
        assert O.fill_count(m, 0, 0) == 0              # B_P = 0: nothing crosses the link
        assert O.fill_count(m, 0, 1) == 0              # the floor never invents a link
    # the paper's "at least one fill" floor lifts the laptop's q = 0 cases
    fq = O.phi_to_q16(11.8 / 47.5)
    for m in (1, 2, 3):
        assert O.fill_count(m, fq, 0) == 0
        assert O.fill_count(m, fq, 1) == 1
    assert O.fill_count(0, fq, 1) == 0


def test_phi_to_q16_is_the_nearest_q16_integer():
    """phi in Q16 is the integer nearest to 65536 phi (exact rational
    arithmetic on the double's value), ties to even, clamped to [0, 65536]."""
    from fractions import Fraction

    def nearest(phi):
        v = Fraction(phi) * O.Q16
        lo = v.numerator // v.denominator
        rem = v - lo
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
            lo += 1
        return min(O.Q16, max(0, lo))

    rng = np.random.default_rng(9)
    grid = [2 / 3, 1 / 3, 0.415, 25.1 / 63.2, 11.8 / 47.5, 1.5 / O.Q16, 2.5 / O.Q16, 0.5 / O.Q16,
            65535.5 / O.Q16, 1.0, 1.2, 0.0, -0.25] + rng.random(500).tolist()
    for phi in grid:
        assert O.phi_to_q16(phi) == nearest(phi), phi
    assert O.phi_to_q16(2 / 3) == 43691                # 43690.67 rounds up
    assert O.phi_to_q16(1.5 / O.Q16) == 2 and O.phi_to_q16(2.5 / O.Q16) == 2   # ties to even


def test_qrule_balance_equation():
    """Eq. 4: q/(m-q) ~ B_P/(B_H-B_P); the continuous optimum q* = m B_P/B_H
    equalises T_fill = qS/B_P and T_cpu = (m-q)S/(B_H-B_P)."""
    for _, bp, bh, _r in _rows("table1_bandwidths.txt"):
        bp, bh = float(bp), float(bh)
        for m in (4, 12, 50):
            qs = m * bp / bh
            assert np.isclose(qs / bp, (m - qs) / (bh - bp))
            q = O.fill_count(m, O.phi_to_q16(bp / bh), 0)
            assert abs(q - qs) <= 1.0


# ------------------------------------------------------------------ router / top-k
def test_topk_against_library_sort():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((200, 37))
    logits[0, :] = 0.0                          # all tied: lowest ids win
    logits[1, [3, 9]] = 5.0                     # a tie inside the selection
    for k in (1, 2, 5, 37):
        ids, w = O.select_topk(logits, k)
        for t in range(logits.shape[0]):
            order = np.argsort(-logits[t], kind="stable")   # stable: ties by lower id
            assert list(ids[t]) == sorted(order[:k].tolist())
            sm = scipy.special.softmax(logits[t])
            assert np.allclose(w[t], sm[ids[t]] / sm[ids[t]].sum(), rtol=1e-13)
        assert np.allclose(w.sum(1), 1.0, rtol=1e-14)
    ids, _ = O.select_topk(logits, 3)
    assert list(ids[0]) == [0, 1, 2]


def test_router_logits_orientation_and_bias():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 7))
    wr = rng.standard_normal((3, 7))
    b = np.array([1.0, -2.0, 0.5])
    ref = np.einsum("th,eh->te", x, wr) + b
    assert np.allclose(O.router_logits(x, wr, b), ref, rtol=1e-14)
    # a unit x row selects the matching router column
    e1 = np.zeros((1, 7)); e1[0, 4] = 1.0
    assert np.allclose(O.router_logits(e1, wr, None)[0], wr[:, 4])


def test_topk_gap():
    logits = np.array([[3.0, 1.0, 2.0, 0.5], [1.0, 1.0, 1.0, 0.0]])
    assert np.allclose(O.topk_gap(logits, 2), [1.0, 0.0])


# ------------------------------------------------------------------ dispatch
def test_dispatch_against_stable_argsort_and_invariants():
    rng = np.random.default_rng(3)
    for T, k, E in ((1, 6, 256), (64, 2, 8), (37, 5, 13), (300, 8, 128)):
        ids = np.stack([np.sort(rng.choice(E, k, replace=False)) for _ in range(T)])
        counts, offsets, perm, inv = O.dispatch(ids, E)
        flat = ids.reshape(-1)
        assert counts.sum() == T * k and offsets[0] == 0 and offsets[-1] == T * k
        assert np.array_equal(np.diff(offsets), counts)
        assert np.array_equal(perm, np.argsort(flat, kind="stable"))
        assert np.array_equal(perm[inv], np.arange(T * k))
        assert np.array_equal(np.sort(perm), np.arange(T * k))
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


def test_dispatch_empty():
    counts, offsets, perm, inv = O.dispatch(np.zeros((0, 2), np.int32), 4)
    assert counts.sum() == 0 and list(offsets) == [0] * 5 and perm.size == 0


# ------------------------------------------------------------------ expert FFN and layer
def test_silu_matches_library():
    z = np.linspace(-40, 40, 2001)
    assert np.allclose(O.silu(z), z * scipy.special.expit(z), rtol=1e-14, atol=1e-300)
    assert O.silu(np.array([-1000.0]))[0] == 0.0


def test_single_expert_is_dense_swiglu():
    """E = 1, k = 1: weight 1, the layer is one dense SwiGLU FFN."""
    rng = np.random.default_rng(11)
    x, wr, b, W = _rand_layer(rng, 9, 12, 1, 1, 20)
    wg, wu, wd = W[0]
    g = x @ wg.T
    dense = (g * scipy.special.expit(g) * (x @ wu.T)) @ wd.T
    res = O.layer_forward(x, wr, b, 1, lambda e: W[e])
    assert np.allclose(res["w"], 1.0)
    assert np.allclose(res["out"], dense, rtol=1e-12, atol=1e-12)


def test_k_equals_E_is_softmax_mixture():
    rng = np.random.default_rng(12)
    E = 5
    x, wr, b, W = _rand_layer(rng, 7, 10, E, E, 6)
    res = O.layer_forward(x, wr, b, E, lambda e: W[e])
    p = scipy.special.softmax(x @ wr.T + b, axis=1)
    ref = np.zeros_like(x)
    for e in range(E):
        g = x @ W[e][0].T
        ref += p[:, e:e + 1] * ((g * scipy.special.expit(g) * (x @ W[e][1].T)) @ W[e][2].T)
    assert np.allclose(res["out"], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shape", [(1, 8, 4, 1, 6), (16, 8, 8, 2, 12), (11, 6, 7, 3, 5), (4, 10, 3, 3, 4)])
def test_bruteforce_matches_dispatch_path(shape):
    T, H, E, k, I = shape
    rng = np.random.default_rng(sum(shape))
    x, wr, b, W = _rand_layer(rng, T, H, E, k, I)
    res = O.layer_forward(x, wr, b, k, lambda e: W[e])
    brute = O.layer_forward_bruteforce(x, wr, b, k, lambda e: W[e])
    assert np.allclose(res["out"], brute, rtol=1e-12, atol=1e-12)


def test_bruteforce_matches_on_tiny_workload():
    cfg = CONFIGS["tiny"]
    x = gen.bf16_bits_to_f64(gen.x_bits(cfg))[:16]
    wr = gen.w_router(cfg)
    W = {e: gen.expert_f64(cfg, 0, e) for e in range(cfg.E)}
    res = O.layer_forward(x, wr, None, cfg.k, W.__getitem__)
    brute = O.layer_forward_bruteforce(x, wr, None, cfg.k, W.__getitem__)
    assert np.allclose(res["out"], brute, rtol=1e-12, atol=1e-12)


def test_linear_in_w_down():
    rng = np.random.default_rng(5)
    x, wr, b, W = _rand_layer(rng, 12, 8, 6, 2, 10)
    W2 = [(g, u, rng.standard_normal(d.shape)) for g, u, d in W]
    f = lambda Ws: O.layer_forward(x, wr, b, 2, lambda e: Ws[e])["out"]
    o1, o2 = f(W), f(W2)
    o12 = f([(g, u, d1 + 2.5 * d2) for (g, u, d1), (_, _, d2) in zip(W, W2)])
    assert np.allclose(o12, o1 + 2.5 * o2, rtol=1e-12, atol=1e-12)


def test_split_merge_is_exact():
    """[P] 3.2: the F and C partial sums merge into the exact layer output."""
    rng = np.random.default_rng(21)
    x, wr, b, W = _rand_layer(rng, 24, 8, 10, 3, 6)
    full = O.layer_forward(x, wr, b, 3, lambda e: W[e])
    active = np.nonzero(full["counts"])[0]
    for _ in range(120):
        F = [int(e) for e in active if rng.random() < 0.5]
        merged, pF, pC = O.layer_forward_split(x, wr, b, 3, lambda e: W[e], F)
        assert np.array_equal(merged, full["out"])           # bitwise: same rows, same order
        assert np.allclose(pF + pC, full["out"], rtol=1e-13, atol=1e-13)
    merged, pF, pC = O.layer_forward_split(x, wr, b, 3, lambda e: W[e], [])
    assert np.array_equal(pF, np.zeros_like(pF)) and np.array_equal(merged, full["out"])


def test_combine_weights_and_order():
    y = np.arange(12, dtype=np.float64).reshape(4, 3)      # 4 dispatch rows, H = 3
    inv = np.array([2, 0, 3, 1])                           # T = 2, k = 2
    w = np.array([[0.25, 0.75], [1.0, 0.0]])
    out = O.combine(y, inv, w, 2)
    assert np.allclose(out[0], 0.25 * y[2] + 0.75 * y[0])
    assert np.allclose(out[1], y[3])


# ------------------------------------------------------------------ residency / bind
def test_splitmix64_reference_sequence():
    """The published SplitMix64 stream for seed 0 starts e220a8397b1dcdaf,
    6e789e6aa1b965f4, 06c45d188009454f."""
    golden = 0x9E3779B97F4A7C15
    outs = [O.splitmix64((i * golden) & O.MASK64) for i in range(3)]
    assert outs == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def _state(n_slots, E, L=1, resident=()):
    table = np.array([O.STAGING_TAG | i for i in range(L * E)], np.int64)
    owner = np.full(n_slots, -1, np.int64)
    for v, pair in enumerate(resident):
        table[pair] = v
        owner[v] = pair
    return {"table": table, "owner": owner, "stamp": np.zeros(n_slots, np.int64), "clock": 0}


def test_bind_figure2_scenario():
    """Figure 2: 12 routed, 8 hits, m = 4 -> 1 fill and 3 in place."""
    g = {r[0]: int(r[1]) for r in _rows("figure2_decode.txt")}
    E = 64
    routed = np.arange(0, 24, 2).reshape(2, 6)             # 12 distinct experts
    hits = routed.reshape(-1)[:8]
    st = _state(16, E, resident=[int(e) for e in hits] + [40, 41, 42])
    for bp, bh in ((25.1, 63.2), (11.8, 47.5), (51.5, 178.0)):
        new, res = O.bind(st, 0, routed, E, O.phi_to_q16(bp / bh), min_fill=1)
        s = res["stats"]
        assert s["n_unique"] == g["routed"] and s["n_hit"] == g["hits"] and s["n_miss"] == g["misses"]
        assert s["n_fill"] == g["fills"] and s["n_staged"] == g["in_place"]
        assert res["F"] == [16] and res["C"] == [18, 20, 22]
        # the fill takes the least (stamp, slot) slot not hit this call: slot 8,
        # whose pair 40 goes back to the staging pool; the hits keep their slots
        assert res["fills"] == [(16, 8)]
        assert new["table"][16] == 8 and new["owner"][8] == 16 and new["stamp"][8] == 1
        assert new["table"][40] == O.STAGING_TAG | 40
        for e in (18, 20, 22):
            assert new["table"][e] == O.STAGING_TAG | e
        for v, e in enumerate(hits):
            assert new["table"][e] == v and new["stamp"][v] == 1


def test_bind_evicts_least_recent_and_rebinds_victim():
    E = 8
    st = _state(3, E, resident=[0, 1, 2])
    st, _ = O.bind(st, 0, np.array([[1]]), E, O.Q16)       # clock 1: 1 refreshed
    st, _ = O.bind(st, 0, np.array([[2]]), E, O.Q16)       # clock 2: 2 refreshed
    st, res = O.bind(st, 0, np.array([[5, 6]]), E, O.Q16)  # two misses, q = 2
    # victims in (stamp, slot) order: slot 0 (stamp 0), slot 1 (stamp 1)
    assert res["fills"] == [(5, 0), (6, 1)]
    assert st["table"][0] == O.STAGING_TAG | 0 and st["table"][1] == O.STAGING_TAG | 1
    assert list(st["owner"]) == [5, 6, 2]


def test_bind_overflow_when_all_slots_hit():
    E = 8
    st = _state(2, E, resident=[0, 1])
    st, res = O.bind(st, 0, np.array([[0, 1, 3, 4]]), E, O.Q16)
    s = res["stats"]
    assert s["q"] == 2 and s["n_fill"] == 0 and s["n_overflow"] == 2 and res["C"] == [3, 4]


def test_bind_random_policy_is_seeded_subset():
    E = 32
    st = _state(8, E)
    ids = np.arange(16).reshape(2, 8)
    picks = set()
    for seed in range(20):
        _, res = O.bind(st, 0, ids, E, O.Q16 // 4, policy=O.FILL_RANDOM, seed=seed)
        assert len(res["F"]) == 4 and set(res["F"]) <= set(range(16))
        _, res2 = O.bind(st, 0, ids, E, O.Q16 // 4, policy=O.FILL_RANDOM, seed=seed)
        assert res2["F"] == res["F"]
        picks.add(tuple(res["F"]))
    assert len(picks) > 10


def _lru_recency_sim(cfg, traces):
    """Independent model: an ordered recency list instead of stamps.  The
    cache starts full; pairs touched in one call move to the most-recent end
    in slot order; each fill takes the least recent pair not touched yet."""
    st0 = gen.initial_cache(cfg)
    assert np.all(st0["owner"] >= 0)
    resident = collections.OrderedDict((int(p), v) for v, p in enumerate(st0["owner"]))
    outs = []
    for layer, ids in traces:
        base = layer * cfg.E
        U = sorted(set(ids.reshape(-1).tolist()))
        hits = [e for e in U if base + e in resident]
        misses = [e for e in U if base + e not in resident]
        touched = {base + e: resident[base + e] for e in hits}
        q = O.fill_count(len(misses), cfg.phi_q16, cfg.min_fill)
        fills = []
        for e in misses[:q]:
            older = [p for p in resident if p not in touched]
            if not older:
                break
            v = resident.pop(older[0])
            fills.append((base + e, v))
            touched[base + e] = v
        for p in touched:
            resident.pop(p, None)
        for p, v in sorted(touched.items(), key=lambda kv: kv[1]):
            resident[p] = v
        outs.append(fills)
    return outs, resident


def test_bind_matches_recency_list_model_on_decode_trace():
    cfg = CONFIGS["decode"]
    wr = gen.w_router(cfg)
    b = gen.bias(cfg)
    traces = []
    for s in range(cfg.steps):
        x = gen.bf16_bits_to_f64(gen.x_bits(cfg, 0, s))
        ids, _ = O.select_topk(O.router_logits(x, wr, b), cfg.k)
        traces.append((0, ids))
    st = gen.initial_cache(cfg)
    fills_stamp = []
    for layer, ids in traces:
        st, res = O.bind(st, layer, ids, cfg.E, cfg.phi_q16, cfg.min_fill, cfg.fill_policy)
        fills_stamp.append(res["fills"])
    fills_list, resident = _lru_recency_sim(cfg, traces)
    assert fills_stamp == fills_list
    assert sum(len(f) for f in fills_stamp) > 5
    for p, v in resident.items():
        assert st["table"][p] == v and st["owner"][v] == p


def test_bind_dedup_count_closed_form():
    """Uniform routing: mean unique experts = E (1 - (1 - k/E)^B) (the write-up's
    batch-dedup section)."""
    rng = np.random.default_rng(0)
    E, k, B = 256, 6, 4
    st = _state(4, E)
    n = []
    for _ in range(3000):
        ids = np.stack([np.sort(rng.choice(E, k, replace=False)) for _ in range(B)])
        n.append(O.bind(st, 0, ids, E, 0)[1]["stats"]["n_unique"])
    assert np.isclose(np.mean(n), E * (1 - (1 - k / E) ** B), rtol=5e-3)


# ------------------------------------------------------------------ generated inputs
@pytest.mark.parametrize("name", ["tiny", "decode", "batched_decode"])
def test_redraw_maps_give_gap(name):
    cfg = CONFIGS[name]
    for layer in range(cfg.n_layers):
        wr = gen.w_router(cfg, layer)
        for step in range(gen.steps_covered(cfg)):
            x = gen.bf16_bits_to_f64(gen.x_bits(cfg, layer, step))
            gaps = O.topk_gap(O.router_logits(x, wr, gen.bias(cfg, layer, step)), cfg.k)
            assert gaps.min() >= 1e-3, (name, layer, step)


def test_batched_decode_locality():
    """Realised reuse of the active expert set between decode steps is 0.70 +- 0.05."""
    cfg = CONFIGS["batched_decode"]
    wr = gen.w_router(cfg)
    prev, reuse = None, []
    for s in range(cfg.steps):
        x = gen.bf16_bits_to_f64(gen.x_bits(cfg, 0, s))
        ids, _ = O.select_topk(O.router_logits(x, wr, gen.bias(cfg, 0, s)), cfg.k)
        A = set(ids.reshape(-1).tolist())
        if prev is not None:
            reuse.append(len(A & prev) / len(A))
        prev = A
    assert abs(np.mean(reuse) - 0.70) <= 0.05


def test_zipf_bias_tilts_softmax_by_zipf_weights():
    cfg = CONFIGS["decode"]
    p = np.exp(gen.bias(cfg).astype(np.float64))
    assert np.isclose(p.sum(), 1.0, rtol=1e-6)
    ranks = np.sort(p)[::-1]
    r = np.arange(1, cfg.E + 1)
    ref = r ** -1.1 / (r ** -1.1).sum()
    assert np.allclose(ranks, ref, rtol=1e-6)


def test_bf16_rounding():
    vals = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-3], np.float32)
    bits = gen.f32_to_bf16_bits(vals)
    back = gen.bf16_bits_to_f32(bits)
    assert back[0] == 1.0 and back[1] == 1.0          # halfway rounds to even (down)
    assert back[2] == np.float32(1.015625)            # halfway rounds to even (up)
    assert back[3] == -2.5
    assert abs(back[4] - 3.0e-3) <= 3.0e-3 * 2 ** -8


# ------------------------------------------------------------------ MXFP4 experts
def _e2m1_table():
    return {int(c, 16): float(v) for c, _bits, v in _rows("e2m1_ocp_mx.txt")}


def test_e2m1_matches_the_mx_spec_table():
    table = _e2m1_table()
    assert sorted(table) == list(range(16))
    for code, v in table.items():
        got = O.e2m1_value(code)
        assert got == v and np.signbit(got) == np.signbit(v), code
    mags = [O.e2m1_value(c) for c in range(8)]
    assert mags == sorted(mags) and max(mags) == 6.0


def test_e8m0_is_a_power_of_two_with_bias_127():
    for s in (0, 1, 100, 126, 127, 128, 200, 254):
        assert O.e8m0_value(s) == np.ldexp(1.0, s - 127), s
    assert np.isnan(O.e8m0_value(255))


def _mx_encode_exact(dense):
    """Brute-force MX encoder for weights that are exactly representable:
    per block, the scale exponent is found by search and each element's code
    by search over the spec table (values from the golden file)."""
    table = _e2m1_table()
    rows, K = dense.shape
    codes = np.zeros((rows, K // 2), np.uint8)
    scales = np.zeros((rows, K // 32), np.uint8)
    for r in range(rows):
        for b in range(K // 32):
            blk = dense[r, 32 * b:32 * b + 32]
            for s in range(255):
                sc = np.ldexp(1.0, s - 127)
                found = []
                for v in blk:
                    hit = [c for c, tv in table.items() if tv * sc == v and np.signbit(tv) == np.signbit(v)]
                    if not hit:
                        break
                    found.append(hit[0])
                if len(found) == 32:
                    scales[r, b] = s
                    for i, c in enumerate(found):
                        col = 32 * b + i
                        codes[r, col // 2] |= np.uint8(c << (4 * (col % 2)))
                    break
            else:
                raise AssertionError("not representable")
    return codes, scales


def test_mx_dequant_round_trips_exactly_representable_weights():
    """Rows of per-block scaled E2M1 values survive encode -> dequantise
    exactly; each block has its own scale (a block holds the value 6, so its
    scale is unique), so a wrong nibble order, block index or scale mapping
    moves a value."""
    rng = np.random.default_rng(17)
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    rows, K = 5, 96
    dense = np.zeros((rows, K))
    for r in range(rows):
        for b in range(K // 32):
            v = rng.choice(mags, 32) * rng.choice([-1.0, 1.0], 32)
            v[rng.integers(32)] = 6.0
            dense[r, 32 * b:32 * b + 32] = v * np.ldexp(1.0, int(rng.integers(-12, 3)))
    codes, scales = _mx_encode_exact(dense)
    assert np.array_equal(O.mx_dequant(codes, scales), dense)


def test_mx_dequant_layout_by_hand():
    """One row, K = 64: byte 0 = 0x71 holds element 0 (code 1 = 0.5) low and
    element 1 (code 7 = 6.0) high; the second block's scale 2^1 doubles it."""
    codes = np.zeros((1, 32), np.uint8)
    codes[0, 0] = 0x71
    codes[0, 16] = 0xA3          # element 32: code 3 = 1.5, element 33: code A = -1.0
    scales = np.array([[127, 128]], np.uint8)
    W = O.mx_dequant(codes, scales)
    assert W[0, 0] == 0.5 and W[0, 1] == 6.0 and W[0, 32] == 3.0 and W[0, 33] == -2.0
    assert np.count_nonzero(W) == 4


def test_e8m0_equals_the_library_decoder_for_every_byte():
    import torch
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    ours = np.array([O.e8m0_value(s) for s in range(256)])
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    assert np.array_equal(lib[~np.isnan(lib)], ours[~np.isnan(ours)])


# ------------------------------------------------------------------ NVFP4 experts
def test_e4m3_matches_the_ofp8_spec_values():
    for b, _bits, v in _rows("e4m3_ocp_fp8.txt"):
        got = O.e4m3_value(int(b, 16))
        if v == "nan":
            assert np.isnan(got), b
        else:
            assert got == float(v), b


def test_e4m3_equals_the_library_decoder_for_every_byte():
    import torch
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    ours = np.array([O.e4m3_value(b) for b in range(256)])
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    ok = ~np.isnan(lib)
    assert np.array_equal(lib[ok], ours[ok]) and np.array_equal(np.signbit(lib[ok]), np.signbit(ours[ok]))


def test_nvfp4_dequant_layout_by_hand():
    """K = 32: two blocks of 16.  Byte 0 = 0x71: element 0 = 0.5, element 1 =
    6.0 under scale 0x38 (1.0); byte 8 = 0xA3: element 16 = 1.5, element 17 =
    -1.0 under scale 0x40 (2.0); tensor scale 0.25."""
    codes = np.zeros((1, 16), np.uint8)
    codes[0, 0] = 0x71
    codes[0, 8] = 0xA3
    scales = np.array([[0x38, 0x40]], np.uint8)
    W = O.nvfp4_dequant(codes, scales, 0.25)
    assert W[0, 0] == 0.125 and W[0, 1] == 1.5 and W[0, 16] == 0.75 and W[0, 17] == -0.5
    assert np.count_nonzero(W) == 4


def test_nvfp4_dequant_round_trips_exactly_representable_weights():
    """Per 16-input block: E2M1 values times one E4M3 scale (drawn from exact
    E4M3 values), times one tensor scale; a brute-force encoder over the spec
    tables recovers bytes that dequantise back exactly."""
    import torch
    e2m1 = _e2m1_table()
    e4m3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    rng = np.random.default_rng(23)
    rows, K, ts = 4, 64, np.float32(0.0078125 * 3)
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    scale_bytes = rng.integers(0x30, 0x50, size=(rows, K // 16))
    dense = np.zeros((rows, K))
    for r in range(rows):
        for b in range(K // 16):
            v = rng.choice(mags, 16) * rng.choice([-1.0, 1.0], 16)
            v[rng.integers(16)] = 6.0
            dense[r, 16 * b:16 * b + 16] = v * e4m3[scale_bytes[r, b]] * float(ts)
    codes = np.zeros((rows, K // 2), np.uint8)
    for r in range(rows):
        for i in range(K):
            sc = e4m3[scale_bytes[r, i // 16]] * float(ts)
            hit = [c for c, tv in e2m1.items() if tv * sc == dense[r, i] and np.signbit(tv) == np.signbit(dense[r, i])]
            codes[r, i // 2] |= np.uint8(hit[0] << (4 * (i % 2)))
    assert np.array_equal(O.nvfp4_dequant(codes, scale_bytes.astype(np.uint8), ts), dense)
