"""Seeded synthetic inputs for the routed MoE layer (numpy, host side).

This module is shared by the CPU oracle's tests and by the GPU harness, and
it holds none of the layer's arithmetic: it only draws numbers and rounds
them to the storage formats (bf16 bit patterns, fp32).

Recipe (every draw comes from numpy's PCG64 seeded by a SeedSequence whose
key names the tensor, the layer and the step):

* x           N(0, 1) per element, rounded to bf16.  Rows listed in the
              workload's redraw map are replaced by fresh draws (key
              ``TAG_XREDRAW, layer, step, t, r``) so that every token's k-th
              and (k+1)-th router logits differ by at least 1e-3; the map is
              written by ``moe_inputs/make_redraws.py``.
* w_router    N(0, 0.02) per element, fp32, [E, H].
* bias        'zipf': b[e] = ln p[pi(e)] with p_r proportional to r^-1.1
              (r = 1..E) and pi a seeded permutation, so that softmax routing
              is tilted by exactly the Zipf weights.  'hotset': b[e] = beta for
              e in a hot set that keeps a fixed share of its members from one
              decode step to the next.  Stored as fp32.
* experts     each bank (gate [I,H], up [I,H], down [H,I]) of each layer has
              one pool of P = 2*I*H values drawn N(0, 0.02) and rounded to bf16;
              expert e's matrix is the window of I*H consecutive pool values
              starting at a seeded offset.  Every element is marginally
              N(0, 0.02); the windows keep generation of 50 GB of expert weights
              fast on any host while every expert still occupies its own bytes.
* MXFP4       block-scaled FP4 expert banks (OCP MX encoding): code bytes
              uniform over 0..255, so every E2M1 code of every element is
              equally likely (RMS magnitude 2.93), and E8M0 block scales drawn
              uniformly from 119..120 (2^-8, 2^-7): weights with standard
              deviation 0.018, near the bf16 experts' N(0, 0.02).  Key ``TAG_MX, seed,
              layer, expert, bank``.
* NVFP4       FP4 E2M1 code bytes uniform over 0..255, E4M3 block scales (one
              per 16 inputs) uniform over the bytes 0x40..0x47 (2.0 .. 3.75)
              and a tensor scale of 2^-9 per bank: weight standard deviation
              about 0.017.  Key ``TAG_NV, seed, layer, expert, bank``.
* cache       the initial residency: a seeded random subset of the
              (layer, expert) pairs in cache slots 0..S-1, all stamps 0.
"""
import json
import os
from functools import lru_cache

import numpy as np

from .configs import LayerConfig

TAG_X, TAG_XREDRAW, TAG_WR, TAG_BIAS, TAG_HOT, TAG_POOL, TAG_OFF, TAG_CACHE, TAG_MX, TAG_NV = range(1, 11)
BANKS = ("gate", "up", "down")
STAGING_TAG = 1 << 30          # slot-table tag of the staging pool (pool B)
REDRAW_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "redraws")


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(v) for v in key])))


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); uint16 bits."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = (b.astype(np.uint64) + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(bits) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------- redraw maps
@lru_cache(maxsize=None)
def _load_redraws(name: str):
    path = os.path.join(REDRAW_DIR, f"{name}.json")
    if not os.path.exists(path):
        return {}, 0
    with open(path) as f:
        doc = json.load(f)
    out = {}
    for layer, step, t, r in doc["entries"]:
        out.setdefault((layer, step), {})[t] = r
    return out, int(doc.get("steps_covered", 0))


def redraws_for(cfg: LayerConfig, layer: int, step: int) -> dict:
    """Rows of x(layer, step) that are replaced, as {token: draw index}."""
    table, _ = _load_redraws(cfg.name)
    return dict(table.get((layer, step), {}))


def steps_covered(cfg: LayerConfig) -> int:
    return _load_redraws(cfg.name)[1]


# ---------------------------------------------------------------- tensors
def layer_seed(cfg: LayerConfig, layer: int) -> int:
    return cfg.seed + layer


def x_row_redraw(cfg: LayerConfig, layer: int, step: int, t: int, r: int) -> np.ndarray:
    g = _rng(layer_seed(cfg, layer), TAG_XREDRAW, step, t, r)
    return f32_to_bf16_bits(g.standard_normal(cfg.H).astype(np.float32))


def x_bits(cfg: LayerConfig, layer: int = 0, step: int = 0, redraws=None, tokens=None) -> np.ndarray:
    """bf16 bits [T, H] of the layer input at (layer, step).

    ``redraws`` defaults to the stored map; pass ``{}`` for the raw draw."""
    g = _rng(layer_seed(cfg, layer), TAG_X, step)
    x = f32_to_bf16_bits(g.standard_normal((cfg.T, cfg.H), dtype=np.float32))
    if redraws is None:
        redraws = redraws_for(cfg, layer, step)
    for t, r in redraws.items():
        x[t] = x_row_redraw(cfg, layer, step, t, r)
    return x


def w_router(cfg: LayerConfig, layer: int = 0) -> np.ndarray:
    g = _rng(layer_seed(cfg, layer), TAG_WR)
    return (g.standard_normal((cfg.E, cfg.H)) * 0.02).astype(np.float32)


def hot_sets(cfg: LayerConfig, layer: int, n_steps: int):
    """Hot expert sets for steps 0..n_steps-1 (bias kind 'hotset')."""
    sets = []
    prev = None
    keep_n = int(round(cfg.hot_keep * cfg.hot_size))
    for s in range(n_steps):
        g = _rng(layer_seed(cfg, layer), TAG_HOT, s)
        if prev is None:
            cur = np.sort(g.choice(cfg.E, cfg.hot_size, replace=False))
        else:
            kept = g.choice(prev, keep_n, replace=False)
            rest = np.setdiff1d(np.arange(cfg.E), prev)
            fresh = g.choice(rest, cfg.hot_size - keep_n, replace=False)
            cur = np.sort(np.concatenate([kept, fresh]))
        sets.append(cur)
        prev = cur
    return sets


def bias(cfg: LayerConfig, layer: int = 0, step: int = 0):
    """fp32 expert bias [E] added to the router logits, or None."""
    if cfg.bias == "none":
        return None
    if cfg.bias == "zipf":
        g = _rng(layer_seed(cfg, layer), TAG_BIAS)
        perm = g.permutation(cfg.E)
        p = np.arange(1, cfg.E + 1, dtype=np.float64) ** (-cfg.zipf_s)
        p /= p.sum()
        return np.log(p[perm]).astype(np.float32)
    if cfg.bias == "hotset":
        b = np.zeros(cfg.E, np.float32)
        b[hot_sets(cfg, layer, step + 1)[step]] = cfg.hot_beta
        return b
    raise ValueError(cfg.bias)


def bank_shape(cfg: LayerConfig, bank: int):
    return (cfg.I, cfg.H) if bank < 2 else (cfg.H, cfg.I)


def pool_len(cfg: LayerConfig) -> int:
    return 2 * cfg.I * cfg.H


@lru_cache(maxsize=16)
def bank_pool(cfg: LayerConfig, layer: int, bank: int) -> np.ndarray:
    g = _rng(layer_seed(cfg, layer), TAG_POOL, bank)
    vals = (g.standard_normal(pool_len(cfg), dtype=np.float32) * np.float32(0.02))
    out = f32_to_bf16_bits(vals)
    out.setflags(write=False)
    return out


@lru_cache(maxsize=64)
def bank_offsets(cfg: LayerConfig, layer: int, bank: int) -> np.ndarray:
    g = _rng(layer_seed(cfg, layer), TAG_OFF, bank)
    n = cfg.I * cfg.H
    out = g.integers(0, pool_len(cfg) - n + 1, size=cfg.E, dtype=np.int64)
    out.setflags(write=False)
    return out


def expert_bits(cfg: LayerConfig, layer: int, bank: int, e: int) -> np.ndarray:
    """bf16 bits of one bank matrix of logical expert (layer, e)."""
    off = int(bank_offsets(cfg, layer, bank)[e])
    return bank_pool(cfg, layer, bank)[off: off + cfg.I * cfg.H].reshape(bank_shape(cfg, bank))


def expert_f64(cfg: LayerConfig, layer: int, e: int):
    """(W_gate [I,H], W_up [I,H], W_down [H,I]) of expert (layer, e) as fp64."""
    return tuple(bf16_bits_to_f64(expert_bits(cfg, layer, b, e)) for b in range(3))


def initial_cache(cfg: LayerConfig):
    """Initial residency state: slot table [L*E], owner [S], stamp [S], clock.

    Slot-table entries: ``slot`` for the cache pool, ``STAGING_TAG | (l*E+e)``
    for the staging pool, -1 for unbound."""
    LE = cfg.n_layers * cfg.E
    if cfg.cache_slots is None:
        table = np.arange(LE, dtype=np.int32)
        owner = np.arange(LE, dtype=np.int32)
    else:
        g = _rng(cfg.seed, TAG_CACHE)
        pairs = g.choice(LE, cfg.cache_slots, replace=False).astype(np.int32)
        table = (STAGING_TAG | np.arange(LE, dtype=np.int64)).astype(np.int32)
        table[pairs] = np.arange(cfg.cache_slots, dtype=np.int32)
        owner = pairs.copy()
    stamp = np.zeros(owner.size, np.uint32)
    return {"table": table, "owner": owner, "stamp": stamp, "clock": 0}


# ---------------------------------------------------------------- MXFP4 experts
MX_SCALE_EXPONENTS = (119, 120)   # inclusive range of the drawn E8M0 scale bytes


def mx_bank(seed: int, layer: int, e: int, bank: int, rows: int, K: int):
    """(codes uint8 [rows, K/2], scales uint8 [rows, K/32]) of one MXFP4 bank."""
    g = _rng(TAG_MX, seed, layer, e, bank)
    codes = np.frombuffer(g.bytes(rows * (K // 2)), dtype=np.uint8).reshape(rows, K // 2)
    lo, hi = MX_SCALE_EXPONENTS
    scales = g.integers(lo, hi + 1, size=(rows, K // 32), dtype=np.uint8)
    return codes, scales


def mx_expert(seed: int, layer: int, e: int, H: int, I: int):
    """(gate_q, gate_s, up_q, up_s, down_q, down_s) of MXFP4 expert (layer, e):
    gate and up rows [I] of H inputs, down rows [H] of I inputs."""
    gq, gs = mx_bank(seed, layer, e, 0, I, H)
    uq, us = mx_bank(seed, layer, e, 1, I, H)
    dq, ds = mx_bank(seed, layer, e, 2, H, I)
    return gq, gs, uq, us, dq, ds


# ---------------------------------------------------------------- NVFP4 experts
NV_SCALE_BYTES = (0x40, 0x47)     # inclusive range of the drawn E4M3 block-scale bytes
NV_TENSOR_SCALE = 2.0 ** -9


def nvfp4_bank(seed: int, layer: int, e: int, bank: int, rows: int, K: int):
    """(codes uint8 [rows, K/2], E4M3 scales uint8 [rows, K/16], fp32 tensor scale)."""
    g = _rng(TAG_NV, seed, layer, e, bank)
    codes = np.frombuffer(g.bytes(rows * (K // 2)), dtype=np.uint8).reshape(rows, K // 2)
    lo, hi = NV_SCALE_BYTES
    scales = g.integers(lo, hi + 1, size=(rows, K // 16), dtype=np.uint8)
    return codes, scales, np.float32(NV_TENSOR_SCALE)



def nvfp4_expert(seed: int, layer: int, e: int, H: int, I: int):
    """((gate_q, gate_s, gate_ts), (up_q, up_s, up_ts), (down_q, down_s, down_ts))
    of NVFP4 expert (layer, e): gate and up rows [I] of H inputs, down rows [H]
    of I inputs."""
    return (nvfp4_bank(seed, layer, e, 0, I, H), nvfp4_bank(seed, layer, e, 1, I, H),
            nvfp4_bank(seed, layer, e, 2, H, I))
