"""The oracle's pins are sensitive: each plausible slip, planted in a copy of
one oracle function on the CPU, makes at least one pin of test_oracle.py fail.

A mutant is the function's own source with one or two substrings replaced
(each must occur exactly once, so a mutant that no longer applies fails
loudly instead of passing vacuously), compiled in the oracle module's
namespace and patched over the original for the duration of one test.
Slips that change nothing on valid inputs (the clamp q <= m in fill_count
is never active for phi <= 1) are not listed.
"""
import importlib.util
import inspect
import os
import textwrap

import numpy as np
import pytest

from oracle import moe_oracle as O

_HERE = os.path.dirname(os.path.abspath(__file__))


def _load_pins():
    spec = importlib.util.spec_from_file_location("oracle_pins", os.path.join(_HERE, "test_oracle.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    pins = []
    for name, fn in vars(mod).items():
        if not name.startswith("test_") or not callable(fn):
            continue
        # generator pins (input maps, locality) only re-check the inputs
        if name in ("test_redraw_maps_give_gap", "test_batched_decode_locality"):
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if marks:
            argname, values = marks[0].args[0], marks[0].args[1]
            pins += [(f"{name}[{i}]", fn, {argname: v}) for i, v in enumerate(values)]
        else:
            pins.append((name, fn, {}))
    return pins


PINS = _load_pins()

# (what the slip is, oracle function, [(original text, planted text), ...])
MUTANTS = [
    ("router bias subtracted", "router_logits",
     [("logits = logits + np.asarray(bias", "logits = logits - np.asarray(bias")]),
    ("router rows taken in reverse order", "router_logits",
     [("np.asarray(w_router, np.float64).T", "np.asarray(w_router, np.float64)[::-1].T")]),
    ("top-k ties go to the higher id", "select_topk",
     [("np.lexsort((expert, -logits[t]))", "np.lexsort((-expert, -logits[t]))")]),
    ("top-k ids left in score order", "select_topk",
     [("chosen = np.sort(order[:k])", "chosen = order[:k]")]),
    ("top-k off by one", "select_topk",
     [("np.sort(order[:k])", "np.sort(order[1:k + 1])")]),
    ("weights not renormalised over the selection", "select_topk",
     [("w[t] = z / z.sum()", "w[t] = z / np.exp(logits[t] - logits[t, chosen].max()).sum()")]),
    ("dispatch not stable within an expert", "dispatch",
     [("cursor = offsets[:-1].copy()", "cursor = offsets[1:].copy() - 1"),
      ("cursor[e] += 1", "cursor[e] -= 1")]),
    ("dispatch offsets as an inclusive scan", "dispatch",
     [("offsets[1:] = np.cumsum(counts)", "offsets[:-1] = np.cumsum(counts)")]),
    ("silu with the sign of the exponent flipped", "silu",
     [("1.0 + np.exp(-z)", "1.0 + np.exp(z)")]),
    ("activation on the up projection", "swiglu_expert",
     [("(silu(g) * u)", "(silu(u) * g)")]),
    ("activation dropped", "swiglu_expert",
     [("(silu(g) * u)", "(g * u)")]),
    ("gate and up weights swapped", "swiglu_expert",
     [("g = x_rows @ w_gate.T", "g = x_rows @ w_up.T"), ("u = x_rows @ w_up.T", "u = x_rows @ w_gate.T")]),
    ("expert rows index tokens by i mod k", "expert_rows",
     [("[rows // k]", "[rows % k]")]),
    ("combine pairs weights in reverse", "combine",
     [("topk_w[:, j:j + 1]", "topk_w[:, k - 1 - j:k - j]")]),
    ("combine reads rows transposed", "combine",
     [("inv_perm[np.arange(T) * k + j]", "inv_perm[(np.arange(T) + j * T) % inv_perm.size]")]),
    ("layer drops the router bias", "layer_forward",
     [("router_logits(x, w_router, bias)", "router_logits(x, w_router, None)")]),
    ("split merge takes rows from the wrong side", "layer_forward_split",
     [("np.where(row_in_F[:, None], yF, yC)", "np.where(row_in_F[:, None], yC, yF)")]),
    ("brute force not renormalised", "layer_forward_bruteforce",
     [("denom = sum(full[e] for e in chosen)", "denom = sum(full)")]),
    ("q: makespan tie goes to the larger count", "fill_count",
     [("makespan(base + 1) < makespan(base)", "makespan(base + 1) <= makespan(base)")]),
    ("q: branch costs swapped", "fill_count",
     [("max(f * (Q16 - phi_q16), (m - f) * phi_q16)", "max(f * phi_q16, (m - f) * (Q16 - phi_q16))")]),
    ("q: floor of one applied at phi = 0", "fill_count",
     [("if min_fill and phi_q16 > 0 and m > 0:", "if min_fill and m > 0:")]),
    ("q: plain rounding of m * phi", "fill_count",
     [("q = base + 1 if makespan(base + 1) < makespan(base) else base",
       "q = (m * phi_q16 + Q16 // 2) // Q16")]),
    ("phi truncated instead of rounded", "phi_to_q16",
     [("round(phi * Q16)", "int(phi * Q16)")]),
    ("SplitMix64 last shift", "splitmix64",
     [("return z ^ (z >> 31)", "return z ^ (z >> 30)")]),
    ("SplitMix64 multiplier", "splitmix64",
     [("0xBF58476D1CE4E5B9", "0xBF58476D1CE4E5B8")]),
    ("victims most recent first", "bind",
     [("key=lambda v: (int(stamp[v]), v)", "key=lambda v: (-int(stamp[v]), v)")]),
    ("victim ties to the higher slot", "bind",
     [("key=lambda v: (int(stamp[v]), v)", "key=lambda v: (int(stamp[v]), -v)")]),
    ("evicted pair not rebound to staging", "bind",
     [("table[old] = STAGING_TAG | old", "pass")]),
    ("hits not refreshed", "bind",
     [("stamp[int(table[base + e])] = now", "pass")]),
    ("slots hit this call may be evicted", "bind",
     [("candidates = [v for v in range(n_slots) if stamp[v] != now]", "candidates = list(range(n_slots))")]),
    ("fill set = highest-id misses", "bind",
     [("F = misses[:q]", "F = misses[len(misses) - q:]")]),
    ("in-place misses left unbound", "bind",
     [("table[base + e] = STAGING_TAG | (base + e)", "table[base + e] = -1")]),
    ("clock not advanced", "bind",
     [("now = st[\"clock\"] + 1", "now = st[\"clock\"]")]),
    ("fills not stamped", "bind",
     [("        stamp[v] = now\n", "\n")]),
    ("E2M1 exponent bias 0", "e2m1_value",
     [("2.0 ** (exp - 1)", "2.0 ** exp")]),
    ("E2M1 subnormal read as 1.0", "e2m1_value",
     [("return sign * 0.5 * man", "return sign * 1.0 * man")]),
    ("E8M0 bias 128", "e8m0_value",
     [("2.0 ** (s - 127)", "2.0 ** (s - 128)")]),
    ("MX nibbles swapped", "mx_dequant",
     [("nib[:, 0::2] = codes & 0xF", "nib[:, 0::2] = codes >> 4"),
      ("nib[:, 1::2] = codes >> 4", "nib[:, 1::2] = codes & 0xF")]),
    ("MX scale per element index mod 32", "mx_dequant",
     [("np.repeat(scale[scales], MX_BLOCK, axis=1)", "np.tile(scale[scales], (1, MX_BLOCK))")]),
    ("E4M3 exponent bias 8", "e4m3_value",
     [("2.0 ** (exp - 7)", "2.0 ** (exp - 8)")]),
    ("E4M3 subnormal without the 2^-6", "e4m3_value",
     [("sign * 2.0 ** -6 * (man / 8.0)", "sign * (man / 8.0)")]),
    ("E4M3 S.1111.110 read as NaN", "e4m3_value",
     [("if exp == 0xF and man == 0x7:", "if exp == 0xF and man >= 0x6:")]),
    ("NVFP4 blocks of 32", "nvfp4_dequant",
     [("np.repeat(scale[scales], NV_BLOCK, axis=1)", "np.repeat(scale[scales], 2 * NV_BLOCK, axis=1)[:, :K]")]),
    ("NVFP4 tensor scale dropped", "nvfp4_dequant",
     [(" * float(np.float32(tensor_scale))", "")]),
]


def _mutant(name, subs):
    src = textwrap.dedent(inspect.getsource(getattr(O, name)))
    for old, new in subs:
        assert src.count(old) == 1, f"mutant of {name} no longer applies: {old!r}"
        src = src.replace(old, new)
    ns = dict(vars(O))
    exec(compile(src, f"<mutant of {name}>", "exec"), ns)
    return ns[name]


def _fails(fn, kwargs):
    try:
        with np.errstate(all="ignore"):
            fn(**kwargs)
    except Exception:            # an assertion, or the slip breaking a later step outright
        return True
    return False


def test_pins_pass_on_the_unmodified_oracle():
    failing = [label for label, fn, kw in PINS if _fails(fn, kw)]
    assert not failing, failing


@pytest.mark.parametrize("what,name,subs", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_a_pin_catches_the_planted_slip(what, name, subs, monkeypatch):
    monkeypatch.setattr(O, name, _mutant(name, subs))
    caught = any(_fails(fn, kw) for _label, fn, kw in PINS)   # stops at the first pin that fails
    assert caught, f"no pin fails when the oracle has this slip: {what}"
