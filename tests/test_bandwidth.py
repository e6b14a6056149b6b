"""Host arithmetic of the bandwidth profile (moe_phi_to_q16, moe_bw_derive)
pinned to the paper's Table 1 and the values the write-up prints for it, and
the argument checks of moe_bench_bandwidth, which answer without a GPU."""
import math
import os

import numpy as np
import pytest

import edge_moe_serving_gb300 as moe
from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def test_phi_to_q16_rounds_half_to_even_and_clamps():
    q = moe.moe_phi_to_q16
    assert q(0.5 / 65536) == 0 and q(1.5 / 65536) == 2 and q(2.5 / 65536) == 2 and q(3.5 / 65536) == 4
    assert q(0.0) == 0 and q(-0.3) == 0 and q(float("nan")) == 0
    assert q(1.0) == 65536 and q(1.7) == 65536 and q(float("inf")) == 65536
    for phi in np.linspace(0.0, 1.0, 2001):
        assert q(float(phi)) == O.phi_to_q16(float(phi)), phi


def test_derive_reproduces_table1_values_printed_by_the_writeup():
    table = {r[0]: (float(r[1]), float(r[2])) for r in _rows("table1_bandwidths.txt")}
    printed = _rows("phi_gate_writeup.txt")
    assert len(printed) == 6
    for name, phi_s, q4, gate in printed:
        bp, bh = table[name]
        prof = moe.moe_bw_derive(bp, bh)
        assert round(prof.phi, 3) == float(phi_s), name
        assert prof.phi_q16 == O.phi_to_q16(bp / bh), name
        assert O.fill_count(4, prof.phi_q16, min_fill=0) == int(q4), name
        assert prof.hybrid_ok == (1 if gate == "pass" else 0), name


def test_contended_fraction_reduces_to_eq4_under_full_contention():
    """With the copy taking its full B_P and the in-place path the residual
    B_H - B_P (Eq. 3's model), the copy's share of the contended total is
    B_P / B_H: the contended phi equals Eq. 4's."""
    for _, bp, bh, _r in _rows("table1_bandwidths.txt"):
        bp, bh = float(bp), float(bh)
        prof = moe.moe_bw_derive(bp, bh, bp, bh - bp)
        assert math.isclose(prof.phi_contended, prof.phi, rel_tol=1e-12)
        assert prof.phi_contended_q16 == prof.phi_q16
    # a copy that never slows the in-place path: the share falls below B_P / B_H
    prof = moe.moe_bw_derive(40.0, 100.0, 40.0, 100.0)
    assert math.isclose(prof.phi_contended, 40.0 / 140.0) and prof.phi_contended < prof.phi


def test_derive_endpoints_and_bad_rates():
    p = moe.moe_bw_derive(50.0, 0.0)          # no in-place path: every miss fills
    assert p.phi == 1.0 and p.phi_q16 == 65536 and p.hybrid_ok == 0
    assert O.fill_count(9, p.phi_q16) == 9
    p = moe.moe_bw_derive(0.0, 80.0)          # no copy path: nothing crosses (Eq. 4 endpoint)
    assert p.phi == 0.0 and p.phi_q16 == 0 and p.hybrid_ok == 1
    assert O.fill_count(9, p.phi_q16, min_fill=1) == 0
    p = moe.moe_bw_derive(0.0, 0.0)
    assert p.phi == 0.0 and p.phi_contended == 0.0 and p.hybrid_ok == 0
    assert moe.moe_bw_derive(10.0, 20.0).hybrid_ok == 0   # B_H = 2 B_P: not above the gate
    assert moe.moe_bw_derive(10.0, 20.001).hybrid_ok == 1
    for bad in ((-1.0, 5.0), (5.0, float("nan")), (float("inf"), 5.0), (1.0, 1.0, -2.0, 0.0)):
        with pytest.raises(moe.MoeError) as e:
            moe.moe_bw_derive(*bad)
        assert e.value.status == moe.MOE_ERR_INVALID_ARG


def test_bench_bandwidth_rejects_bad_arguments_before_any_cuda_call():
    bad = [(0, 4096, 1 << 20, 2, 1, 2),          # null host buffer
           (4096, 4096, 15, 2, 1, 2),            # not a multiple of 16 bytes
           (4096, 4096, 0, 2, 1, 2),             # empty
           (4096, 4096, 1 << 20, 0, 1, 2),       # no repetition
           (4096, 4096, 1 << 20, 2, 3, 3),       # one stream for both sides
           (4104, 4096, 1 << 20, 2, 1, 2),      # host buffer not 16-byte aligned
           (4096, 4096, 1 << 20, 2, 0, 2)]       # the legacy default stream
    for args in bad:
        with pytest.raises(moe.MoeError) as e:
            moe.moe_bench_bandwidth(*args)
        assert e.value.status == moe.MOE_ERR_INVALID_ARG, args
