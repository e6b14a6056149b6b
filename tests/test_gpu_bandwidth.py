"""moe_bench_bandwidth on the GPU: the four rates are measured, the derived
fields are moe_bw_derive's, the copy lands, and the in-place read sees every
byte of the pinned host buffer (its XOR checksum equals the host's)."""
import math

import numpy as np
import pytest
import torch

import edge_moe_serving_gb300 as moe

pytestmark = pytest.mark.gpu


def test_bench_bandwidth_measures_and_reads_every_byte():
    n = 48 << 20
    rng = np.random.default_rng(5)
    words = rng.integers(0, 2 ** 32, n // 4, dtype=np.uint64).astype(np.uint32)
    host = torch.from_numpy(words.view(np.int32)).pin_memory()
    dev = torch.zeros(n // 4, dtype=torch.int32, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    prof = moe.moe_bench_bandwidth(host, dev, n, 3, s1, s2)
    torch.cuda.synchronize()
    for r in (prof.b_p_gbs, prof.b_h_gbs, prof.b_p_contended_gbs, prof.b_h_contended_gbs):
        assert math.isfinite(r) and r > 0.0
    assert prof.read_checksum == int(np.bitwise_xor.reduce(words))
    assert torch.equal(dev.cpu(), host)
    ref = moe.moe_bw_derive(prof.b_p_gbs, prof.b_h_gbs, prof.b_p_contended_gbs, prof.b_h_contended_gbs)
    assert ref.phi == prof.phi and ref.phi_contended == prof.phi_contended
    assert (ref.phi_q16, ref.phi_contended_q16, ref.hybrid_ok) == (prof.phi_q16, prof.phi_contended_q16,
                                                                   prof.hybrid_ok)


def test_bench_bandwidth_ragged_size():
    """A size that is not a multiple of the read grid's stride: the tail loop."""
    n = (3 << 20) + 48
    words = (np.arange(n // 4, dtype=np.uint64) * 2654435761 % (1 << 32)).astype(np.uint32)
    host = torch.from_numpy(words.view(np.int32)).pin_memory()
    dev = torch.zeros(n // 4, dtype=torch.int32, device="cuda")
    prof = moe.moe_bench_bandwidth(host, dev, n, 1, torch.cuda.Stream(), torch.cuda.Stream())
    assert prof.read_checksum == int(np.bitwise_xor.reduce(words))
    assert torch.equal(dev.cpu(), host)
