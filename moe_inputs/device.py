"""Upload the seeded inputs of ``moe_inputs.gen`` into CUDA tensors (torch).

Plain copies only: expert banks are filled by slicing the uploaded pools at
the generator's offsets, the cache pool by copying staging slots, and the
residency state is uploaded as is.  No step of the layer is computed here.
"""
import numpy as np
import torch

import edge_moe_serving_gb300 as moe

from . import gen
from .configs import LayerConfig


def to_dev_bf16(bits: np.ndarray, device) -> torch.Tensor:
    # writable and C-contiguous (copied only when needed): torch.from_numpy warns on read-only arrays
    return torch.from_numpy(np.require(bits, requirements=["C", "W"]).view(np.int16)).to(device).view(torch.bfloat16)


def to_dev(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.require(a, requirements=["C", "W"])).to(device)


class DeviceCache:
    """Cache pool (A), staging pool (B) and residency state on one device."""

    def __init__(self, cfg: LayerConfig, device="cuda", staging_layers=None, staging_host=False):
        """staging_host: the staging pool (every (layer, expert) pair) lives in
        pinned host memory, which the GPU reads in place and copies from; the
        cache pool stays in device memory."""
        self.cfg = cfg
        self.device = device
        self.staging_host = staging_host
        L, E, H, I = cfg.n_layers, cfg.E, cfg.H, cfg.I
        LE = L * E
        where = dict(device="cpu", pin_memory=True) if staging_host else dict(device=device)
        self.staging = [torch.empty((LE,) + gen.bank_shape(cfg, b), dtype=torch.bfloat16, **where)
                        for b in range(3)]
        n = I * H
        for layer in range(L):
            for b in range(3):
                bits = gen.bank_pool(cfg, layer, b)
                pool = to_dev_bf16(bits, "cpu" if staging_host else device)
                offs = gen.bank_offsets(cfg, layer, b)
                dst = self.staging[b]
                for e in range(E):
                    o = int(offs[e])
                    dst[layer * E + e].copy_(pool[o:o + n].view(gen.bank_shape(cfg, b)))
                del pool
        st = gen.initial_cache(cfg)
        self.identity = cfg.cache_slots is None
        if self.identity and not staging_host:
            self.cache = self.staging
        else:
            self.cache = [self._gather(b, st["owner"]) for b in range(3)]
        self.table = to_dev(st["table"].astype(np.int32), device)
        self.owner = to_dev(st["owner"].astype(np.int32), device)
        self.stamp = to_dev(st["stamp"].astype(np.uint32).view(np.int32), device)
        self.clock = torch.zeros(1, dtype=torch.int32, device=device)
        self.initial = st
        self.struct = self._make_struct()

    def _gather(self, b, owner):
        """Cache-pool contents of bank b: the staging slots the owners name."""
        idx = torch.from_numpy(np.asarray(owner, np.int64))
        src = self.staging[b]
        if self.staging_host:
            return src.index_select(0, idx).to(self.device)
        return src.index_select(0, idx.to(self.device))

    def n_cache_slots(self):
        return self.cache[0].shape[0]

    def _make_struct(self):
        c = moe.moe_cache()
        c.cache = moe.moe_pool(self.cache[0].data_ptr(), self.cache[1].data_ptr(), self.cache[2].data_ptr(),
                               self.n_cache_slots())
        c.staging = moe.moe_pool(self.staging[0].data_ptr(), self.staging[1].data_ptr(),
                                 self.staging[2].data_ptr(), self.staging[0].shape[0], 1 if self.staging_host else 0)
        c.slot_table = self.table.data_ptr()
        c.owner = self.owner.data_ptr()
        c.stamp = self.stamp.data_ptr()
        c.clock = self.clock.data_ptr()
        c.n_layers, c.E, c.H, c.I = self.cfg.n_layers, self.cfg.E, self.cfg.H, self.cfg.I
        return c

    def state(self):
        """Residency state as numpy, in the oracle's format."""
        return {"table": self.table.cpu().numpy().astype(np.int64),
                "owner": self.owner.cpu().numpy().astype(np.int64),
                "stamp": self.stamp.cpu().numpy().view(np.uint32).astype(np.int64),
                "clock": int(self.clock.cpu().numpy().view(np.uint32)[0])}

    def reset(self):
        """Restore the initial residency state and the cache pool contents."""
        st = self.initial
        self.table.copy_(to_dev(st["table"].astype(np.int32), self.device))
        self.owner.copy_(to_dev(st["owner"].astype(np.int32), self.device))
        self.stamp.zero_()
        self.clock.zero_()
        if self.cache is not self.staging:
            for b in range(3):
                self.cache[b].copy_(self._gather(b, st["owner"]))


class DeviceLayer:
    """Router weights, bias and struct of one layer of a workload."""

    def __init__(self, cfg: LayerConfig, layer: int, device="cuda", step: int = 0):
        self.cfg = cfg
        self.layer = layer
        self.w_router = to_dev(gen.w_router(cfg, layer), device)
        b = gen.bias(cfg, layer, step)
        self.bias = None if b is None else to_dev(b, device)
        self.struct = moe.moe_layer(self.w_router.data_ptr(), None if self.bias is None else self.bias.data_ptr(),
                                    layer, cfg.E, cfg.k, cfg.H, cfg.I)

    def set_bias(self, step: int):
        b = gen.bias(self.cfg, self.layer, step)
        if b is not None:
            self.bias.copy_(to_dev(b, self.bias.device))


def x_dev(cfg: LayerConfig, layer: int, step: int, device="cuda") -> torch.Tensor:
    return to_dev_bf16(gen.x_bits(cfg, layer, step), device)


class MxPool:
    """One MXFP4 pool on the device: six slot-major uint8 banks (codes and
    scales of gate, up, down) and the moe_pool_mxfp4 struct naming them.
    ``experts`` maps slot -> (gate_q, gate_s, up_q, up_s, down_q, down_s)
    arrays; slots not listed stay zero (never read)."""

    def __init__(self, n_slots, H, I, experts, device="cuda"):
        shapes = [(I, H // 2), (I, H // 32), (I, H // 2), (I, H // 32), (H, I // 2), (H, I // 32)]
        self.banks = [torch.zeros((n_slots,) + s, dtype=torch.uint8, device=device) for s in shapes]
        for slot, arrays in experts.items():
            self.set(slot, arrays)
        self.struct = moe.moe_pool_mxfp4(*[b.data_ptr() for b in self.banks], n_slots, 0)

    def set(self, slot, arrays):
        for bank, a in zip(self.banks, arrays):
            bank[slot].copy_(torch.from_numpy(np.require(a, requirements=["C", "W"])))


class NvPool:
    """One NVFP4 pool on the device: six slot-major uint8 banks (codes and
    E4M3 scales of gate, up, down), the fp32 tensor scales [n_slots, 3] and
    the moe_pool_nvfp4 struct naming them.  ``experts`` maps slot ->
    ((gate_q, gate_s, gate_ts), (up_q, up_s, up_ts), (down_q, down_s,
    down_ts)); slots not listed stay zero (never read)."""

    def __init__(self, n_slots, H, I, experts, device="cuda"):
        shapes = [(I, H // 2), (I, H // 16), (I, H // 2), (I, H // 16), (H, I // 2), (H, I // 16)]
        self.banks = [torch.zeros((n_slots,) + s, dtype=torch.uint8, device=device) for s in shapes]
        self.tscale = torch.zeros((n_slots, 3), dtype=torch.float32, device=device)
        for slot, banks in experts.items():
            self.set(slot, banks)
        self.struct = moe.moe_pool_nvfp4(*[b.data_ptr() for b in self.banks], self.tscale.data_ptr(), n_slots, 0)

    def set(self, slot, banks):
        for b, (codes, scales, ts) in enumerate(banks):
            self.banks[2 * b][slot].copy_(torch.from_numpy(np.require(codes, requirements=["C", "W"])))
            self.banks[2 * b + 1][slot].copy_(torch.from_numpy(np.require(scales, requirements=["C", "W"])))
            self.tscale[slot, b] = float(ts)


class Fp4Cache:
    """An FP4 expert cache on one device: the staging pool (every (layer,
    expert) pair of ``cfg`` at slot layer*E + expert), the cache pool holding
    the initial owners of gen.initial_cache(cfg), the residency arrays and the
    moe_cache_fp4 struct.  ``fmt``: moe.MOE_FP4_MXFP4 (banks from
    gen.mx_expert) or moe.MOE_FP4_NVFP4 (gen.nvfp4_expert)."""

    def __init__(self, cfg: LayerConfig, fmt, seed, device="cuda"):
        self.cfg, self.fmt, self.seed, self.device = cfg, fmt, seed, device
        nv = fmt == moe.MOE_FP4_NVFP4
        sb = 16 if nv else 32
        L, E, H, I = cfg.n_layers, cfg.E, cfg.H, cfg.I
        LE = L * E
        shapes = [(I, H // 2), (I, H // sb), (I, H // 2), (I, H // sb), (H, I // 2), (H, I // sb)]
        host = [np.zeros((LE,) + s, np.uint8) for s in shapes]
        tscale = np.zeros((LE, 3), np.float32)
        for layer in range(L):
            for e in range(E):
                slot = layer * E + e
                if nv:
                    for b, (codes, scales, ts) in enumerate(gen.nvfp4_expert(seed, layer, e, H, I)):
                        host[2 * b][slot], host[2 * b + 1][slot], tscale[slot, b] = codes, scales, ts
                else:
                    for b, a in enumerate(gen.mx_expert(seed, layer, e, H, I)):
                        host[b][slot] = a
        self.staging = [torch.from_numpy(a).to(device) for a in host]
        self.staging_ts = torch.from_numpy(tscale).to(device) if nv else None
        st = gen.initial_cache(cfg)
        idx = torch.from_numpy(np.asarray(st["owner"], np.int64)).to(device)
        self.cache = [b.index_select(0, idx) for b in self.staging]
        self.cache_ts = self.staging_ts.index_select(0, idx) if nv else None
        self.table = to_dev(st["table"].astype(np.int32), device)
        self.owner = to_dev(st["owner"].astype(np.int32), device)
        self.stamp = to_dev(st["stamp"].astype(np.uint32).view(np.int32), device)
        self.clock = torch.zeros(1, dtype=torch.int32, device=device)
        self.initial = st
        c = moe.moe_cache_fp4()
        ptr = lambda t: None if t is None else t.data_ptr()
        c.cache = moe.moe_pool_nvfp4(*[b.data_ptr() for b in self.cache], ptr(self.cache_ts), len(st["owner"]), 0)
        c.staging = moe.moe_pool_nvfp4(*[b.data_ptr() for b in self.staging], ptr(self.staging_ts), LE, 0)
        c.slot_table, c.owner, c.stamp, c.clock = (self.table.data_ptr(), self.owner.data_ptr(),
                                                   self.stamp.data_ptr(), self.clock.data_ptr())
        c.n_layers, c.E, c.H, c.I, c.format = L, E, H, I, fmt
        self.struct = c

    def state(self):
        """Residency state as numpy, in the oracle's format."""
        return {"table": self.table.cpu().numpy().astype(np.int64),
                "owner": self.owner.cpu().numpy().astype(np.int64),
                "stamp": self.stamp.cpu().numpy().view(np.uint32).astype(np.int64),
                "clock": int(self.clock.cpu().numpy().view(np.uint32)[0])}

    def reset(self):
        """Restore the initial residency state and the cache pool contents."""
        st = self.initial
        self.table.copy_(to_dev(st["table"].astype(np.int32), self.device))
        self.owner.copy_(to_dev(st["owner"].astype(np.int32), self.device))
        self.stamp.zero_()
        self.clock.zero_()
        idx = torch.from_numpy(np.asarray(st["owner"], np.int64)).to(self.device)
        for c, s in zip(self.cache, self.staging):
            c.copy_(s.index_select(0, idx))
        if self.cache_ts is not None:
            self.cache_ts.copy_(self.staging_ts.index_select(0, idx))

    def cache_matches_owners(self):
        """Whether every cache slot's banks (and tensor scales) equal, byte for
        byte, the staging slot of the (layer, expert) pair that owns it."""
        idx = self.owner.to(torch.int64)
        pairs = list(zip(self.cache, self.staging))
        if self.cache_ts is not None:
            pairs.append((self.cache_ts, self.staging_ts))
        return all(torch.equal(c, s.index_select(0, idx)) for c, s in pairs)
