"""Shared pieces of the GPU parity tests: device workspaces, oracle caches and
the tolerance check written in the contract (relative Frobenius error
<= 1e-2 and max-abs error <= 2e-2 for layer outputs)."""
import collections
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import edge_moe_serving_gb300 as moe
from moe_inputs import gen
from oracle import moe_oracle as O

REL_FRO = 1e-2
MAX_ABS = 2e-2
DEV = "cuda"


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(gpu, ref, rel_fro=REL_FRO, max_abs=MAX_ABS, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    d = gpu - ref
    denom = np.linalg.norm(ref)
    rel = np.linalg.norm(d) / denom if denom > 0 else np.linalg.norm(d)
    mx = float(np.abs(d).max()) if d.size else 0.0
    assert rel <= rel_fro and mx <= max_abs, f"{what}: rel_fro={rel:.3e} max_abs={mx:.3e}"
    return rel, mx


class ExpertCache:
    """fp64 weights of logical experts, most recently used kept."""

    def __init__(self, cfg, cap=24):
        self.cfg = cfg
        self.cap = cap
        self.d = collections.OrderedDict()

    def __call__(self, layer, e):
        key = (layer, e)
        if key in self.d:
            self.d.move_to_end(key)
            return self.d[key]
        w = gen.expert_f64(self.cfg, layer, e)
        self.d[key] = w
        if len(self.d) > self.cap:
            self.d.popitem(last=False)
        return w


def zeros_i32(n):
    return torch.zeros(max(int(n), 1), dtype=torch.int32, device=DEV)


def ws(nbytes):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=DEV)


def status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def status_bits(s):
    return int(s.cpu().numpy().view(np.uint32)[0])


def token_major(ref):
    """The oracle's expert rows (dispatch order) in the token-major order the
    library writes: row t*k + j = output of token t's j-th expert."""
    return ref["y_rows"][ref["inv_perm"]]


def oracle_layer(cfg, layer, step, wcache, x_bits=None, tokens=None):
    """Oracle forward of (layer, step) on the workload's inputs."""
    xb = gen.x_bits(cfg, layer, step) if x_bits is None else x_bits
    x = gen.bf16_bits_to_f64(xb)
    return O.layer_forward(x, gen.w_router(cfg, layer), gen.bias(cfg, layer, step), cfg.k,
                           lambda e: wcache(layer, e), E=cfg.E)


def run_layer(dc, dl, x, T, phi_q16, min_fill, policy, seed=0, ffn_mode=moe.MOE_FFN_AUTO, stream=None,
              want_y_rows=True):
    """moe_layer_forward with caller buffers for the intermediates.

    ``want_y_rows=False`` leaves the fp32 expert rows inside the library's
    workspace, which is how the benchmark calls the layer (on the GEMM path
    the rows are then kept in bf16)."""
    cfg = dc.cfg
    R = T * cfg.k
    bufs = {"topk_ids": torch.empty(R, dtype=torch.int32, device=DEV),
            "topk_w": torch.empty(R, dtype=torch.float32, device=DEV),
            "counts": torch.empty(cfg.E, dtype=torch.int32, device=DEV),
            "offsets": torch.empty(cfg.E + 1, dtype=torch.int32, device=DEV),
            "perm": torch.empty(R, dtype=torch.int32, device=DEV),
            "inv_perm": torch.empty(R, dtype=torch.int32, device=DEV)}
    if want_y_rows:
        bufs["y_rows"] = torch.empty((R, cfg.H), dtype=torch.float32, device=DEV)
    b = moe.moe_layer_buffers(*[bufs[f].data_ptr() if f in bufs else None for f, _ in moe.moe_layer_buffers._fields_])
    nbytes = moe.moe_layer_workspace_size(dl.struct, dc.struct, T, ffn_mode)
    w = ws(nbytes)
    out = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=DEV)
    st = status()
    stats = torch.zeros(8, dtype=torch.int32, device=DEV)
    moe.moe_layer_forward(dl.struct, dc.struct, x, T, out, phi_q16, min_fill, policy, seed, ffn_mode, b, w,
                          nbytes, st, stats, stream)
    torch.cuda.synchronize()
    bufs["out"] = out
    bufs["status"] = status_bits(st)
    bufs["stats"] = dict(zip(moe.BIND_STATS_FIELDS, stats.cpu().numpy().tolist()))
    return bufs


def oracle_tokens(cfg, layer, step, toks, workers=8):
    """Oracle layer output of the listed tokens of (layer, step).

    Router, top-k, dispatch, per-expert SwiGLU and combine are the oracle's
    own functions, applied to those token rows; every step of the layer acts
    per token, so this is the full block's output restricted to them.  The
    experts are evaluated in worker threads (numpy releases the GIL in its
    conversions and matmuls).  Returns (out [n, H], ids [n, k])."""
    toks = np.asarray(toks)
    x = gen.bf16_bits_to_f64(gen.x_bits(cfg, layer, step)[toks])
    ids, w = O.select_topk(O.router_logits(x, gen.w_router(cfg, layer), gen.bias(cfg, layer, step)), cfg.k)
    counts, offsets, perm, inv = O.dispatch(ids, cfg.E)
    for b in range(3):
        gen.bank_pool(cfg, layer, b)           # fill the generator's cache once, before the threads

    def one(e):
        return e, O.expert_rows(x, ids, offsets, perm, lambda ee: gen.expert_f64(cfg, layer, ee), [e], cfg.k)[e]

    y = np.zeros((ids.size, cfg.H))
    with ThreadPoolExecutor(workers) as ex:
        for e, rows in ex.map(one, np.nonzero(counts)[0]):
            y[offsets[e]:offsets[e + 1]] = rows
    return O.combine(y, inv, w, cfg.k), ids
