"""Plain CPU fp64 oracle of one routed MoE layer's forward pass (FreeToken).

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline may import this module.  The GPU library never calls it and shares
no code with it.

Source pages
------------
[P]  "FreeToken: Efficient Edge-Native MoE Serving with Bandwidth-Adaptive
     Execution" (arXiv 2608.16157): section 3 (two-level expert hierarchy,
     (layer, expert) slots), section 3.2 (router + cache lookup, Eq. 1-4,
     integer q, exact merge of partial sums), section 4.1 (device-side cache
     control, single-pass K-LRU victims, fused fill copy), section 4.2 (expert
     banks with leading dimension lE+e).
[W]  "FreeToken: bandwidth-adaptive edge MoE serving" (write-up of the
     repository): section "The split, and what it is actually optimising"
     (the Q16 integer rounding of q*), section "Decode residency: one LRU
     across all layers" (overflow misses).

Readings where the pages are silent:
  * router scores: softmax over the router logits, top-k, renormalised over
    the k selected experts (the tiny workload's "top-2 softmax-renormalised");
  * top-k ties go to the lower expert id; selected ids are listed ascending;
  * SwiGLU expert: y = W_down (silu(W_gate x) * (W_up x)), silu(z) = z/(1+e^-z);
  * the "at least one fill" floor of [P] 3.2 applies when min_fill=1, phi>0
    and m>=1; [W] records that the shipped rule has no floor (min_fill=0);
  * LRU: one clock shared by all layers, +1 per bind call; hits and fills
    take the current stamp; victims are the least (stamp, slot) slots not
    stamped by this call; F is paired with victims in ascending order;
  * F is the q lowest-id misses (policy 0) or a seeded random q-subset
    (policy 1, SplitMix64 keys); misses left in C, including overflow when
    fewer victims than q exist, are bound to the staging pool.

Block-scaled FP4 experts ([P] section 5.1 "Models": the routed experts of
DeepSeek-V4-Flash are natively MXFP4; section 4.1: expert kernels dequantise
in-kernel).  The element and scale encodings follow the OCP Microscaling
Formats (MX) v1.0 specification: FP4 E2M1 elements, one E8M0 scale per block
of 32 consecutive elements along the input dimension.  Readings: two codes per
byte, the even element in the low nibble; a weight row of K inputs is K/2 code
bytes and K/32 scale bytes.

NVFP4 experts ([P] section 5.1 "Models": GLM-5.2's routed experts and the
laptop build of Qwen3.6-35B-A3B are NVFP4): FP4 E2M1 elements with one FP8
E4M3 scale per block of 16 consecutive inputs and one fp32 scale per weight
tensor, as NVIDIA describes the format; E4M3 as in the OCP 8-bit floating
point specification (the variant without infinities).  Readings: the same
nibble packing as MXFP4; the block scale is the raw E4M3 byte; one tensor
scale per bank of an expert.

Everything is fp64 except where the inputs are stored (bf16 / fp32 values are
widened exactly).  Library primitives used as steps: numpy matmul, exp,
bincount, cumsum, sort.
"""
import numpy as np

Q16 = 1 << 16
STAGING_TAG = 1 << 30
MASK64 = (1 << 64) - 1
FILL_LOWEST_ID = 0
FILL_RANDOM = 1


# ------------------------------------------------------------------ router
def router_logits(x, w_router, bias=None):
    """[P] 3.2: the router scores every expert for every token.

    logits[t, e] = sum_h x[t, h] * W_r[e, h] + b[e]   (fp64)."""
    logits = np.asarray(x, np.float64) @ np.asarray(w_router, np.float64).T
    if bias is not None:
        logits = logits + np.asarray(bias, np.float64)[None, :]
    return logits


def select_topk(logits, k):
    """Top-k by (logit descending, id ascending); ids listed ascending.

    Weights are the softmax over the selected logits (max-subtracted), which
    is the full softmax renormalised over the k selected experts."""
    logits = np.asarray(logits, np.float64)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    expert = np.arange(E)
    for t in range(T):
        order = np.lexsort((expert, -logits[t]))      # last key is primary
        chosen = np.sort(order[:k])
        ids[t] = chosen
        z = logits[t, chosen]
        z = np.exp(z - z.max())
        w[t] = z / z.sum()
    return ids, w


def topk_gap(logits, k):
    """Per token: k-th largest logit minus (k+1)-th largest."""
    s = -np.sort(-np.asarray(logits, np.float64), axis=1)
    return s[:, k - 1] - s[:, k]


# ------------------------------------------------------------------ dispatch
def dispatch(topk_ids, E):
    """[P] 3.2: group routed rows per expert for the grouped evaluation.

    Counting sort of the flat rows i = t*k + j by expert id, stable in i:
    counts[e], offsets = exclusive scan (offsets[E] = T*k), perm[pos] = i,
    inv_perm[i] = pos."""
    flat = np.asarray(topk_ids, np.int64).reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    cursor = offsets[:-1].copy()
    perm = np.empty(flat.size, np.int64)
    inv_perm = np.empty(flat.size, np.int64)
    for i, e in enumerate(flat):
        pos = cursor[e]
        cursor[e] += 1
        perm[pos] = i
        inv_perm[i] = pos
    return counts, offsets, perm, inv_perm


# ------------------------------------------------------------------ expert FFN
def silu(z):
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_expert(x_rows, w_gate, w_up, w_down):
    """One expert on a block of rows: y = (silu(x Wg^T) * (x Wu^T)) Wd^T.

    Shapes: x_rows [n, H]; w_gate, w_up [I, H]; w_down [H, I] (out x in)."""
    x_rows = np.asarray(x_rows, np.float64)
    g = x_rows @ w_gate.T
    u = x_rows @ w_up.T
    return (silu(g) * u) @ w_down.T


def expert_rows(x, topk_ids, offsets, perm, weights_of, experts, k):
    """y rows (dispatch order) of the listed experts: {e: [n_e, H]}."""
    out = {}
    for e in experts:
        rows = perm[offsets[e]:offsets[e + 1]]
        if rows.size == 0:
            out[e] = np.zeros((0, np.asarray(x).shape[1]))
            continue
        wg, wu, wd = weights_of(e)
        out[e] = swiglu_expert(np.asarray(x, np.float64)[rows // k], wg, wu, wd)
    return out


def combine(y_rows, inv_perm, topk_w, k):
    """[P] 3.2: out[t] = sum_j w[t, j] * y[inv_perm[t*k + j]], j ascending."""
    T = topk_w.shape[0]
    out = np.zeros((T, y_rows.shape[1]))
    for j in range(k):
        out += topk_w[:, j:j + 1] * y_rows[inv_perm[np.arange(T) * k + j]]
    return out


def layer_forward(x, w_router, bias, k, weights_of, E=None):
    """Router -> top-k -> dispatch -> per-expert SwiGLU -> combine (fp64).

    ``weights_of(e)`` returns (W_gate, W_up, W_down) of logical expert e."""
    x = np.asarray(x, np.float64)
    logits = router_logits(x, w_router, bias)
    E = logits.shape[1] if E is None else E
    ids, w = select_topk(logits, k)
    counts, offsets, perm, inv_perm = dispatch(ids, E)
    y_rows = np.zeros((ids.size, x.shape[1]))
    for e, rows in expert_rows(x, ids, offsets, perm, weights_of, np.nonzero(counts)[0], k).items():
        y_rows[offsets[e]:offsets[e + 1]] = rows
    out = combine(y_rows, inv_perm, w, k)
    return {"logits": logits, "ids": ids, "w": w, "counts": counts, "offsets": offsets,
            "perm": perm, "inv_perm": inv_perm, "y_rows": y_rows, "out": out}


def layer_forward_split(x, w_router, bias, k, weights_of, subset_F):
    """The same layer with the active experts split into F and C = rest.

    Each subset is evaluated on its own (as the GPU branch and the in-place
    branch of [P] 3.2 would) and the merge picks every routed row from the
    subset that owns its expert, then sums in the fixed expert order.  Returns
    (merged output, partial sum over F, partial sum over C)."""
    x = np.asarray(x, np.float64)
    logits = router_logits(x, w_router, bias)
    ids, w = select_topk(logits, k)
    E = logits.shape[1]
    counts, offsets, perm, inv_perm = dispatch(ids, E)
    active = np.nonzero(counts)[0]
    in_F = np.zeros(E, bool)
    in_F[list(subset_F)] = True
    yF = np.zeros((ids.size, x.shape[1]))
    yC = np.zeros((ids.size, x.shape[1]))
    for e, rows in expert_rows(x, ids, offsets, perm, weights_of, active[in_F[active]], k).items():
        yF[offsets[e]:offsets[e + 1]] = rows
    for e, rows in expert_rows(x, ids, offsets, perm, weights_of, active[~in_F[active]], k).items():
        yC[offsets[e]:offsets[e + 1]] = rows
    row_in_F = in_F[np.asarray(ids).reshape(-1)[perm]]       # per dispatch position
    merged_rows = np.where(row_in_F[:, None], yF, yC)
    merged = combine(merged_rows, inv_perm, w, k)
    wF = np.where(in_F[ids], w, 0.0)
    wC = np.where(in_F[ids], 0.0, w)
    return merged, combine(yF, inv_perm, wF, k), combine(yC, inv_perm, wC, k)


def layer_forward_bruteforce(x, w_router, bias, k, weights_of):
    """Per-token definition with no dispatch: loop tokens, loop all experts.

    Selection is k rounds of arg-max (ties to the lower id); weights are the
    full softmax over all E logits renormalised over the selected ones."""
    x = np.asarray(x, np.float64)
    wr = np.asarray(w_router, np.float64)
    T, H = x.shape
    E = wr.shape[0]
    out = np.zeros((T, H))
    for t in range(T):
        logit = [float(np.dot(x[t], wr[e])) + (0.0 if bias is None else float(bias[e]))
                 for e in range(E)]
        chosen = []
        for _ in range(k):
            best = None
            for e in range(E):
                if e in chosen:
                    continue
                if best is None or logit[e] > logit[best]:
                    best = e
            chosen.append(best)
        mx = max(logit)
        full = [np.exp(v - mx) for v in logit]
        denom = sum(full[e] for e in chosen)
        for e in range(E):
            if e in chosen:
                wg, wu, wd = weights_of(e)
                g = wg @ x[t]
                u = wu @ x[t]
                h = np.array([gi / (1.0 + np.exp(-gi)) * ui for gi, ui in zip(g, u)])
                out[t] += (full[e] / denom) * (wd @ h)
    return out


# ------------------------------------------------------------------ q* rule
def fill_count(m, phi_q16, min_fill=0):
    """Integer fetch count q for m misses at fetch fraction phi = B_P/B_H.

    [P] 3.2 Eq. 4 gives q* ~ m * B_P / B_H and rounds it to an integer; [W]
    ("The split, and what it is actually optimising") gives the rounding in
    Q16 integers: start from floor(m * phi), and take that or one more,
    whichever gives the smaller makespan max(f * (1 - phi), (m - f) * phi) of
    the two concurrent branches of Eq. 3 (the lower one when equal), never
    above m.  ``min_fill`` applies [P] 3.2's "at least one fill" floor."""
    m = int(m)
    phi_q16 = int(phi_q16)
    base = (m * phi_q16) // Q16

    def makespan(f):
        return max(f * (Q16 - phi_q16), (m - f) * phi_q16)

    q = base + 1 if makespan(base + 1) < makespan(base) else base
    q = min(q, m)
    if min_fill and phi_q16 > 0 and m > 0:
        q = max(q, 1)
    return q


def phi_to_q16(phi):
    """Fetch fraction to Q16, rounded half to even and clamped to [0, 1]."""
    return int(min(Q16, max(0, round(phi * Q16))))


# ------------------------------------------------------------------ residency
def splitmix64(z):
    """SplitMix64 output for state increment z (Steele, Lea & Flood 2014)."""
    z = (z + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def random_fill_key(seed, now, layer, e):
    """Key that orders the misses for the random F policy (smaller first)."""
    counter = ((int(now) & 0xFFFFFFFF) << 32) | ((int(layer) & 0xFFFF) << 16) | (int(e) & 0xFFFF)
    return splitmix64((int(seed) ^ counter) & MASK64)


def copy_state(state):
    return {"table": np.array(state["table"], np.int64), "owner": np.array(state["owner"], np.int64),
            "stamp": np.array(state["stamp"], np.int64), "clock": int(state["clock"])}


def bind(state, layer, topk_ids, E, phi_q16, min_fill=1, policy=FILL_LOWEST_ID, seed=0):
    """Device-side cache control of [P] 4.1 for one MoE layer, fp-free.

    Deduplicate the routed experts, classify them against the residency
    table (hit H / miss M), derive q from m, choose F (policy) and the
    eviction victims (least recently used, [P] 3.2 and 4.1), rebind the
    evicted pairs to the staging pool, admit F into the victims' slots and
    bind the rest of the misses, C, to the staging pool (the analogue of the
    CPU-assignment flag).  Returns (new state, result dict)."""
    st = copy_state(state)
    table, owner, stamp = st["table"], st["owner"], st["stamp"]
    n_slots = owner.size
    now = st["clock"] + 1
    base = layer * E
    U = sorted(set(int(e) for e in np.asarray(topk_ids).reshape(-1)))
    hits, misses = [], []
    for e in U:
        ent = int(table[base + e])
        if 0 <= ent < n_slots:
            hits.append(e)
        else:
            misses.append(e)
    for e in hits:
        stamp[int(table[base + e])] = now
    m = len(misses)
    q = fill_count(m, phi_q16, min_fill)
    if policy == FILL_LOWEST_ID:
        F = misses[:q]
    else:
        ranked = sorted(misses, key=lambda e: (random_fill_key(seed, now, layer, e), e))
        F = sorted(ranked[:q])
    # repeated evict-min over the slots this call has not stamped
    candidates = [v for v in range(n_slots) if stamp[v] != now]
    victims = []
    for _ in range(len(F)):
        if not candidates:
            break
        best = min(candidates, key=lambda v: (int(stamp[v]), v))
        victims.append(best)
        candidates.remove(best)
    fills = []
    for e, v in zip(F, victims):
        old = int(owner[v])
        if old >= 0:
            table[old] = STAGING_TAG | old
        table[base + e] = v
        owner[v] = base + e
        stamp[v] = now
        fills.append((base + e, v))
    filled = set(F[:len(victims)])
    C = [e for e in misses if e not in filled]
    for e in C:
        table[base + e] = STAGING_TAG | (base + e)
    st["clock"] = now
    result = {"H": hits, "M": misses, "F": sorted(filled), "C": C, "fills": fills,
              "stats": {"n_unique": len(U), "n_hit": len(hits), "n_miss": m, "q": q,
                        "n_fill": len(fills), "n_overflow": q - len(fills), "n_staged": len(C)}}
    return st, result


# ------------------------------------------------------------------ MXFP4 experts
MX_BLOCK = 32


def e2m1_value(code):
    """FP4 E2M1 element (OCP MX v1.0): 1 sign bit, 2 exponent bits (bias 1),
    1 mantissa bit; exponent field 0 is subnormal (0.5 * mantissa)."""
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    exp = (code >> 1) & 0x3
    man = code & 0x1
    if exp == 0:
        return sign * 0.5 * man
    return sign * 2.0 ** (exp - 1) * (1.0 + 0.5 * man)


def e8m0_value(s):
    """E8M0 block scale (OCP MX v1.0): 2^(s - 127); s = 255 is NaN."""
    s = int(s) & 0xFF
    return float("nan") if s == 0xFF else 2.0 ** (s - 127)


def mx_dequant(codes, scales):
    """Dequantise MXFP4 weight rows to fp64.

    codes uint8 [rows, K/2] (element 2c in the low nibble of byte c, 2c+1 in
    the high nibble); scales uint8 [rows, K/32]; returns [rows, K] with
    W[r, i] = e2m1(code of i) * e8m0(scales[r, i // 32])."""
    codes = np.asarray(codes, np.uint8)
    scales = np.asarray(scales, np.uint8)
    rows, half = codes.shape
    K = 2 * half
    assert K % MX_BLOCK == 0 and scales.shape == (rows, K // MX_BLOCK)
    elem = np.array([e2m1_value(c) for c in range(16)])
    scale = np.array([e8m0_value(v) for v in range(256)])
    nib = np.empty((rows, K), np.int64)
    nib[:, 0::2] = codes & 0xF
    nib[:, 1::2] = codes >> 4
    return elem[nib] * np.repeat(scale[scales], MX_BLOCK, axis=1)


def mx_expert_weights(gate_q, gate_s, up_q, up_s, down_q, down_s):
    """(W_gate, W_up, W_down) in fp64 of one MXFP4 expert (out x in rows)."""
    return mx_dequant(gate_q, gate_s), mx_dequant(up_q, up_s), mx_dequant(down_q, down_s)


# ------------------------------------------------------------------ NVFP4 experts
NV_BLOCK = 16


def e4m3_value(b):
    """FP8 E4M3 (OCP 8-bit floating point, no infinities): 1 sign bit, 4
    exponent bits (bias 7), 3 mantissa bits; exponent field 0 is subnormal
    (2^-6 * mantissa / 8); exponent and mantissa all ones is NaN."""
    b = int(b) & 0xFF
    sign = -1.0 if b & 0x80 else 1.0
    exp = (b >> 3) & 0xF
    man = b & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * 2.0 ** -6 * (man / 8.0)
    return sign * 2.0 ** (exp - 7) * (1.0 + man / 8.0)


def nvfp4_dequant(codes, scales, tensor_scale):
    """Dequantise NVFP4 weight rows to fp64.

    codes uint8 [rows, K/2] (element 2c in the low nibble of byte c); scales
    uint8 [rows, K/16] (E4M3 bytes); tensor_scale: the fp32 scale of the
    whole matrix.  W[r, i] = e2m1(code of i) * e4m3(scales[r, i // 16]) * tensor_scale."""
    codes = np.asarray(codes, np.uint8)
    scales = np.asarray(scales, np.uint8)
    rows, half = codes.shape
    K = 2 * half
    assert K % NV_BLOCK == 0 and scales.shape == (rows, K // NV_BLOCK)
    elem = np.array([e2m1_value(c) for c in range(16)])
    scale = np.array([e4m3_value(v) for v in range(256)])
    nib = np.empty((rows, K), np.int64)
    nib[:, 0::2] = codes & 0xF
    nib[:, 1::2] = codes >> 4
    return elem[nib] * np.repeat(scale[scales], NV_BLOCK, axis=1) * float(np.float32(tensor_scale))

