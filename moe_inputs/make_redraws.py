"""Write the gap-redraw maps of the synthetic workloads.

For every (layer, step) of a workload, any token whose k-th and (k+1)-th
router logits (fp64, bias included) differ by less than 1e-3 gets its x row
redrawn from its own seeded stream until the gap is at least 1e-3.  The map
{(layer, step, token): draw index} is stored as JSON under
``moe_inputs/redraws/``.  The logits come from the CPU oracle only.

    python -m moe_inputs.make_redraws [workload ...]
"""
import json
import os
import sys

import numpy as np

from moe_inputs import CONFIGS, gen
from oracle import moe_oracle as O

GAP = 1e-3
# decode streams are longer than the 32-step parity trace so that benchmark
# runs with many steps still see gap-filtered tokens
STEPS_COVERED = {"tiny": 1, "decode": 1024, "batched_decode": 64, "prefill": 1, "long_prefill": 1}


def redraw_map(cfg, steps):
    entries = []
    for layer in range(cfg.n_layers):
        wr = gen.w_router(cfg, layer)
        for step in range(steps):
            b = gen.bias(cfg, layer, step)
            x = gen.x_bits(cfg, layer, step, redraws={})
            gaps = O.topk_gap(O.router_logits(gen.bf16_bits_to_f64(x), wr, b), cfg.k)
            for t in np.nonzero(gaps < GAP)[0]:
                r = 0
                while True:
                    r += 1
                    row = gen.x_row_redraw(cfg, layer, step, int(t), r)
                    g = O.topk_gap(O.router_logits(gen.bf16_bits_to_f64(row[None, :]), wr, b), cfg.k)[0]
                    if g >= GAP:
                        break
                entries.append([layer, step, int(t), r])
    return entries


def main(names):
    for name in names:
        cfg = CONFIGS[name]
        steps = STEPS_COVERED[name]
        entries = redraw_map(cfg, steps)
        doc = {"workload": name, "gap": GAP, "steps_covered": steps,
               "tokens_checked": cfg.n_layers * steps * cfg.T, "entries": entries}
        path = os.path.join(gen.REDRAW_DIR, f"{name}.json")
        with open(path, "w") as f:
            json.dump(doc, f, separators=(",", ":"))
            f.write("\n")
        print(f"{name}: {len(entries)} redraws over {doc['tokens_checked']} tokens -> {path}")


if __name__ == "__main__":
    main(sys.argv[1:] or list(CONFIGS))
