"""Write synth_first_values.json: the first six raw values (fp32 bit patterns
or bf16 bit patterns) of every workload tensor, as the generator defines them.
Used only as a drift check of the generator; it calls no product code."""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from synth import workloads as W  # noqa: E402


def main():
    out = {}
    for w in W.ALL:
        out[w.name] = {}
        for t in w.tensors:
            rows = 1 if (w.chain != "add_relu_scale" and not t.per_column) else None
            a = w.generate(t, rows=rows).reshape(-1)[:6]
            vals = a if a.dtype == np.uint16 else a.view(np.uint32)
            out[w.name][t.name] = [int(v) for v in vals]
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "synth_first_values.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(path)


if __name__ == "__main__":
    main()
