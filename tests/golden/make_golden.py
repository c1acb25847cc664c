"""Write tests/golden/pattern_oracle.json from the float64 oracle.

Run from the repository root: ``python tests/golden/make_golden.py``.
It calls only the oracle and the formula-defined input pattern (no random
draws, no GPU), so the stored values are independent of the CUDA library.
The pages give no worked numeric example; this file is a regression fixture
for the oracle across machines and a fixed target for the GPU tests.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import gqa_paged_decode_oracle  # noqa: E402
from paged_kv_gqa_split_gb300.workloads import make_pattern_workload  # noqa: E402

HEADS = [0, 9, 18, 31]


def main():
    w = make_pattern_workload()
    o, lse = gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale)
    doc = {
        "source": "float64 oracle on paged_kv_gqa_split_gb300.workloads.make_pattern_workload()",
        "lens": w.lens,
        "lse": [[float(x) for x in row] for row in lse],
        "o_row_sums": [[float(o[b, h].sum()) for h in range(32)] for b in range(w.batch)],
        "o_rows": {f"{b},{h}": [float(x) for x in o[b, h]] for b in range(w.batch) for h in HEADS},
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "pattern_oracle.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=0)
    print("wrote", path)


if __name__ == "__main__":
    main()
