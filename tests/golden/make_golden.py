"""Writes tests/golden/synth_sha256.json: SHA-256 digests of the seeded
inputs of the small workloads, so that a change to the generator (which both
the oracle and the CUDA path consume) is caught.  Calls only the input
generator; no value here comes from the CUDA path."""
import hashlib
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
from exact_attention_40_gb300 import synth  # noqa: E402


def digests():
    out = {}
    q, k, v = synth.prefill_inputs(synth.PREFILL["tiny"])
    for name, a in (("tiny.q", q), ("tiny.k", k), ("tiny.v", v)):
        out[name] = hashlib.sha256(a.tobytes()).hexdigest()
    lens = synth.ctx_lengths(5, 64, 512, 8192)
    out["decode_paged.ctx_lens"] = hashlib.sha256(lens.tobytes()).hexdigest()
    table, nb = synth.paged_layout(lens, 16, 5)
    out["decode_paged.block_table"] = hashlib.sha256(table.tobytes()).hexdigest()
    out["decode_paged.num_blocks"] = int(nb)
    x, r, w = synth.norm_inputs(synth.NORM["rmsnorm_64x8192"])
    for name, a in (("rmsnorm_64x8192.x", x), ("rmsnorm_64x8192.residual", r),
                    ("rmsnorm_64x8192.weight", w)):
        out[name] = hashlib.sha256(a.tobytes()).hexdigest()
    return out


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "synth_sha256.json")
    with open(path, "w") as f:
        json.dump(digests(), f, indent=1, sort_keys=True)
        f.write("\n")
    print(path)
