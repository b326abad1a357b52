"""Load the hand-derived fixtures of hand_derived.json as numpy arrays."""
import json
import os
import struct

import numpy as np

from decode_q1_gemv_gb300.synth import assemble_blocks

_HERE = os.path.dirname(os.path.abspath(__file__))


def _f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def load_cases():
    with open(os.path.join(_HERE, "hand_derived.json")) as f:
        spec = json.load(f)
    out = []
    for c in spec["cases"]:
        n = c["n"]
        nb = n // 128
        d0 = np.array([int(h, 16) for h in c["d0"]], dtype=np.uint16).reshape(1, nb)
        fill = {"all0": 0x00, "all1": 0xFF}[c["bits"]]
        signs = np.full((1, nb, 16), fill, dtype=np.uint8)
        blocks = assemble_blocks(d0, signs)
        q = np.full(n, c["q_fill"], dtype=np.int16)
        for key, val in c["q_set"].items():
            if "-" in key:
                a, b = (int(t) for t in key.split("-"))
                q[a:b + 1] = val
            else:
                q[int(key)] = val
        d1 = np.array([int(h, 16) for h in c["d1"]], dtype=np.uint16)
        expected = np.float32(c["expected"])
        if "expected_hex" in c:
            assert _f32_bits(float(expected)) == int(c["expected_hex"], 16), c["name"]
        out.append((c["name"], blocks, q.astype(np.int8), d1, expected))
    return out
