"""Reader for the hand-assembled Q4_K block fixtures in q4k_blocks.txt."""
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def load_blocks():
    """List of dicts: name, d_bits, dmin_bits, sc[8], m[8], block (144 uint8)."""
    out, cur = [], {}
    with open(os.path.join(HERE, "q4k_blocks.txt")) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                if cur:
                    out.append(cur)
                    cur = {}
                continue
            key, val = line.split(":", 1)
            val = val.strip()
            if key == "name":
                cur["name"] = val
            elif key in ("d_bits", "dmin_bits"):
                cur[key] = int(val, 16)
            elif key in ("sc", "m"):
                cur[key] = [int(v) for v in val.split()]
            elif key == "header":
                hdr = bytes(int(v, 16) for v in val.split())
                assert len(hdr) == 16
                cur["block"] = np.frombuffer(hdr + bytes(range(128)), dtype=np.uint8).copy()
    if cur:
        out.append(cur)
    return out


def fixture_codes():
    """q(s, l) for the fixtures' qs = 0x00..0x7F, from the rule stated in the file."""
    q = np.zeros((8, 32), dtype=np.int64)
    for s in range(8):
        g = s // 2
        for l in range(32):
            q[s, l] = (l % 16) if s % 2 == 0 else (2 * g + l // 16)
    return q
