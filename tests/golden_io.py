"""Readers for the hand-written fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_stream_fixture(name="stream64.txt"):
    """Returns (elements uint16, lut bytes, stream bytes) of a stream fixture."""
    n = total = None
    lut = b""
    elems = []
    nonzero = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = line.split(":", 1)
            key = key.strip()
            if key == "n":
                n = int(val)
            elif key == "total_bytes":
                total = int(val)
            elif key == "lut":
                lut = bytes(int(t, 16) for t in val.split())
            elif key == "elements":
                elems += [int(t, 16) for t in val.split()]
            elif key.startswith("bytes @"):
                off = int(key.split("@")[1])
                for i, t in enumerate(val.split()):
                    nonzero[off + i] = int(t, 16)
    stream = bytearray(total)
    for off, b in nonzero.items():
        stream[off] = b
    x = np.array(elems, dtype=np.uint16)
    assert x.size == n
    return x, lut, bytes(stream)
