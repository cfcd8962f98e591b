"""Readers for the hand-derived fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def path(name):
    return os.path.join(GOLDEN, name)


def _lines(name):
    with open(path(name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if line:
                yield line


def f32(tok):
    """A float32 from a decimal literal or a 0x bit pattern."""
    if tok.lower().startswith("0x"):
        return np.array([int(tok, 16)], dtype=np.uint32).view(np.float32)[0]
    return np.float32(float(tok))


def f32_bits(tok):
    return int(np.array([f32(tok)], dtype=np.float32).view(np.uint32)[0])


def chunk_sizes():
    for line in _lines("dynamic_chunk_sizes.txt"):
        n, eb, count, piece = (int(x) for x in line.split())
        yield n, eb, count, piece


def keyed_cases(name):
    """'case <name>' blocks of 'key values...' lines -> list of (name, dict)."""
    cases, cur = [], None
    for line in _lines(name):
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = (rest.strip(), {})
            cases.append(cur)
        else:
            if cur is None:
                cur = ("", {})
                cases.append(cur)
            cur[1][key] = rest.split()
    return cases


def bucket_cases():
    for line in _lines("bucket_assignment.txt"):
        eb, tensors, buckets = (p.strip() for p in line.split("|"))
        yield int(eb), [int(x) for x in tensors.split()], [int(x) for x in buckets.split()]
