"""Readers for the hand-worked fixtures under tests/golden/."""
import os
import struct

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [part.strip() for part in line.split("|")]


def i32_cases():
    for inp, k, exp in _lines("topk_i32_hand.txt"):
        yield (np.array([int(v) for v in inp.split()], dtype=np.int32), int(k),
               np.array([int(v) for v in exp.split()], dtype=np.int32))


def rows_cases():
    for inp, k, idx, vals in _lines("topk_rows_hand.txt"):
        yield (np.array([float(v) for v in inp.split()], dtype=np.float32), int(k),
               np.array([int(v) for v in idx.split()], dtype=np.int32),
               np.array([float(v) for v in vals.split()], dtype=np.float32))


def reduce_cases():
    for dtype, op, inp, exp in _lines("reduce_hand.txt"):
        if dtype == "i32":
            yield dtype, op, np.array([int(v) for v in inp.split()], dtype=np.int32), int(exp)
        else:
            yield dtype, op, np.array([float(v) for v in inp.split()], dtype=np.float32), float(exp)


def items_cases():
    for sc, it, kp, k, es, ei, cnt in _lines("topk_items_hand.txt"):
        yield (np.array([float(v) for v in sc.split()], dtype=np.float32),
               None if it == "-" else np.array([int(v) for v in it.split()], dtype=np.int64),
               None if kp == "-" else np.array([int(v) for v in kp.split()], dtype=np.uint8), int(k),
               np.array([float(v) for v in es.split()], dtype=np.float32),
               np.array([int(v) for v in ei.split()], dtype=np.int64), int(cnt))


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def f32_from_bits(u):
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


def u32_cases():
    for inp, k, exp in _lines("topk_u32_hand.txt"):
        yield (np.array([int(v) for v in inp.split()], dtype=np.uint32), int(k),
               np.array([int(v) for v in exp.split()], dtype=np.uint32))


def f32_cases():
    """(input patterns, k, expected patterns), all uint32 bit patterns."""
    for inp, k, exp in _lines("topk_f32_hand.txt"):
        yield (np.array([int(v, 16) for v in inp.split()], dtype=np.uint32), int(k),
               np.array([int(v, 16) for v in exp.split()], dtype=np.uint32))
