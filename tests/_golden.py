"""Readers for the hand-worked fixtures under tests/golden/."""

from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if line:
                yield line


def e4m3_cases():
    out = []
    for line in _lines("e4m3_ocp.txt"):
        code, val = line.split()
        out.append((int(code, 16), float(val)))
    return out


def resolve_case():
    d = {"block_table": {}, "topk": {}, "slots": {}}
    for line in _lines("resolve_p4.txt"):
        key, rest = line.split(None, 1)
        if ":" in rest:
            idx, vals = rest.split(":", 1)
            d[key][int(idx)] = [int(v) for v in vals.split()]
        else:
            vals = [int(v) for v in rest.split()]
            d[key] = vals[0] if len(vals) == 1 and key in ("page_size", "num_pages", "error") else vals
    n_bt, n_t = len(d["block_table"]), len(d["topk"])
    return dict(
        page_size=d["page_size"], num_pages=d["num_pages"], error=d["error"],
        block_table=np.array([d["block_table"][i] for i in range(n_bt)], np.int32),
        seq_lens=np.array(d["seq_lens"], np.int32), req_of_token=np.array(d["req_of_token"], np.int32),
        topk_len=np.array(d["topk_len"], np.int32),
        topk=np.array([d["topk"][i] for i in range(n_t)], np.int32),
        slots=np.array([d["slots"][i] for i in range(n_t)], np.int64),
    )


def union_cases():
    cases, cur = [], None
    for line in _lines("union_small.txt"):
        tok = line.split()
        if tok[0] == "case":
            cur = {"name": tok[1], "rows": [], "lens_rows": [], "groups": {}}
        elif tok[0] == "G":
            cur["G"], cur["K"], cur["num_slots"] = int(tok[1]), int(tok[3]), int(tok[5])
        elif tok[0] == "row":
            body, ln = line[4:].split(":")
            cur["rows"].append([int(v) for v in body.split()])
            cur["lens_rows"].append(int(ln))
        elif tok[0] == "group":
            g, lens = int(tok[1]), int(tok[3])
            pairs = [tuple(int(x) for x in p.split(":")) for p in tok[5:]]
            cur["groups"][g] = (lens, pairs)
        elif tok[0] == "end":
            cases.append(cur)
    return cases


def encode(mask: int, slot: int) -> int:
    """(mask << 24) | slot as a signed int32 value."""
    return int(np.array([(mask << 24) | slot], np.uint32).view(np.int32)[0])


def topk_cases():
    """Hand-worked top-k selections: dicts with K, scores (float32), len (int or None), expect."""
    cases, cur = [], None
    for line in _lines("topk_small.txt"):
        tok = line.split()
        if tok[0] == "case":
            cur = {"name": tok[1]}
        elif tok[0] == "K":
            cur["K"] = int(tok[1])
        elif tok[0] == "scores":
            cur["scores"] = np.array([float(v) for v in tok[1:]], np.float32)
        elif tok[0] == "len":
            cur["len"] = None if tok[1] == "all" else int(tok[1])
        elif tok[0] == "expect":
            cur["expect"] = np.array([int(v) for v in tok[1:]], np.int32)
        elif tok[0] == "end":
            cases.append(cur)
    return cases
