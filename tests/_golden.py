"""Materialise the hand-derived cases of tests/golden/closed_form.json as arrays.

Input construction only: places the listed rows in their pages (pool layout
[num_pages][Hkv][P][d], NaN elsewhere) and builds the per-sequence page table
and the ubatch (tok_seq, tok_pos, q).  The expected outputs come from the
file, where each is derived by hand.
"""
import json
import math
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
NAN16 = np.uint16(0x7E00)


def _vec(sparse, d):
    x = np.zeros(d, np.float32)
    for i, val in sparse:
        x[int(i)] = val
    return x


def _rows(spec, L, d):
    out = np.zeros((L, d), np.float32)
    if "linear" in spec:
        lin = spec["linear"]
        out[:, lin["dim"]] = lin["start"] + lin["step"] * np.arange(L)
    for j, sparse in spec.get("rows", {}).items():
        out[int(j)] = _vec(sparse, d)
    return out


def load_cases():
    with open(os.path.join(HERE, "golden", "closed_form.json")) as f:
        return json.load(f)["cases"]


def materialise(case):
    P, Hq, Hkv, d, N = case["P"], case["Hq"], case["Hkv"], case["d"], case["num_pages"]
    scale = math.log(3.0) if case["scale"] == "ln3" else float(case["scale"])
    kp = np.full((N, Hkv, P, d), NAN16, np.uint16)
    vp = np.full((N, Hkv, P, d), NAN16, np.uint16)
    max_pages = max(len(s["pages"]) for s in case["seqs"])
    spt = np.full((len(case["seqs"]), max_pages), -1, np.int32)
    for si, s in enumerate(case["seqs"]):
        L = s["len"]
        spt[si, :len(s["pages"])] = s["pages"]
        for h in range(Hkv):
            ks = s["k_heads"][h] if "k_heads" in s else s["k"]
            vs = s["v_heads"][h] if "v_heads" in s else s["v"]
            K = _rows(ks, L, d).astype(np.float16).view(np.uint16)
            V = _rows(vs, L, d).astype(np.float16).view(np.uint16)
            for j in range(L):
                page = s["pages"][j // P]
                kp[page, h, j % P] = K[j]
                vp[page, h, j % P] = V[j]
    T = len(case["tokens"])
    tok_seq = np.array([t["seq"] for t in case["tokens"]], np.int32)
    tok_pos = np.array([t["pos"] for t in case["tokens"]], np.int32)
    q = np.zeros((T, Hq, d), np.float32)
    for i, t in enumerate(case["tokens"]):
        for h in range(Hq):
            q[i, h] = _vec(t["q_heads"][h] if "q_heads" in t else t["q"], d)
    q = q.astype(np.float16).view(np.uint16)
    expected = np.zeros((T, Hq, d), np.float64)
    for i, per_tok in enumerate(case["expected"]):
        for h in range(Hq):
            sparse = per_tok[h] if len(per_tok) == Hq else per_tok[0]
            for idx, val in sparse:
                expected[i, h, int(idx)] = val
    return dict(P=P, Hq=Hq, Hkv=Hkv, d=d, num_pages=N, scale=scale, k_pages=kp, v_pages=vp,
                seq_page_table=spt, tok_seq=tok_seq, tok_pos=tok_pos, q=q, expected=expected)
