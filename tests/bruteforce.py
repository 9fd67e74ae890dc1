"""Independent brute-force evaluation of the layer for tiny inputs (test helper).

Written separately from the oracle, in a different shape: plain Python floats,
exactly rounded sums (math.fsum), exact bf16 rounding through fractions.Fraction,
and a DENSE evaluation -- every token goes through every expert and the routing
only enters as a mask times weight, so the oracle's expert grouping, permutation
and top-k gather are not reused.
"""
from __future__ import annotations

import math
from fractions import Fraction


def bf16_exact(x: float) -> float:
    """Nearest bfloat16 to x (ties to even), via exact rational arithmetic."""
    if x != x or math.isinf(x) or x == 0.0:
        return x
    _, e = math.frexp(x)
    e = max(e, -125)
    quantum = Fraction(2) ** (e - 8)
    return float(round(Fraction(x) / quantum) * quantum)


def dot(a, b) -> float:
    return math.fsum(float(x) * float(y) for x, y in zip(a, b))


def sigmoid(z: float) -> float:
    return 1.0 / (1.0 + math.exp(-z)) if z >= 0 else math.exp(z) / (1.0 + math.exp(z))


def topk_bruteforce(keys, k):
    """Ids of the k largest keys, larger first, lower id first among equal keys."""
    return sorted(range(len(keys)), key=lambda e: (-keys[e], e))[:k]


def dense_layer(x, logits, w1, w2, top_k, method, bias=None, rsf=1.0, A_gu=None, B_gu=None,
                A_dn=None, B_dn=None, slot_idx=None, ranks=(), scalings=(), keys_fn=None, shared_outer=False,
                quant=None):
    """Dense evaluation on nested lists.  `keys_fn(logit_row)` gives the DeepSeekV3
    selection keys (the float32 key definition is pinned separately).  `quant(row)`, if
    given, is applied to the two base GEMMs' inputs (the FP8 path)."""
    T, H = len(x), len(x[0])
    E = len(w1)
    I = len(w1[0]) // 2
    out = []
    ids_all, w_all = [], []
    for t in range(T):
        row = [(-math.inf if v != v else float(v)) for v in logits[t]]
        if method == 0:
            ids = topk_bruteforce(row, top_k)
            m = max(row[e] for e in ids)
            ex = [math.exp(row[e] - m) for e in ids]
            tot = math.fsum(ex)
            wts = [v / tot for v in ex]
        else:
            keys, scores = keys_fn(row)
            ids = topk_bruteforce(keys, top_k)
            tot = math.fsum(scores[e] for e in ids)
            wts = [scores[e] / tot * rsf for e in ids]
        ids_all.append(ids)
        w_all.append(wts)
        weight_of = {e: wv for e, wv in zip(ids, wts)}
        s = -1 if slot_idx is None else int(slot_idx[t])
        out.append(_dense_token(x[t], range(E), weight_of, w1, w2, s, A_gu, B_gu, A_dn, B_dn, ranks, scalings,
                                shared_outer=shared_outer, quant=quant))
    return out, ids_all, w_all


def _dense_token(xt, experts, weight_of, w1, w2, s, A_gu, B_gu, A_dn, B_dn, ranks, scalings, gid=lambda e: e,
                 shared_outer=False, quant=None):
    """One token through every expert e in `experts` (weight index e, routing id gid(e)),
    masked by the routing: bf16(fsum over e of mask * w * (y + dd)).  shared_outer: A_gu
    and B_dn hold one weight set per slot (index 0) used by every expert."""
    H = len(xt)
    I = len(w1[0]) // 2
    use_lora = (s >= 0 and s < len(ranks) and ranks[s] > 0 and scalings[s] != 0.0)
    terms = []
    xg = xt if quant is None else quant(xt)      # the gate_up GEMM's input
    for e in experts:                            # dense: every expert
        g = [bf16_exact(dot(w1[e][n], xg)) for n in range(2 * I)]
        if use_lora:
            r, sc = ranks[s], scalings[s]
            u = [dot(A_gu[s][0 if shared_outer else e][q], xt) for q in range(r)]
            d = [bf16_exact(sc * dot([B_gu[s][e][n][q] for q in range(r)], u)) for n in range(2 * I)]
        else:
            d = [0.0] * (2 * I)
        a = []
        for i in range(I):
            zg = g[i] + d[i]
            a.append(bf16_exact(zg * sigmoid(zg) * (g[I + i] + d[I + i])))
        ag = a if quant is None else quant(a)    # the down GEMM's input
        y = [dot(w2[e][h], ag) for h in range(H)]
        if use_lora:
            v = [dot(A_dn[s][e][q], a) for q in range(r)]
            dd = [sc * dot([B_dn[s][0 if shared_outer else e][h][q] for q in range(r)], v) for h in range(H)]
        else:
            dd = [0.0] * H
        mask = 1.0 if gid(e) in weight_of else 0.0
        wt = weight_of.get(gid(e), 0.0)
        terms.append([mask * wt * (y[h] + dd[h]) for h in range(H)])
    return [bf16_exact(math.fsum(terms[i][h] for i in range(len(terms)))) for h in range(H)]


def dense_layer_routed(x, ids_all, w_all, local_offset, w1, w2, A_gu=None, B_gu=None, A_dn=None, B_dn=None,
                       slot_idx=None, ranks=(), scalings=()):
    """Dense evaluation with the routing given (global ids and weights per token) and only
    the local experts present: weight index e has global id local_offset + e; a routed
    pair whose expert is not local contributes nothing."""
    out = []
    for t in range(len(x)):
        weight_of = {int(e): float(wv) for e, wv in zip(ids_all[t], w_all[t])}
        s = -1 if slot_idx is None else int(slot_idx[t])
        out.append(_dense_token(x[t], range(len(w1)), weight_of, w1, w2, s, A_gu, B_gu, A_dn, B_dn, ranks,
                                scalings, gid=lambda e: local_offset + e))
    return out



def fake_quant_torch(row, group=128):
    """FP8 group quantisation of one row, built on torch's float8_e4m3fn conversion
    instead of the oracle's own e4m3 rounding: per group of `group` values,
    s = max(amax, 1e-10) / 448 and q = fp8(clamp(v / s, +-448)) in float32, returned
    dequantised (q * s, exact in Python floats)."""
    import torch
    out = []
    for g0 in range(0, len(row), group):
        t = torch.tensor(row[g0:g0 + group], dtype=torch.float32)
        amax = t.abs().max()
        s = torch.maximum(amax, torch.tensor(1e-10, dtype=torch.float32)) / torch.tensor(448.0)
        q = (t / s).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).to(torch.float64)
        out.extend(float(v) * float(s) for v in q)
    return out


def dequant_weight_torch(codes, scales, block=128):
    """Nested-list weight [N][K] from uint8 codes [N, K] and block scales, decoded by
    torch's float8_e4m3fn view (not the oracle's decoder)."""
    import torch
    c = torch.as_tensor(codes, dtype=torch.uint8)
    w = c.view(torch.float8_e4m3fn).to(torch.float64)
    s = torch.as_tensor(scales, dtype=torch.float64)
    N, K = w.shape
    return [[float(w[n, k]) * float(s[n // block, k // block]) for k in range(K)] for n in range(N)]


E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # the format's magnitudes, code order


def e2m1_nearest(y: float) -> float:
    """Nearest e2m1 value by exhaustive search over the 8 magnitudes (ties to the code
    with the even last bit), saturating at 6."""
    a = min(abs(y), 6.0)
    best = min(range(8), key=lambda c: (abs(a - E2M1_TABLE[c]), c & 1))
    return math.copysign(E2M1_TABLE[best], y)


def fake_quant_nvfp4(row, block=16):
    """NVFP4 quantisation of one row with a per-row tensor scale, built on torch's float8
    conversion for the block scales and an exhaustive nearest search for the codes
    (instead of the oracle's own roundings); returns the dequantised values."""
    import torch
    t = torch.tensor(row, dtype=torch.float32)
    g = torch.maximum(t.abs().max(), torch.tensor(1e-10, dtype=torch.float32)) / torch.tensor(2688.0)
    six_g = torch.tensor(6.0) * g
    out = []
    for b0 in range(0, len(row), block):
        blk = t[b0:b0 + block]
        sb = (blk.abs().max() / six_g).to(torch.float8_e4m3fn).to(torch.float32)
        eff = sb * g
        for v in blk:
            if float(eff) == 0.0:
                out.append(0.0)
            else:
                y = float((v / eff).to(torch.float32))
                out.append(e2m1_nearest(y) * float(sb) * float(g))
    return out


def dequant_weight_nvfp4_bruteforce(packed, scale_codes, gscale, block=16):
    """Nested-list weight [N][K] decoded nibble by nibble from the table and the block
    scales by torch's float8_e4m3fn view."""
    import torch
    p = torch.as_tensor(packed, dtype=torch.uint8)
    s = torch.as_tensor(scale_codes, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    N, K2 = p.shape
    gs = float(torch.as_tensor(gscale, dtype=torch.float32))
    rows = []
    for n in range(N):
        r = []
        for i in range(K2):
            byte = int(p[n, i])
            for k, c in ((2 * i, byte & 0xF), (2 * i + 1, byte >> 4)):
                val = E2M1_TABLE[c & 7] * (-1.0 if c & 8 else 1.0)
                r.append(val * float(s[n, k // block]) * gs)
        rows.append(r)
    return rows
