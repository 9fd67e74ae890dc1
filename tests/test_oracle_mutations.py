"""Planted mistakes: each mutant copy of the oracle must fail at least one pin.

A mutant is the oracle's source with one plausible slip substituted (a swapped
operand, a dropped term, a wrong sign or index, a different tie rule), executed as
a separate module on the CPU.  If some mutant passed every check below, the pins
would not be strong enough to vouch for the oracle.
"""
import json
import os
import types

import numpy as np
import pytest
import torch

import bruteforce as bf
from routed_moe_expert_gb300 import workloads as wl

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "moe_lora_oracle.py")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_example.json")

MUTATIONS = [
    ("gate/up swapped", "silu(g[:, :I] + d[:, :I]) * (g[:, I:] + d[:, I:])",
     "silu(g[:, I:] + d[:, I:]) * (g[:, :I] + d[:, :I])"),
    ("delta dropped from gate", "silu(g[:, :I] + d[:, :I])", "silu(g[:, :I])"),
    ("scaling dropped", "d[m] = round_bf16(sc * (u @ B.T))", "d[m] = round_bf16(u @ B.T)"),
    ("down delta dropped", "res[(int(ts[i]), int(js[i]))] = (y[i] + dd[i], a[i])",
     "res[(int(ts[i]), int(js[i]))] = (y[i], a[i])"),
    ("routing weight dropped", "acc = acc + w[t, j] * rows[(int(t), j)][0]", "acc = acc + rows[(int(t), j)][0]"),
    ("down weight of the wrong expert", "W2 = _f64(w2[e])", "W2 = _f64(w2[(e + 1) % len(w2)])"),
    ("silu sign", "return z / (1.0 + np.exp(-z))", "return z / (1.0 + np.exp(z))"),
    ("rank tail read", "A = _f64(lora_A_gu[s, eo(e)])[:r]", "A = _f64(lora_A_gu[s, eo(e)])"),
    ("tie to higher id", "order = np.argsort(-keys, axis=1, kind=\"stable\")",
     "order = (keys.shape[1] - 1 - np.argsort(-keys[:, ::-1], axis=1, kind=\"stable\"))"),
    ("softmax over all experts, not renormalised", "w = ex / ex.sum(axis=1, keepdims=True)",
     "w = ex / np.exp(logit.astype(np.float64) - sel[:, :1]).sum(axis=1, keepdims=True)"),
    ("deepseek bias ignored", "key = (s + bias[None, :]).astype(np.float32)", "key = s"),
    ("deepseek rsf dropped", "* float(routed_scaling_factor)", "* 1.0"),
    ("bf16 truncation", "q = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)",
     "q = np.ldexp(np.trunc(np.ldexp(x, 8 - e)), e - 8)"),
    ("perm descending in expert", "perm = np.argsort(flat, kind=\"stable\").astype(np.int32)",
     "perm = (flat.size - 1 - np.argsort(flat[::-1], kind=\"stable\")).astype(np.int32)"),
    ("no-adapter token gets slot 0", "slots = np.full(T, -1, dtype=np.int64) if slot_idx is None else np.asarray(slot_idx, dtype=np.int64)\n    inter",
     "slots = np.maximum(np.asarray(slot_idx, dtype=np.int64), 0)\n    inter"),
    # the externally routed entry
    ("packed weight read from the id half", "w = ((u & 0xFFFF) << 16)", "w = ((u >> 16) << 16)"),
    ("packed weight truncated", "w = round_bf16(np.asarray(topk_weights, dtype=np.float64)).astype(np.float32)",
     "w = np.asarray(topk_weights, dtype=np.float32)"),
    ("experts below the local range kept", "local = (lid >= 0) & (lid < E_loc)", "local = lid < E_loc"),
    # shared-outer LoRA
    ("shared-outer weights read per expert", "eo = (lambda e: 0) if shared_outer else (lambda e: e)",
     "eo = lambda e: e"),
    ("shared-outer down LoRA from the per-expert weights", "B = _f64(lora_B_dn[s, eo(e)])[:, :r]",
     "B = _f64(lora_B_dn[s, 0])[:, :r]"),
]


def _mutant(old, new):
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


def np_(t):
    return None if t is None else t.float().numpy() if t.dtype == torch.bfloat16 else t.numpy()


def _dense_check(orc, seed):
    cfg = wl.LayerConfig("m", T=5, H=16, I=8, E=4, top_k=2, method=seed % 2,
                         ranks=(2, 4), scalings=(2.0, 0.5), slot_mode="uniform_none10",
                         bias_std=0.1, rsf=2.0)
    inp = wl.make_inputs(cfg, seed=seed)
    bias = np_(inp["correction_bias"])
    res = orc.moe_lora_forward(np_(inp["hidden"]), np_(inp["router_logits"]), np_(inp["w1"]),
                               np_(inp["w2"]), cfg.top_k, cfg.method, bias, cfg.rsf,
                               np_(inp["lora_A_gu"]), np_(inp["lora_B_gu"]), np_(inp["lora_A_dn"]),
                               np_(inp["lora_B_dn"]), inp["slot_idx"].numpy(), inp["ranks"], inp["scalings"])
    from oracle import moe_lora_oracle as good

    def keys_fn(row):
        s = good.sigmoid_f32(np.asarray(row, np.float32))
        return list((s + bias).astype(np.float32).astype(np.float64)), list(s.astype(np.float64))

    L = lambda a: None if a is None else np.asarray(a, np.float64).tolist()
    dense, ids, w = bf.dense_layer(L(np_(inp["hidden"])), L(np_(inp["router_logits"])), L(np_(inp["w1"])),
                                   L(np_(inp["w2"])), cfg.top_k, cfg.method, rsf=cfg.rsf,
                                   A_gu=L(np_(inp["lora_A_gu"])), B_gu=L(np_(inp["lora_B_gu"])),
                                   A_dn=L(np_(inp["lora_A_dn"])), B_dn=L(np_(inp["lora_B_dn"])),
                                   slot_idx=inp["slot_idx"].tolist(), ranks=inp["ranks"],
                                   scalings=inp["scalings"], keys_fn=keys_fn)
    ok = res["topk_ids"].tolist() == ids and np.array_equal(res["out"], np.array(dense))
    ok = ok and np.allclose(res["topk_weights"], np.array(w), rtol=1e-12)
    # permutation invariant: ascending expanded index inside each expert
    off, perm = res["expert_offsets"], res["perm"]
    ok = ok and all((np.diff(perm[off[e]:off[e + 1]]) > 0).all() for e in range(cfg.E))
    return ok


def _hand_check(orc):
    G = json.load(open(GOLDEN))
    for case in G["cases"]:
        res = orc.moe_lora_forward(
            np.array(G["hidden"], float), np.array(case["logits"], float), np.array(G["w1"], float),
            np.array(G["w2"], float), case["top_k"], case["method"],
            correction_bias=np.array(case.get("bias", [0, 0]), np.float32),
            routed_scaling_factor=case.get("rsf", 1.0),
            lora_A_gu=np.array(G["lora_A_gu"], float), lora_B_gu=np.array(G["lora_B_gu"], float),
            lora_A_dn=np.array(G["lora_A_dn"], float), lora_B_dn=np.array(G["lora_B_dn"], float),
            slot_idx=np.array(case.get("slot_idx", [0, 0])), ranks=G["ranks"], scalings=G["scalings"],
            lora_off=not case["lora"])
        if res["topk_ids"].tolist() != case["topk_ids"] or not np.array_equal(res["out"], np.array(case["out"], float)):
            return False
    return True


def _routed_check(orc, seed):
    cfg = wl.LayerConfig("mr", T=5, H=16, I=8, E=3, top_k=2, ranks=(2, 4), scalings=(2.0, 0.5),
                         slot_mode="uniform_none10")
    inp = wl.make_inputs(cfg, seed=seed)
    ids, w = wl.make_routing(5, 6, 2, seed=seed)
    w = w.numpy().astype(np.float64) * 0.7 + 0.013      # not bf16-exact: packing must round
    from oracle import moe_lora_oracle as good
    packed = orc.pack_topk(ids.numpy(), w)
    if not np.array_equal(packed, good.pack_topk(ids.numpy(), w)):
        return False
    lora = dict(lora_A_gu=np_(inp["lora_A_gu"]), lora_B_gu=np_(inp["lora_B_gu"]),
                lora_A_dn=np_(inp["lora_A_dn"]), lora_B_dn=np_(inp["lora_B_dn"]),
                slot_idx=inp["slot_idx"].numpy(), ranks=inp["ranks"], scalings=inp["scalings"])
    res = orc.moe_lora_forward_routed(np_(inp["hidden"]), packed, np_(inp["w1"]), np_(inp["w2"]), 2,
                                      num_experts=6, local_expert_offset=2, **lora)
    L = lambda a: None if a is None else np.asarray(a, np.float64).tolist()
    wb = good.round_bf16(w)
    dense = bf.dense_layer_routed(L(np_(inp["hidden"])), ids.tolist(), wb.tolist(), 2, L(np_(inp["w1"])),
                                  L(np_(inp["w2"])), A_gu=L(lora["lora_A_gu"]), B_gu=L(lora["lora_B_gu"]),
                                  A_dn=L(lora["lora_A_dn"]), B_dn=L(lora["lora_B_dn"]),
                                  slot_idx=lora["slot_idx"].tolist(), ranks=lora["ranks"], scalings=lora["scalings"])
    return np.array_equal(res["out"], np.array(dense))


def _shared_check(orc, seed):
    cfg = wl.LayerConfig("ms", T=5, H=16, I=8, E=3, top_k=2, ranks=(2, 4), scalings=(2.0, 0.5),
                         slot_mode="uniform_none10", shared_outer=(seed % 2 == 0))
    inp = wl.make_inputs(cfg, seed=seed)
    L = lambda a: None if a is None else np.asarray(a, np.float64).tolist()
    lora = dict(lora_A_gu=np_(inp["lora_A_gu"]), lora_B_gu=np_(inp["lora_B_gu"]),
                lora_A_dn=np_(inp["lora_A_dn"]), lora_B_dn=np_(inp["lora_B_dn"]))
    res = orc.moe_lora_forward(np_(inp["hidden"]), np_(inp["router_logits"]), np_(inp["w1"]), np_(inp["w2"]), 2,
                               slot_idx=inp["slot_idx"].numpy(), ranks=inp["ranks"], scalings=inp["scalings"],
                               shared_outer=cfg.shared_outer, **lora)
    dense, _, _ = bf.dense_layer(L(np_(inp["hidden"])), L(np_(inp["router_logits"])), L(np_(inp["w1"])),
                                 L(np_(inp["w2"])), 2, 0, A_gu=L(lora["lora_A_gu"]), B_gu=L(lora["lora_B_gu"]),
                                 A_dn=L(lora["lora_A_dn"]), B_dn=L(lora["lora_B_dn"]),
                                 slot_idx=inp["slot_idx"].tolist(), ranks=inp["ranks"], scalings=inp["scalings"],
                                 shared_outer=cfg.shared_outer)
    return np.array_equal(res["out"], np.array(dense))


def _bf16_check(orc):
    vals = np.random.default_rng(0).standard_normal(2000).astype(np.float32)
    return np.array_equal(orc.round_bf16(vals.astype(np.float64)),
                          torch.from_numpy(vals).to(torch.bfloat16).double().numpy())


def test_unmutated_oracle_passes_the_checks():
    from oracle import moe_lora_oracle as good
    assert all(_dense_check(good, s) for s in range(4))
    assert all(_routed_check(good, s) for s in range(2))
    assert all(_shared_check(good, s) for s in range(2))
    assert _hand_check(good) and _bf16_check(good)


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutant_is_caught(name, old, new):
    m = _mutant(old, new)
    results = []
    for check in (lambda: _bf16_check(m), lambda: _hand_check(m),
                  *[(lambda s=s: _dense_check(m, s)) for s in range(4)],
                  *[(lambda s=s: _routed_check(m, s)) for s in range(2)],
                  *[(lambda s=s: _shared_check(m, s)) for s in range(2)]):
        try:
            results.append(bool(check()))
        except Exception:
            results.append(False)
    assert not all(results), f"mutant '{name}' passed every pin"


# FP8 block-scale path: each mutant must fail the e4m3 pins or the FP8 dense brute force
FP8_MUTATIONS = [
    ("e4m3 exponent bias 8", "(1.0 + m / 8.0) * np.exp2(ex - 7.0)", "(1.0 + m / 8.0) * np.exp2(ex - 8.0)"),
    ("e4m3 ties away from zero", "quantum = np.exp2(e - 3.0)      # 3 mantissa bits\n        q = np.rint(ax / quantum) * quantum",
     "quantum = np.exp2(e - 3.0)      # 3 mantissa bits\n        q = np.floor(ax / quantum + 0.5) * quantum"),
    ("e4m3 without saturation", "q = np.minimum(q, E4M3_MAX)", "q = q"),
    ("e4m3 without the subnormal step", "e = np.maximum(e - 1, -6)", "e = e - 1"),
    ("weight block scale transposed", "return w * sc[rows[:, None], cols[None, :]]",
     "return w * sc.T[rows[:, None] % sc.shape[1], cols[None, :] % sc.shape[0]]"),
    ("activation scale from the whole row", "amax = np.abs(g).max(axis=2)",
     "amax = np.repeat(np.abs(g).max(axis=(1, 2))[:, None], K // group, axis=1)"),
    ("scale without the 448", "s = (np.maximum(amax, FP8_EPS) / np.float32(E4M3_MAX)).astype(np.float32)",
     "s = np.maximum(amax, FP8_EPS).astype(np.float32)"),
    ("down GEMM input not quantised", "ag = a if act_quant is None else act_quant(a)", "ag = a"),
    ("gate_up LoRA shrink reads the quantised input", "u = xe[m] @ A.T", "u = xg[m] @ A.T"),
]


def _e4m3_check(orc):
    codes = np.arange(256)
    d = orc.e4m3_decode(codes)
    ref = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    if not (np.array_equal(np.isnan(d), np.isnan(ref)) and np.array_equal(d[~np.isnan(d)], ref[~np.isnan(ref)])):
        return False
    x = np.random.default_rng(0).uniform(-500, 500, 4000).astype(np.float32)
    x = np.concatenate([x, x * 1e-3]).astype(np.float32)
    ref = torch.from_numpy(x).clamp(-448, 448).to(torch.float8_e4m3fn).double().numpy()
    return np.array_equal(orc.round_e4m3(x.astype(np.float64)), ref)


def test_unmutated_oracle_passes_the_fp8_checks():
    from oracle import moe_lora_oracle as good
    from test_oracle_fp8 import fp8_dense_check
    assert _e4m3_check(good)
    assert all(fp8_dense_check(good, s) for s in range(2))


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name,old,new", FP8_MUTATIONS, ids=[m[0] for m in FP8_MUTATIONS])
def test_fp8_mutant_is_caught(name, old, new):
    from test_oracle_fp8 import fp8_dense_check
    m = _mutant(old, new)
    results = []
    for check in (lambda: _e4m3_check(m), *[(lambda s=s: fp8_dense_check(m, s)) for s in range(2)]):
        try:
            results.append(bool(check()))
        except Exception:
            results.append(False)
    assert not all(results), f"mutant '{name}' passed every FP8 pin"


# NVFP4 path: each mutant must fail the e2m1 pins or the NVFP4 dense brute force
NVFP4_MUTATIONS = [
    ("e2m1 exponent bias 0", "(1.0 + m / 2.0) * np.exp2(ex - 1.0)", "(1.0 + m / 2.0) * np.exp2(ex)"),
    ("e2m1 ties away from zero", "quantum = np.exp2(e - 1.0)       # 1 mantissa bit\n        q = np.rint(ax / quantum) * quantum",
     "quantum = np.exp2(e - 1.0)       # 1 mantissa bit\n        q = np.floor(ax / quantum + 0.5) * quantum"),
    ("e2m1 without saturation", "q = np.minimum(q, E2M1_MAX)", "q = q"),
    ("e2m1 without the subnormal step", "e = np.maximum(e - 1, 0)", "e = e - 1"),
    ("nibbles swapped", "out[..., 0::2] = b & 0xF\n    out[..., 1::2] = b >> 4",
     "out[..., 0::2] = b >> 4\n    out[..., 1::2] = b & 0xF"),
    ("block scale not rounded to e4m3",
     "sb = round_e4m3((amax_b / six_g[:, None]).astype(np.float32).astype(np.float64))",
     "sb = (amax_b / six_g[:, None]).astype(np.float64)"),
    ("token scale from the first block", "amax_t = np.abs(v32).max(axis=1)",
     "amax_t = np.abs(v32[:, :block]).max(axis=1)"),
    ("weight tensor scale dropped", "return w * np.repeat(sb, block, axis=1)[:, :K] * float(np.float32(global_scale))",
     "return w * np.repeat(sb, block, axis=1)[:, :K]"),
]


def _e2m1_check(orc):
    if orc.e2m1_decode(np.arange(16)).tolist() != bf.E2M1_TABLE + [-v for v in bf.E2M1_TABLE]:
        return False
    x = np.concatenate([np.random.default_rng(0).uniform(-8, 8, 2000), np.arange(-7, 7.25, 0.25)])
    if orc.round_e2m1(x).tolist() != [bf.e2m1_nearest(float(v)) for v in x]:
        return False
    return orc.unpack_nvfp4(np.array([[0x21]], dtype=np.uint8)).tolist() == [[1, 2]]


def test_unmutated_oracle_passes_the_nvfp4_checks():
    from oracle import moe_lora_oracle as good
    from test_oracle_nvfp4 import nvfp4_dense_check
    assert _e2m1_check(good)
    assert all(nvfp4_dense_check(good, s) for s in range(2))


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name,old,new", NVFP4_MUTATIONS, ids=[m[0] for m in NVFP4_MUTATIONS])
def test_nvfp4_mutant_is_caught(name, old, new):
    from test_oracle_nvfp4 import nvfp4_dense_check
    m = _mutant(old, new)
    results = []
    for check in (lambda: _e2m1_check(m), *[(lambda s=s: nvfp4_dense_check(m, s)) for s in range(2)]):
        try:
            results.append(bool(check()))
        except Exception:
            results.append(False)
    assert not all(results), f"mutant '{name}' passed every NVFP4 pin"
