"""Pins of the oracle's NVFP4 path (CPU).

The e2m1 decoder is checked against the format's value table, the rounding against an
exhaustive nearest search, the packing against hand-written bytes, and the quantiser
against closed forms, its error bound and an independent quantiser built on torch's
float8 conversion.  The weight decode is checked nibble by nibble, and the whole NVFP4
layer against the dense brute force of tests/bruteforce.py.
"""
import numpy as np
import pytest
import torch

import bruteforce as bf
from oracle import moe_lora_oracle as orc
from routed_moe_expert_gb300 import workloads as wl


def test_e2m1_decode_is_the_format_table():
    want = bf.E2M1_TABLE + [-v for v in bf.E2M1_TABLE]
    got = orc.e2m1_decode(np.arange(16))
    assert got.tolist() == want
    assert np.copysign(1.0, got[8]) == -1.0          # code 8 is -0


def test_round_e2m1_matches_exhaustive_search():
    rng = np.random.default_rng(0)
    grid = np.array(bf.E2M1_TABLE)
    mids = (grid[1:] + grid[:-1]) / 2                # ties: 0.25 -> 0, 0.75 -> 1, 5 -> 4, ...
    x = np.concatenate([grid, mids, -mids, rng.uniform(-8, 8, 4000), rng.uniform(-1, 1, 2000), [7.0, 100.0, -9.0]])
    got = orc.round_e2m1(x)
    want = np.array([bf.e2m1_nearest(float(v)) for v in x])
    assert np.array_equal(got, want)
    assert orc.round_e2m1(0.25) == 0.0 and orc.round_e2m1(0.75) == 1.0 and orc.round_e2m1(5.0) == 4.0
    assert orc.round_e2m1(2.5) == 2.0 and orc.round_e2m1(3.5) == 4.0 and orc.round_e2m1(6.5) == 6.0


def test_unpack_low_nibble_first():
    packed = np.array([[0x21, 0xF8]], dtype=np.uint8)
    assert orc.unpack_nvfp4(packed).tolist() == [[1, 2, 8, 15]]


def test_quant_act_nvfp4_closed_forms():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((4, 64)).astype(np.float32)
    q, sb, g = orc.quant_act_nvfp4(v)
    amax = np.abs(v).max(axis=1)
    assert np.array_equal(g, (np.maximum(amax, np.float32(1e-10)) / np.float32(2688.0)).astype(np.float32))
    for t in range(4):
        j = int(np.argmax(np.abs(v[t])))
        assert sb[t, j // 16] == 448.0 and abs(q[t, j]) == 6.0   # the token's largest value
    # a zero block inside a nonzero row: scale 0, codes 0; an all-zero row: codes 0
    v[0, 16:32] = 0.0
    v[1, :] = 0.0
    q, sb, g = orc.quant_act_nvfp4(v)
    assert sb[0, 1] == 0.0 and np.all(q[0, 16:32] == 0.0) and np.all(q[1] == 0.0)


def test_quant_act_nvfp4_error_bound():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal((32, 128)) * np.exp(rng.uniform(-5, 5, (32, 1)))).astype(np.float32)
    q, sb, g = orc.quant_act_nvfp4(v)
    deq = orc.dequant_act_nvfp4(q, sb, g)
    eff = np.repeat(sb * g[:, None].astype(np.float64), 16, axis=1)
    y = np.abs(v) / eff
    # half an e2m1 step at y (steps 0.5 / 1 / 2), which also covers a block's largest value
    # saturating at 6 after the e4m3 rounding of its scale (y <= 6 / (1 - 2^-4) < 6.5)
    bound = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0)) * eff
    assert np.all(np.abs(deq - v) <= bound * (1 + 1e-6))


def test_quant_act_nvfp4_matches_torch_based_quantiser():
    rng = np.random.default_rng(3)
    for _ in range(6):
        row = (rng.standard_normal(96) * np.exp(rng.uniform(-4, 4))).astype(np.float32)
        row[rng.integers(0, 96)] *= 40.0                                    # one outlier
        got = orc.fake_quant_act_nvfp4(row[None, :])[0]
        assert np.array_equal(got, np.array(bf.fake_quant_nvfp4(row.tolist())))


def test_weight_decode_nibble_by_nibble():
    w = torch.randn(2, 32, 64) * 0.1
    packed, sc, gs = wl.quantize_weights_nvfp4(w)
    for e in range(2):
        got = orc.dequant_weight_nvfp4(packed[e].numpy(), sc[e].numpy(), gs[e].numpy())
        assert np.array_equal(got, np.array(bf.dequant_weight_nvfp4_bruteforce(packed[e], sc[e], gs[e])))
    # the generator's NVFP4 copy is close to the weights it came from (block-relative error)
    deq = orc.dequant_weight_nvfp4(packed[0].numpy(), sc[0].numpy(), gs[0].numpy())
    amax_b = np.repeat(np.abs(w[0].numpy()).reshape(32, 4, 16).max(axis=2), 16, axis=1)
    assert np.all(np.abs(deq - w[0].numpy()) <= amax_b / 6.0 * 1.2 + 1e-7)


def _nvfp4_case(seed):
    cfg = wl.LayerConfig("f4", T=5, H=64, I=32, E=3, top_k=2, method=seed % 2, ranks=(2, 4), scalings=(2.0, 0.5),
                         slot_mode="uniform_none10", bias_std=0.1, rsf=2.0)
    inp = wl.make_inputs(cfg, seed=seed)
    return cfg, inp, wl.quantize_weights_nvfp4(inp["w1"]), wl.quantize_weights_nvfp4(inp["w2"])


def np_(t):
    return None if t is None else t.float().numpy() if t.dtype == torch.bfloat16 else t.numpy()


def nvfp4_dense_check(orc_mod, seed):
    """The oracle module's NVFP4 layer against the dense brute force (independent
    quantiser and weight decode)."""
    cfg, inp, w1, w2 = _nvfp4_case(seed)
    bias = np_(inp["correction_bias"])
    n = lambda t3: tuple(t.numpy() for t in t3)
    res = orc_mod.moe_lora_forward_nvfp4(np_(inp["hidden"]), np_(inp["router_logits"]), n(w1), n(w2), cfg.top_k,
                                         cfg.method, bias, cfg.rsf, np_(inp["lora_A_gu"]), np_(inp["lora_B_gu"]),
                                         np_(inp["lora_A_dn"]), np_(inp["lora_B_dn"]), inp["slot_idx"].numpy(),
                                         inp["ranks"], inp["scalings"])

    def keys_fn(row):
        s = orc.sigmoid_f32(np.asarray(row, np.float32))
        return list((s + bias).astype(np.float32).astype(np.float64)), list(s.astype(np.float64))

    L = lambda a: None if a is None else np.asarray(a, np.float64).tolist()
    W1 = [bf.dequant_weight_nvfp4_bruteforce(w1[0][e], w1[1][e], w1[2][e]) for e in range(cfg.E)]
    W2 = [bf.dequant_weight_nvfp4_bruteforce(w2[0][e], w2[1][e], w2[2][e]) for e in range(cfg.E)]
    dense, ids, _ = bf.dense_layer(L(np_(inp["hidden"])), L(np_(inp["router_logits"])), W1, W2, cfg.top_k,
                                   cfg.method, rsf=cfg.rsf, A_gu=L(np_(inp["lora_A_gu"])),
                                   B_gu=L(np_(inp["lora_B_gu"])), A_dn=L(np_(inp["lora_A_dn"])),
                                   B_dn=L(np_(inp["lora_B_dn"])), slot_idx=inp["slot_idx"].tolist(),
                                   ranks=inp["ranks"], scalings=inp["scalings"], keys_fn=keys_fn,
                                   quant=bf.fake_quant_nvfp4)
    return res["topk_ids"].tolist() == ids and np.array_equal(res["out"], np.array(dense))


@pytest.mark.parametrize("seed", [0, 1])
def test_nvfp4_layer_matches_dense_bruteforce(seed):
    assert nvfp4_dense_check(orc, seed)


def test_nvfp4_tolerance_covers_rounding_flips():
    """Derivation of the NVFP4 parity bounds (gpu_helpers: ten times the bf16 elementwise
    bounds, five times its relative L2 bound).  The NVFP4 GEMMs' products are exact and their
    sums fp32; model those sums' rounding by the probabilistic bound of a K-term sum,
    NVFP4_LAMBDA * sqrt(K) * 2^-24 times its sum of |terms|, and plant errors of that size
    (uniform within it) on the gate_up sums before their bf16 rounding, in a copy of the
    oracle.  The bf16 layer then stays inside the bf16 bounds.  The NVFP4 layer moves much
    further, because both of its GEMM inputs are re-quantised to e2m1: a one-ulp bf16 change
    of a gate_up value, or of a row's largest activation (its row scale), moves codes by a
    whole e2m1 step.  It leaves the bf16 bounds and stays inside the NVFP4 ones."""
    import types
    import os
    import gpu_helpers as gh

    src = open(os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "moe_lora_oracle.py")).read()
    anchor = "g = round_bf16(xg @ W1.T)"
    assert src.count(anchor) == 1
    noisy = types.ModuleType("oracle_noisy")
    noise = (f"g = round_bf16((xg @ W1.T) + {gh.NVFP4_LAMBDA} * np.sqrt(xg.shape[1]) * 2.0 ** -24"
             " * (np.abs(xg) @ np.abs(W1).T) * _NOISE.uniform(-1.0, 1.0, (xg.shape[0], W1.shape[0])))")
    exec(compile(src.replace(anchor, noise), "oracle_noisy", "exec"), noisy.__dict__)

    def rel(a, b):
        return np.linalg.norm(a - b) / np.linalg.norm(b)

    def within(got, ref, atol, rtol, rl):
        return bool(np.all(np.abs(got - ref) <= atol + rtol * np.abs(ref))) and rel(got, ref) <= rl

    cfgs = [wl.LayerConfig("n4a", T=40, H=256, I=256, E=8, top_k=2, ranks=(8, 16), scalings=(2.0, 0.5),
                           slot_mode="uniform_none10"),
            wl.LayerConfig("n4b", T=70, H=384, I=64, E=16, top_k=4, method=wl.DEEPSEEK_V3, bias_std=0.1, rsf=2.5,
                           ranks=(16,), scalings=(1.0,))]
    outside_bf16 = 0
    for cfg in cfgs:
        for seed in (11, 12):
            inp = wl.make_inputs(cfg, seed=seed)
            w1 = tuple(t.numpy() for t in wl.quantize_weights_nvfp4(inp["w1"]))
            w2 = tuple(t.numpy() for t in wl.quantize_weights_nvfp4(inp["w2"]))
            lora = (np_(inp["lora_A_gu"]), np_(inp["lora_B_gu"]), np_(inp["lora_A_dn"]), np_(inp["lora_B_dn"]),
                    inp["slot_idx"].numpy(), inp["ranks"], inp["scalings"])
            head = (np_(inp["hidden"]), np_(inp["router_logits"]))
            tail = (cfg.top_k, inp["method"], np_(inp["correction_bias"]), inp["rsf"]) + lora
            noisy._NOISE = np.random.default_rng(seed)
            n4_noisy = noisy.moe_lora_forward_nvfp4(*head, w1, w2, *tail)["out"]
            n4 = orc.moe_lora_forward_nvfp4(*head, w1, w2, *tail)["out"]
            assert within(n4_noisy, n4, gh.ATOL_NVFP4, gh.RTOL_NVFP4, gh.REL_L2_NVFP4), (cfg.name, seed)
            outside_bf16 += not within(n4_noisy, n4, gh.ATOL, gh.RTOL, gh.REL_L2)
            W1 = np.stack([orc.dequant_weight_nvfp4(w1[0][e], w1[1][e], w1[2][e]) for e in range(cfg.E)])
            W2 = np.stack([orc.dequant_weight_nvfp4(w2[0][e], w2[1][e], w2[2][e]) for e in range(cfg.E)])
            noisy._NOISE = np.random.default_rng(seed)
            b16_noisy = noisy.moe_lora_forward(*head, W1, W2, *tail)["out"]
            b16 = orc.moe_lora_forward(*head, W1, W2, *tail)["out"]
            assert within(b16_noisy, b16, gh.ATOL, gh.RTOL, gh.REL_L2), (cfg.name, seed)
    assert outside_bf16 >= 2
