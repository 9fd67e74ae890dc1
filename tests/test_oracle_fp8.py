"""Pins of the oracle's FP8 block-scale path (CPU).

The e4m3 decoder and rounding are checked against torch's float8_e4m3fn conversion (a
library routine) and against values the format fixes.  The quantisers are checked
against closed forms and error bounds.  The block-scaled GEMM is checked against a
blockwise brute force.  The whole FP8 layer is checked against the dense brute force of
tests/bruteforce.py run on torch's fp8 conversion.
"""
import math

import numpy as np
import pytest
import torch

import bruteforce as bf
from oracle import moe_lora_oracle as orc
from routed_moe_expert_gb300 import workloads as wl


def test_e4m3_decode_matches_torch_on_every_code():
    codes = np.arange(256)
    ours = orc.e4m3_decode(codes)
    ref = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[~np.isnan(ours)], ref[~np.isnan(ref)])
    assert np.isnan(ours).sum() == 2                 # S.1111.111 only: no infinities


def test_e4m3_values_the_format_fixes():
    d = orc.e4m3_decode
    assert d(0x7E) == 448.0                          # largest finite value
    assert d(0x08) == 2.0 ** -6                      # smallest normal
    assert d(0x01) == 2.0 ** -9                      # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9                  # largest subnormal
    assert d(0x38) == 1.0 and d(0xB8) == -1.0        # exponent field 7 = bias
    assert d(0x3C) == 1.5 and d(0x40) == 2.0
    assert d(0x00) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0


def test_round_e4m3_matches_torch():
    rng = np.random.default_rng(0)
    grid = orc.e4m3_decode(np.arange(256))
    grid = np.unique(grid[np.isfinite(grid)])
    mids = (grid[1:] + grid[:-1]) / 2                # ties: must go to the even mantissa
    x = np.concatenate([grid, mids, rng.uniform(-448, 448, 20000), rng.uniform(-0.05, 0.05, 20000),
                        rng.uniform(-2.0 ** -7, 2.0 ** -7, 5000)]).astype(np.float32)
    ours = orc.round_e4m3(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(ours, ref)


def test_round_e4m3_ties_and_saturation():
    r = orc.round_e4m3
    assert r(1.0625) == 1.0 and r(1.1875) == 1.25    # halfway: even mantissa (000, 010)
    assert r(2.0 ** -10) == 0.0 and r(3 * 2.0 ** -10) == 2 * 2.0 ** -9   # subnormal ties
    for v in (449.0, 463.9, 464.0, 1e6):
        assert r(v) == 448.0 and r(-v) == -448.0     # satfinite
    assert np.isnan(r(np.nan))


def test_quant_act_closed_forms():
    rng = np.random.default_rng(1)
    grid = orc.e4m3_decode(np.arange(0x7F))          # non-negative finite codes
    # a group whose largest magnitude is 448 * 2^k has scale 2^k and quantises exactly
    vals = rng.choice(grid, size=(3, 256)) * rng.choice([-1.0, 1.0], size=(3, 256))
    vals[:, 5] = 448.0
    vals[:, 200] = -448.0
    for k in (-3, 0, 2):
        v = vals * 2.0 ** k
        q, s = orc.quant_act_fp8(v)
        assert np.array_equal(s, np.full((3, 2), 2.0 ** k, np.float32))
        assert np.array_equal(orc.dequant_act_fp8(q, s), v)
    # an all-zero group: codes 0 and the floor scale
    q, s = orc.quant_act_fp8(np.zeros((1, 128)))
    assert np.all(q == 0) and s[0, 0] == np.float32(np.float32(1e-10) / np.float32(448.0))


def test_quant_act_error_bound_and_extreme_code():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal((16, 384)) * np.exp(rng.uniform(-6, 6, (16, 1)))).astype(np.float32)
    q, s = orc.quant_act_fp8(v)
    deq = orc.dequant_act_fp8(q, s)
    sg = np.repeat(s.astype(np.float64), 128, axis=1)
    normal = np.abs(v) / sg >= 2.0 ** -6
    err = np.abs(deq - v)
    # half a unit in the last place: 2^-4 relative for normals, 2^-10 * s below them
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(v[normal]) * (1 + 1e-6))
    assert np.all(err[~normal] <= 2.0 ** -10 * sg[~normal] * (1 + 1e-6))
    # each group's largest magnitude lands on +-448
    g = q.reshape(16, 3, 128)
    assert np.all(np.abs(g).max(axis=2) == 448.0)


def test_block_scaled_gemm_matches_blockwise_bruteforce():
    """sum over K-blocks of s_x * s_w * sum q_x q_w, written blockwise with exact sums,
    equals the oracle's product of the dequantised operands (block index of a weight
    value = (row // 128, col // 128))."""
    rng = np.random.default_rng(3)
    N, K = 256, 256
    codes = rng.integers(0, 0x7E, size=(N, K)) | (rng.integers(0, 2, size=(N, K)) << 7)
    wsc = np.array([[0.5, 3.0], [0.125, 7.0]])       # distinct, not symmetric
    x = rng.standard_normal((3, K)).astype(np.float32)
    qx, sx = orc.quant_act_fp8(x)
    W = orc.dequant_weight_fp8(codes, wsc)
    got = orc.dequant_act_fp8(qx, sx) @ W.T
    qw = orc.e4m3_decode(codes)
    for t in range(3):
        for n in range(0, N, 37):
            acc = []
            for b in range(K // 128):
                inner = math.fsum(qx[t, k] * qw[n, k] for k in range(128 * b, 128 * b + 128))
                acc.append(float(sx[t, b]) * wsc[n // 128, b] * inner)
            assert got[t, n] == pytest.approx(math.fsum(acc), rel=1e-12, abs=1e-12)


def _fp8_layer_case(seed, method=0):
    cfg = wl.LayerConfig("f8", T=5, H=256, I=128, E=4, top_k=2, method=method, ranks=(2, 4),
                         scalings=(2.0, 0.5), slot_mode="uniform_none10", bias_std=0.1, rsf=2.0)
    inp = wl.make_inputs(cfg, seed=seed)
    w1q, w1s = wl.quantize_weights_fp8(inp["w1"])
    w2q, w2s = wl.quantize_weights_fp8(inp["w2"])
    return cfg, inp, (w1q, w1s, w2q, w2s)


def np_(t):
    return None if t is None else t.float().numpy() if t.dtype == torch.bfloat16 else t.numpy()


def fp8_dense_check(orc_mod, seed):
    """The oracle module's FP8 layer against the dense brute force on torch's fp8."""
    cfg, inp, (w1q, w1s, w2q, w2s) = _fp8_layer_case(seed, method=seed % 2)
    bias = np_(inp["correction_bias"])
    res = orc_mod.moe_lora_forward_fp8(np_(inp["hidden"]), np_(inp["router_logits"]), w1q.numpy(), w1s.numpy(),
                                       w2q.numpy(), w2s.numpy(), cfg.top_k, cfg.method, bias, cfg.rsf,
                                       np_(inp["lora_A_gu"]), np_(inp["lora_B_gu"]), np_(inp["lora_A_dn"]),
                                       np_(inp["lora_B_dn"]), inp["slot_idx"].numpy(), inp["ranks"],
                                       inp["scalings"])

    def keys_fn(row):
        s = orc.sigmoid_f32(np.asarray(row, np.float32))
        return list((s + bias).astype(np.float32).astype(np.float64)), list(s.astype(np.float64))

    L = lambda a: None if a is None else np.asarray(a, np.float64).tolist()
    W1 = [bf.dequant_weight_torch(w1q[e], w1s[e]) for e in range(cfg.E)]
    W2 = [bf.dequant_weight_torch(w2q[e], w2s[e]) for e in range(cfg.E)]
    dense, ids, _ = bf.dense_layer(L(np_(inp["hidden"])), L(np_(inp["router_logits"])), W1, W2, cfg.top_k,
                                   cfg.method, rsf=cfg.rsf, A_gu=L(np_(inp["lora_A_gu"])),
                                   B_gu=L(np_(inp["lora_B_gu"])), A_dn=L(np_(inp["lora_A_dn"])),
                                   B_dn=L(np_(inp["lora_B_dn"])), slot_idx=inp["slot_idx"].tolist(),
                                   ranks=inp["ranks"], scalings=inp["scalings"], keys_fn=keys_fn,
                                   quant=bf.fake_quant_torch)
    return res["topk_ids"].tolist() == ids and np.array_equal(res["out"], np.array(dense))


@pytest.mark.parametrize("seed", [0, 1])
def test_fp8_layer_matches_dense_bruteforce(seed):
    assert fp8_dense_check(orc, seed)


def test_fp8_layer_differs_from_bf16_layer_only_by_quantisation():
    """With weights and inputs that FP8 represents exactly (block scales 1, values on the
    e4m3 grid, every activation group holding +-448) the two GEMM inputs quantise without
    error, so the FP8 layer without LoRA equals the bf16 layer on the dequantised weights."""
    rng = np.random.default_rng(4)
    T, H, I, E, k = 4, 128, 128, 3, 2
    grid = orc.e4m3_decode(np.arange(0x7F))
    w1q = rng.integers(0, 0x40, size=(E, 2 * I, H)).astype(np.uint8)    # |w| < 2
    w2q = rng.integers(0, 0x40, size=(E, H, I)).astype(np.uint8)
    w1s = np.full((E, 2, 1), 1.0 / 64)
    w2s = np.full((E, 1, 1), 1.0 / 64)
    x = rng.choice(grid[:0x50], size=(T, H))
    x[:, 0] = 448.0
    logits = rng.standard_normal((T, E)).astype(np.float32)
    f8 = orc.moe_lora_forward_fp8(x, logits, w1q, w1s, w2q, w2s, k)
    W1 = np.stack([orc.dequant_weight_fp8(w1q[e], w1s[e]) for e in range(E)])
    W2 = np.stack([orc.dequant_weight_fp8(w2q[e], w2s[e]) for e in range(E)])
    ref = orc.moe_lora_forward(x, logits, W1, W2, k, keep_intermediates=True)
    # the activations a are not on the e4m3 grid: compare through the oracle's own
    # quantiser applied to the bf16 layer's a (the down GEMM's only extra rounding)
    for p, it in ref["pairs"].items():
        t, j = divmod(p, k)
        e = int(ref["topk_ids"][t, j])
        y8 = orc.fake_quant_act_fp8(it["a"][None, :])[0] @ W2[e].T
        it["y8"] = y8
    acc = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            acc[t] += ref["topk_weights"][t, j] * ref["pairs"][t * k + j]["y8"]
    assert np.array_equal(f8["out"], orc.round_bf16(acc))


def test_fp8_tolerance_covers_accumulation_noise():
    """Derivation of the FP8 parity bounds from the accumulation model of the FP8 GEMM
    (gpu_helpers.FP8_ACC_BITS, which tests/test_gpu_fp8.py holds the GPU GEMM to): the tensor
    cores sum each 128-wide block of e4m3 products with fewer bits than float32 keeps (which is
    why the FP8 recipe promotes every block to float32 with its scales), off by at most
    7 * 2^-FP8_ACC_BITS times the block's sum of |products|.  Plant errors of that size
    (uniform within the bound) on the gate_up GEMM's output before its bf16 rounding, in a copy
    of the oracle, on the shapes of the GPU tests (one and two 128-value groups per activation
    row, one to four adapters) and several inputs.  The bf16 layer then stays inside the bf16
    bounds, while the FP8 layer moves about three times as far in relative L2 and much further
    on single elements: its activation is re-quantised to e4m3, where a one-ulp bf16 change
    moves a code by a whole e4m3 step (2^-3 instead of 2^-8), and a change of a group's largest
    value changes the group's scale (amax / 448) and so every code of the group.  With one
    group per row (I = 128) such a change moves a token's whole output row.  The FP8 bounds
    cover all of it, and the bf16 bounds do not."""
    import types
    import os
    import gpu_helpers as gh

    src = open(os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "moe_lora_oracle.py")).read()
    anchor = "g = round_bf16(xg @ W1.T)"
    assert src.count(anchor) == 1
    noisy = types.ModuleType("oracle_noisy")
    noise = (f"g = round_bf16((xg @ W1.T) + 7 * 2.0 ** -{gh.FP8_ACC_BITS} * (np.abs(xg) @ np.abs(W1).T)"
             " * _NOISE.uniform(-1.0, 1.0, (xg.shape[0], W1.shape[0])))")
    exec(compile(src.replace(anchor, noise), "oracle_noisy", "exec"), noisy.__dict__)

    def rel(a, b):
        return np.linalg.norm(a - b) / np.linalg.norm(b)

    def within(got, ref, atol, rtol, rl):
        return bool(np.all(np.abs(got - ref) <= atol + rtol * np.abs(ref))) and rel(got, ref) <= rl

    cfgs = [wl.LayerConfig("f8n", T=40, H=256, I=256, E=8, top_k=2, ranks=(8, 16), scalings=(2.0, 0.5),
                           slot_mode="uniform_none10"),
            wl.LayerConfig("f8n_tiles", T=300, H=256, I=128, E=4, top_k=2, ranks=(4, 12), scalings=(1.0, 2.0),
                           slot_mode="uniform_none10"),
            wl.LayerConfig("f8n_dis", T=600, H=256, I=128, E=8, top_k=2, ranks=(16, 24, 0, 8),
                           scalings=(1.0, 0.0, 1.0, 2.0), slot_mode="uniform_none10"),
            wl.LayerConfig("f8n_four", T=96, H=512, I=256, E=16, top_k=4, ranks=(8, 16, 32, 64),
                           scalings=(2.0, 1.0, 0.5, 0.25), slot_mode="uniform_none10")]
    ratios = []
    for cfg in cfgs:
        for seed in (11, 12):
            inp = wl.make_inputs(cfg, seed=seed)
            w1q, w1s = wl.quantize_weights_fp8(inp["w1"])
            w2q, w2s = wl.quantize_weights_fp8(inp["w2"])
            W1 = np.stack([orc.dequant_weight_fp8(w1q[e].numpy(), w1s[e].numpy()) for e in range(cfg.E)])
            W2 = np.stack([orc.dequant_weight_fp8(w2q[e].numpy(), w2s[e].numpy()) for e in range(cfg.E)])
            lora = (np_(inp["lora_A_gu"]), np_(inp["lora_B_gu"]), np_(inp["lora_A_dn"]), np_(inp["lora_B_dn"]),
                    inp["slot_idx"].numpy(), inp["ranks"], inp["scalings"])
            x, lg = np_(inp["hidden"]), np_(inp["router_logits"])
            q8 = (w1q.numpy(), w1s.numpy(), w2q.numpy(), w2s.numpy())
            f8 = orc.moe_lora_forward_fp8(x, lg, *q8, cfg.top_k, 0, None, 1.0, *lora)["out"]
            b16 = orc.moe_lora_forward(x, lg, W1, W2, cfg.top_k, 0, None, 1.0, *lora)["out"]
            for ns in range(2):
                noisy._NOISE = np.random.default_rng(ns)
                f8_noisy = noisy.moe_lora_forward_fp8(x, lg, *q8, cfg.top_k, 0, None, 1.0, *lora)["out"]
                noisy._NOISE = np.random.default_rng(ns)
                b16_noisy = noisy.moe_lora_forward(x, lg, W1, W2, cfg.top_k, 0, None, 1.0, *lora)["out"]
                assert within(b16_noisy, b16, gh.ATOL, gh.RTOL, gh.REL_L2), (cfg.name, seed, ns)
                assert not within(f8_noisy, f8, gh.ATOL, gh.RTOL, gh.REL_L2), (cfg.name, seed, ns)
                assert within(f8_noisy, f8, gh.ATOL_FP8, gh.RTOL_FP8, gh.REL_L2_FP8), (cfg.name, seed, ns)
                ratios.append(rel(f8_noisy, f8) / rel(b16_noisy, b16))
    assert 2.0 < float(np.median(ratios)) < 4.5
