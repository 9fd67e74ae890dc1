"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against something its own code does not produce:
a library routine (torch's bf16 conversion, math.exp, scipy's softmax, a torch
float64 MLP), an independent brute force (dense evaluation with exact sums and
exact rational bf16 rounding), closed forms, invariants, and a hand-computed
example stored under tests/golden/.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import bruteforce as bf
from oracle import moe_lora_oracle as orc
from routed_moe_expert_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def np_(t):
    return None if t is None else t.float().numpy() if t.dtype == torch.bfloat16 else t.numpy()


# ---------------------------------------------------------------- bf16 rounding

def test_round_bf16_matches_torch_conversion():
    """float32 inputs: one rounding float32 -> bf16, as torch's conversion does."""
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -130,
                  3 * 2.0 ** -134, 0.0, -0.0, 1e38, 3.3e38]),
    ]).astype(np.float32)
    ours = orc.round_bf16(vals.astype(np.float64))
    ref = torch.from_numpy(vals).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(ours, ref)


def test_round_bf16_matches_exact_rational_rounding():
    """float64 inputs with more than 24 bits: single rounding, checked with Fractions."""
    rng = np.random.default_rng(1)
    vals = rng.standard_normal(3000) * 10.0 ** rng.integers(-20, 20, 3000)
    ties = [1.0 + 2.0 ** -8 + 2.0 ** -40, 1.0 + 2.0 ** -8 - 2.0 ** -40, 1.0 + 2.0 ** -8]
    vals = np.concatenate([vals, ties])
    ours = orc.round_bf16(vals)
    ref = np.array([bf.bf16_exact(float(v)) for v in vals])
    np.testing.assert_array_equal(ours, ref)
    assert orc.round_bf16(1.0 + 2.0 ** -8) == 1.0            # tie to even (down)
    assert orc.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6  # tie to even (up)


# ---------------------------------------------------------------- float32 sigmoid

def test_exp_f32_within_two_ulp_of_math_exp():
    xs = np.concatenate([np.linspace(-86, 88, 20001), np.random.default_rng(2).uniform(-10, 10, 5000)])
    xs = xs.astype(np.float32)
    ours = orc.exp_f32(xs).astype(np.float64)
    ref = np.array([math.exp(float(v)) for v in xs])
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(ours - ref) / ulp) <= 2.0


def test_sigmoid_f32_within_two_ulp_and_exact_points():
    zs = np.concatenate([np.linspace(-30, 30, 30001),
                         torch.randn(5000, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16).float().numpy()])
    zs = zs.astype(np.float32)
    ours = orc.sigmoid_f32(zs).astype(np.float64)
    ref = np.array([bf.sigmoid(float(z)) for z in zs])
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(ours - ref) / ulp) <= 3.0
    assert orc.sigmoid_f32(np.float32(0.0)) == np.float32(0.5)
    # symmetry sigma(-z) = 1 - sigma(z) holds to float32 rounding
    a = orc.sigmoid_f32(zs).astype(np.float64) + orc.sigmoid_f32(-zs).astype(np.float64)
    assert np.max(np.abs(a - 1.0)) < 2e-7


# ---------------------------------------------------------------- routing

@pytest.mark.parametrize("method", [0, 1])
def test_route_matches_bruteforce_sort(method):
    g = torch.Generator().manual_seed(4)
    T, E, k = 40, 24, 5
    logits = torch.randn(T, E, generator=g).to(torch.bfloat16).float().numpy()
    logits[3, :] = 0.25                 # a row of ties
    logits[5, 7] = logits[5, 2]         # a single tie
    bias = (torch.randn(E, generator=g) * 0.1).numpy().astype(np.float32)
    bias[9] = bias[10]
    ids, w = orc.route(logits, k, method, bias, routed_scaling_factor=2.5)
    for t in range(T):
        row = logits[t].astype(np.float64)
        if method == 0:
            keys = list(row)
        else:
            s = orc.sigmoid_f32(logits[t])
            keys = list((s + bias).astype(np.float32).astype(np.float64))
        assert list(ids[t]) == bf.topk_bruteforce(keys, k)
        if method == 0:
            sel = row[ids[t]]
            from scipy.special import softmax
            np.testing.assert_allclose(w[t], softmax(sel), rtol=1e-13)
            np.testing.assert_allclose(w[t].sum(), 1.0, rtol=1e-13)
        else:
            np.testing.assert_allclose(w[t].sum(), 2.5, rtol=1e-13)
    assert list(ids[3]) == [0, 1, 2, 3, 4] if method == 0 else True


def test_renormalize_equals_softmax_then_renormalize():
    """RenormalizeNaive (softmax of all logits, keep top k, renormalise) gives the
    same weights as the softmax of the selected logits."""
    g = torch.Generator().manual_seed(5)
    logits = torch.randn(16, 32, generator=g).to(torch.bfloat16).float().numpy()
    ids, w = orc.route(logits, 4, 0)
    full = torch.softmax(torch.from_numpy(logits).double(), dim=1).numpy()
    sel = np.take_along_axis(full, ids, axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-12)


def test_route_constant_logits_give_lowest_ids():
    ids, w = orc.route(np.zeros((3, 10), np.float32), 4, 0)
    assert (ids == np.arange(4)).all()
    np.testing.assert_allclose(w, 0.25)


def test_deepseek_weights_use_scores_not_keys():
    """Bias changes which experts win but not the weight formula s/sum(s)*rsf."""
    logits = np.array([[2.0, 0.0, -1.0]], np.float32)
    bias = np.array([0.0, 5.0, 5.0], np.float32)
    ids, w = orc.route(logits, 2, 1, bias, routed_scaling_factor=3.0)
    assert list(ids[0]) == [1, 2]
    s1, s2 = bf.sigmoid(0.0), bf.sigmoid(-1.0)
    np.testing.assert_allclose(w[0], [3 * s1 / (s1 + s2), 3 * s2 / (s1 + s2)], rtol=1e-6)


# ---------------------------------------------------------------- align

def test_align_matches_bruteforce_and_invariants():
    rng = np.random.default_rng(6)
    T, k, E = 50, 3, 9
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    ids[ids == 4] = 5   # leave expert 4 empty (ids per token may now repeat; align does not care)
    off, perm, inv = orc.align(ids, E)
    flat = ids.reshape(-1)
    expect = []
    for e in range(E):
        for p in range(flat.size):
            if flat[p] == e:
                expect.append(p)
    assert list(perm) == expect
    assert off[0] == 0 and off[-1] == flat.size and (np.diff(off) >= 0).all()
    assert off[5] == off[4]
    assert (inv[perm] == np.arange(flat.size)).all()
    for e in range(E):
        seg = perm[off[e]:off[e + 1]]
        assert (flat[seg] == e).all() and (np.diff(seg) > 0).all()


# ---------------------------------------------------------------- the layer

def _to_lists(a):
    return None if a is None else np.asarray(a, dtype=np.float64).tolist()


def _run_both(inp, lora_off=False):
    args = dict(
        top_k=inp["top_k"], method=inp["method"],
        correction_bias=np_(inp["correction_bias"]), routed_scaling_factor=inp["rsf"],
        lora_A_gu=np_(inp["lora_A_gu"]), lora_B_gu=np_(inp["lora_B_gu"]),
        lora_A_dn=np_(inp["lora_A_dn"]), lora_B_dn=np_(inp["lora_B_dn"]),
        slot_idx=inp["slot_idx"].numpy(), ranks=inp["ranks"], scalings=inp["scalings"])
    res = orc.moe_lora_forward(np_(inp["hidden"]), np_(inp["router_logits"]), np_(inp["w1"]),
                               np_(inp["w2"]), lora_off=lora_off, **args)
    bias = np_(inp["correction_bias"])

    def keys_fn(row):
        s = orc.sigmoid_f32(np.asarray(row, np.float32))
        return list((s + bias).astype(np.float32).astype(np.float64)), list(s.astype(np.float64))

    ranks = [] if lora_off else inp["ranks"]
    dense, ids, w = bf.dense_layer(
        _to_lists(np_(inp["hidden"])), _to_lists(np_(inp["router_logits"])),
        _to_lists(np_(inp["w1"])), _to_lists(np_(inp["w2"])), inp["top_k"], inp["method"],
        rsf=inp["rsf"], A_gu=_to_lists(np_(inp["lora_A_gu"])), B_gu=_to_lists(np_(inp["lora_B_gu"])),
        A_dn=_to_lists(np_(inp["lora_A_dn"])), B_dn=_to_lists(np_(inp["lora_B_dn"])),
        slot_idx=inp["slot_idx"].tolist(), ranks=ranks, scalings=inp["scalings"], keys_fn=keys_fn)
    return res, np.array(dense), ids, w


@pytest.mark.parametrize("seed", range(8))
def test_layer_matches_dense_bruteforce(seed):
    """Every token through every expert, masked by routing, exact sums: the oracle
    (grouped by expert, permuted, gathered) must give the same bf16 outputs."""
    rng = np.random.default_rng(100 + seed)
    cfg = wl.random_small_config(rng, max_T=6, max_E=5)
    cfg = wl.LayerConfig("bf", T=cfg.T, H=16, I=8, E=cfg.E, top_k=cfg.top_k, method=cfg.method,
                         ranks=cfg.ranks, scalings=cfg.scalings, slot_mode="uniform_none10",
                         bias_std=0.1, rsf=cfg.rsf)
    inp = wl.make_inputs(cfg, seed=seed)
    res, dense, ids, w = _run_both(inp)
    assert res["topk_ids"].tolist() == ids
    np.testing.assert_allclose(res["topk_weights"], np.array(w), rtol=1e-13)
    np.testing.assert_array_equal(res["out"], dense)


def test_layer_matches_dense_bruteforce_tiny_config():
    """The tiny parity configuration (T8 H128 I64 E8 k2, rank 4), dense brute force."""
    inp = wl.make_inputs(wl.CONFIGS["tiny"], seed=0)
    res, dense, _, _ = _run_both(inp)
    np.testing.assert_array_equal(res["out"], dense)


def test_hand_example():
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        G = json.load(f)
    for case in G["cases"]:
        lora = case["lora"]
        res = orc.moe_lora_forward(
            np.array(G["hidden"], float), np.array(case["logits"], float),
            np.array(G["w1"], float), np.array(G["w2"], float), case["top_k"], case["method"],
            correction_bias=np.array(case.get("bias", [0, 0]), np.float32),
            routed_scaling_factor=case.get("rsf", 1.0),
            lora_A_gu=np.array(G["lora_A_gu"], float), lora_B_gu=np.array(G["lora_B_gu"], float),
            lora_A_dn=np.array(G["lora_A_dn"], float), lora_B_dn=np.array(G["lora_B_dn"], float),
            slot_idx=np.array(case.get("slot_idx", [0, 0])), ranks=G["ranks"], scalings=G["scalings"],
            lora_off=not lora)
        assert res["topk_ids"].tolist() == case["topk_ids"], case["name"]
        np.testing.assert_allclose(res["topk_weights"], case["topk_weights"], rtol=1e-7, err_msg=case["name"])
        np.testing.assert_array_equal(res["out"], np.array(case["out"], float), err_msg=case["name"])


def test_single_expert_reduces_to_torch_mlp():
    """E = 1, k = 1, no LoRA: the layer is bf16(w2 @ bf16(silu(bf16(Wg x)) * bf16(Wu x)))
    -- a plain gated MLP, evaluated here with torch float64 ops."""
    g = torch.Generator().manual_seed(7)
    T, H, I = 9, 64, 32
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).double()
    w1 = (torch.randn(1, 2 * I, H, generator=g) / 8).to(torch.bfloat16).double()
    w2 = (torch.randn(1, H, I, generator=g) / 6).to(torch.bfloat16).double()

    def rb(t):
        return torch.from_numpy(orc.round_bf16(t.numpy()))

    gate = rb(x @ w1[0, :I].T)
    up = rb(x @ w1[0, I:].T)
    a = rb(torch.nn.functional.silu(gate) * up)
    ref = rb(a @ w2[0].T)
    res = orc.moe_lora_forward(x.numpy(), np.zeros((T, 1)), w1.numpy(), w2.numpy(), 1)
    np.testing.assert_array_equal(res["out"], ref.numpy())


def test_lora_delta_equals_merged_weight_difference():
    """d = scaling * B A x is the change of the gate_up output when the LoRA is merged
    into the weight (W1 + scaling * B A); checked per pair before bf16 rounding."""
    cfg = wl.CONFIGS["tiny"]
    inp = wl.make_inputs(cfg, seed=1, nan_rank_tail=False)
    res = orc.moe_lora_forward(np_(inp["hidden"]), np_(inp["router_logits"]), np_(inp["w1"]),
                               np_(inp["w2"]), cfg.top_k, lora_A_gu=np_(inp["lora_A_gu"]),
                               lora_B_gu=np_(inp["lora_B_gu"]), lora_A_dn=np_(inp["lora_A_dn"]),
                               lora_B_dn=np_(inp["lora_B_dn"]), slot_idx=inp["slot_idx"].numpy(),
                               ranks=inp["ranks"], scalings=inp["scalings"], keep_intermediates=True)
    x = inp["hidden"].double()
    sc = inp["scalings"][0]
    for p, rec in res["pairs"].items():
        t, j = divmod(p, cfg.top_k)
        e = int(res["topk_ids"][t, j])
        W = inp["w1"][e].double()
        M = W + sc * inp["lora_B_gu"][0, e].double() @ inp["lora_A_gu"][0, e].double()
        diff = (M @ x[t] - W @ x[t]).numpy()
        np.testing.assert_allclose(rec["d"], diff, rtol=2 ** -7, atol=1e-6)
        # and the down delta against the merged down weight
        W2 = inp["w2"][e].double()
        M2 = W2 + sc * inp["lora_B_dn"][0, e].double() @ inp["lora_A_dn"][0, e].double()
        a = torch.from_numpy(rec["a"])
        np.testing.assert_allclose(rec["y"] + rec["dd"], (M2 @ a).numpy(), rtol=1e-10, atol=1e-12)


def test_lora_vanishes_for_zero_scaling_or_no_slot():
    cfg = wl.CONFIGS["multi_slot"]
    cfg = wl.LayerConfig("ms", T=32, H=64, I=64, E=8, top_k=2, ranks=(8, 16, 4),
                         scalings=(0.0, 1.0, 0.5), slot_mode="uniform_none10")
    inp = wl.make_inputs(cfg, seed=2)
    base, _, _, _ = _run_both(inp, lora_off=True)
    res, _, _, _ = _run_both(inp)
    slots = inp["slot_idx"].numpy()
    no_delta = (slots == -1) | (slots == 0)
    assert no_delta.any() and (~no_delta).any()
    np.testing.assert_array_equal(res["out"][no_delta], base["out"][no_delta])
    assert not np.array_equal(res["out"][~no_delta], base["out"][~no_delta])


def test_rank_one_lora_closed_form():
    """A = e_i (picks x[i]), B = c e_n: the gate_up delta is scaling*c*x[i] at row n only."""
    T, H, I, E = 4, 8, 4, 2
    rng = np.random.default_rng(8)
    x = orc.round_bf16(rng.standard_normal((T, H)))
    w1 = orc.round_bf16(rng.standard_normal((E, 2 * I, H)) / 3)
    w2 = orc.round_bf16(rng.standard_normal((E, H, I)) / 2)
    A = np.zeros((1, E, 1, H)); A[0, :, 0, 3] = 1.0
    B = np.zeros((1, E, 2 * I, 1)); B[0, :, I + 1, 0] = 0.75       # an up row
    Ad = np.zeros((1, E, 1, I)); Bd = np.zeros((1, E, H, 1))
    res = orc.moe_lora_forward(x, np.zeros((T, E)), w1, w2, 1, lora_A_gu=A, lora_B_gu=B,
                               lora_A_dn=Ad, lora_B_dn=Bd, slot_idx=np.zeros(T, int), ranks=[1],
                               scalings=[2.0], keep_intermediates=True)
    for p, rec in res["pairs"].items():
        expect = np.zeros(2 * I)
        expect[I + 1] = orc.round_bf16(2.0 * 0.75 * x[p, 3])
        np.testing.assert_array_equal(rec["d"], expect)


def test_up_half_delta_changes_only_up_factor():
    """Regression for the gated-split bug of the fused path (sglang PR #27329,
    Optimizations: "gate_up gated-split fix for the up-half"): a delta on the up rows
    only must enter as silu(gate) * (up + d_up)."""
    cfg = wl.LayerConfig("up", T=6, H=64, I=64, E=4, top_k=2, ranks=(8,), scalings=(1.0,))
    inp = wl.make_inputs(cfg, seed=3, nan_rank_tail=False)
    inp["lora_B_gu"][:, :, :cfg.I, :] = 0     # gate half of B zero
    res = orc.moe_lora_forward(np_(inp["hidden"]), np_(inp["router_logits"]), np_(inp["w1"]),
                               np_(inp["w2"]), cfg.top_k, lora_A_gu=np_(inp["lora_A_gu"]),
                               lora_B_gu=np_(inp["lora_B_gu"]), lora_A_dn=np_(inp["lora_A_dn"]),
                               lora_B_dn=np_(inp["lora_B_dn"]), slot_idx=inp["slot_idx"].numpy(),
                               ranks=inp["ranks"], scalings=inp["scalings"], keep_intermediates=True)
    I = cfg.I
    for rec in res["pairs"].values():
        assert (rec["d"][:I] == 0).all() and (rec["d"][I:] != 0).any()
        g = rec["g"]
        np.testing.assert_array_equal(rec["a"], orc.round_bf16(orc.silu(g[:I]) * (g[I:] + rec["d"][I:])))


def test_slot_permutation_permutes_outputs():
    """Regression for the slot-0 bug (sglang PR #28091, Motivation 2: slot 0's weights
    and scaling applied to every request): relabelling slots while permuting the
    stacked adapters must leave every token's output unchanged."""
    cfg = wl.LayerConfig("sl", T=24, H=64, I=64, E=6, top_k=2, ranks=(4, 8, 16, 2),
                         scalings=(2.0, 1.0, 0.5, 0.25), slot_mode="uniform_none10")
    inp = wl.make_inputs(cfg, seed=4)
    ref, _, _, _ = _run_both(inp)
    pi = [2, 0, 3, 1]                     # new slot n holds old slot pi[n]
    new = dict(inp)
    for key in ("lora_A_gu", "lora_B_gu", "lora_A_dn", "lora_B_dn"):
        new[key] = inp[key][pi]
    new["ranks"] = [inp["ranks"][i] for i in pi]
    new["scalings"] = [inp["scalings"][i] for i in pi]
    old_to_new = {o: n for n, o in enumerate(pi)}
    new["slot_idx"] = torch.tensor([old_to_new.get(int(s), -1) for s in inp["slot_idx"]], dtype=torch.int32)
    res, _, _, _ = _run_both(new)
    np.testing.assert_array_equal(res["out"], ref["out"])
    # and a slot-0-for-everyone mistake would not: slots differ in output
    assert len(set(int(s) for s in inp["slot_idx"])) > 2


# ---------------------------------------------------------------- shared-outer LoRA

@pytest.mark.parametrize("seed", range(4))
def test_shared_outer_matches_dense_bruteforce(seed):
    """One A_gu and one B_dn per slot for every expert: the dense brute force (every token
    through every expert, exact sums) gives the same bf16 outputs."""
    rng = np.random.default_rng(400 + seed)
    base = wl.random_small_config(rng, max_T=6, max_E=5)
    cfg = wl.LayerConfig("so", T=base.T, H=16, I=8, E=base.E, top_k=base.top_k, ranks=(4, 2),
                         scalings=(2.0, 0.5), slot_mode="uniform_none10", shared_outer=True)
    inp = wl.make_inputs(cfg, seed=seed)
    assert tuple(inp["lora_A_gu"].shape[:2]) == (2, 1) and tuple(inp["lora_B_dn"].shape[:2]) == (2, 1)
    lora = dict(lora_A_gu=np_(inp["lora_A_gu"]), lora_B_gu=np_(inp["lora_B_gu"]),
                lora_A_dn=np_(inp["lora_A_dn"]), lora_B_dn=np_(inp["lora_B_dn"]))
    res = orc.moe_lora_forward(np_(inp["hidden"]), np_(inp["router_logits"]), np_(inp["w1"]), np_(inp["w2"]),
                               cfg.top_k, slot_idx=inp["slot_idx"].numpy(), ranks=inp["ranks"],
                               scalings=inp["scalings"], shared_outer=True, **lora)
    dense, _, _ = bf.dense_layer(
        _to_lists(np_(inp["hidden"])), _to_lists(np_(inp["router_logits"])), _to_lists(np_(inp["w1"])),
        _to_lists(np_(inp["w2"])), cfg.top_k, 0, A_gu=_to_lists(lora["lora_A_gu"]),
        B_gu=_to_lists(lora["lora_B_gu"]), A_dn=_to_lists(lora["lora_A_dn"]), B_dn=_to_lists(lora["lora_B_dn"]),
        slot_idx=inp["slot_idx"].tolist(), ranks=inp["ranks"], scalings=inp["scalings"], shared_outer=True)
    np.testing.assert_array_equal(res["out"], np.array(dense))


def test_shared_outer_equals_per_expert_with_copies():
    """Shared-outer is the per-expert layer whose A_gu and B_dn are the same for every
    expert: copying the shared weights to every expert gives the same bits."""
    cfg = wl.LayerConfig("so2", T=7, H=16, I=8, E=4, top_k=2, ranks=(4,), scalings=(1.5,), shared_outer=True)
    inp = wl.make_inputs(cfg, seed=3)
    E = cfg.E
    A_gu, B_dn = np_(inp["lora_A_gu"]), np_(inp["lora_B_dn"])
    common = dict(lora_B_gu=np_(inp["lora_B_gu"]), lora_A_dn=np_(inp["lora_A_dn"]), slot_idx=inp["slot_idx"].numpy(),
                  ranks=inp["ranks"], scalings=inp["scalings"])
    args = (np_(inp["hidden"]), np_(inp["router_logits"]), np_(inp["w1"]), np_(inp["w2"]), 2)
    a = orc.moe_lora_forward(*args, lora_A_gu=A_gu, lora_B_dn=B_dn, shared_outer=True, **common)
    b = orc.moe_lora_forward(*args, lora_A_gu=np.repeat(A_gu, E, axis=1), lora_B_dn=np.repeat(B_dn, E, axis=1),
                             **common)
    np.testing.assert_array_equal(a["out"], b["out"])


# ---------------------------------------------------------------- externally routed entry

def test_pack_topk_golden():
    """(expert << 16) | bf16 bits of the weight, written out by hand: 5 with 0.5 is
    0x00053F00, 1023 with -1.0 is 0x03FFBF80, 2 with 0.1 is 0x00023DCD (0.1 rounds to the
    bf16 0x3DCD = 0.10009765625); unpacking returns the ids and those bf16 values."""
    packed = orc.pack_topk(np.array([[5, 1023, 2]]), np.array([[0.5, -1.0, 0.1]]))
    assert [int(v) & 0xFFFFFFFF for v in packed.reshape(-1)] == [0x00053F00, 0x03FFBF80, 0x00023DCD]
    ids, w = orc.unpack_topk(packed)
    assert ids.tolist() == [[5, 1023, 2]]
    assert w.tolist() == [[0.5, -1.0, 0.10009765625]]


def test_pack_topk_equals_the_input_encoding():
    """The oracle's packing (numpy, bf16 by frexp/rint) and the seeded input generator's
    (torch bfloat16 conversion and int64 shifts) agree on every word, ids up to 65535."""
    ids, w = wl.make_routing(200, 40000, 8, seed=4)
    ids[0, 0] = 65535
    w[1, 0] = 0.1
    np.testing.assert_array_equal(orc.pack_topk(ids.numpy(), w.numpy()), wl.packed_routing_words(ids, w).numpy())


def _routed_case(seed, E_loc, E_glob, offset, T=5, k=2):
    rng = np.random.default_rng(300 + seed)
    cfg = wl.LayerConfig("rt", T=T, H=16, I=8, E=E_loc, top_k=k, ranks=(4, 2), scalings=(2.0, 0.5),
                         slot_mode="uniform_none10")
    inp = wl.make_inputs(cfg, seed=seed)
    ids, w = wl.make_routing(T, E_glob, k, seed=int(rng.integers(1 << 30)))
    packed = orc.pack_topk(ids.numpy(), w.numpy())
    lora = dict(lora_A_gu=np_(inp["lora_A_gu"]), lora_B_gu=np_(inp["lora_B_gu"]),
                lora_A_dn=np_(inp["lora_A_dn"]), lora_B_dn=np_(inp["lora_B_dn"]),
                slot_idx=inp["slot_idx"].numpy(), ranks=inp["ranks"], scalings=inp["scalings"])
    return inp, packed, lora


@pytest.mark.parametrize("seed", range(6))
def test_routed_matches_dense_bruteforce_with_dropped_experts(seed):
    """Given routing over 6 global experts of which 3 are local (offset 2): every token
    through every local expert, masked by the given routing, exact sums.  Pairs routed
    to other experts contribute nothing."""
    inp, packed, lora = _routed_case(seed, E_loc=3, E_glob=6, offset=2)
    res = orc.moe_lora_forward_routed(np_(inp["hidden"]), packed, np_(inp["w1"]), np_(inp["w2"]), 2,
                                      num_experts=6, local_expert_offset=2, **lora)
    gid, w = orc.unpack_topk(packed)
    dense = bf.dense_layer_routed(
        _to_lists(np_(inp["hidden"])), gid.tolist(), w.tolist(), 2, _to_lists(np_(inp["w1"])),
        _to_lists(np_(inp["w2"])), A_gu=_to_lists(lora["lora_A_gu"]), B_gu=_to_lists(lora["lora_B_gu"]),
        A_dn=_to_lists(lora["lora_A_dn"]), B_dn=_to_lists(lora["lora_B_dn"]),
        slot_idx=lora["slot_idx"].tolist(), ranks=lora["ranks"], scalings=lora["scalings"])
    np.testing.assert_array_equal(res["out"], np.array(dense))
    local = (gid >= 2) & (gid < 5)
    assert np.array_equal(res["expanded_idx_to_permuted_idx"] >= 0, local.reshape(-1))


def test_routed_expert_parallel_partials_sum_to_one_rank():
    """Two ranks owning experts [0, 3) and [3, 6): their unrounded partial outputs add up
    to the single-rank output (the all-reduce of the pages' expert-parallel layout)."""
    inp, packed, lora = _routed_case(7, E_loc=6, E_glob=6, offset=0, T=8, k=3)
    x, w1, w2 = np_(inp["hidden"]), np_(inp["w1"]), np_(inp["w2"])

    def part(lo, hi):
        sub = {key: (v[:, lo:hi] if key.startswith("lora_") else v) for key, v in lora.items()}
        return orc.moe_lora_forward_routed(x, packed, w1[lo:hi], w2[lo:hi], 3, num_experts=6,
                                           local_expert_offset=lo, **sub)["out_acc"]

    full = part(0, 6)
    np.testing.assert_allclose(part(0, 3) + part(3, 6), full, rtol=1e-12, atol=1e-14)


def test_unfinalized_outputs_refinalize_to_the_output():
    """do_finalize=False: summing w[t,j] * gemm2_output[idx[t*k+j]] over the pairs with
    idx >= 0, in j order, gives exactly the do_finalize=True accumulator; dropped pairs
    have idx -1 and zero activation rows."""
    inp, packed, lora = _routed_case(3, E_loc=4, E_glob=7, offset=1, T=6, k=3)
    args = (np_(inp["hidden"]), packed, np_(inp["w1"]), np_(inp["w2"]), 3)
    fin = orc.moe_lora_forward_routed(*args, num_experts=7, local_expert_offset=1, **lora)
    nf = orc.moe_lora_forward_routed(*args, num_experts=7, local_expert_offset=1, do_finalize=False, **lora)
    idx = nf["expanded_idx_to_permuted_idx"]
    w = nf["expert_weights"]
    acc = np.zeros_like(fin["out_acc"])
    for t in range(6):
        row = np.zeros(acc.shape[1])
        for j in range(3):
            if idx[t * 3 + j] >= 0:
                row = row + w[t, j] * nf["gemm2_output"][idx[t * 3 + j]]
        acc[t] = row
    np.testing.assert_array_equal(acc, fin["out_acc"])
    P_loc = int(fin["expert_offsets"][-1])
    assert sorted(idx[idx >= 0].tolist()) == list(range(P_loc))
    assert not np.any(nf["activation"][P_loc:])


def test_routed_all_local_equals_logit_routing():
    """All experts local and the packed routing taken from the logit routing with weights
    that bf16 holds exactly (constant logits, k = 2: ids 0 and 1, weights 1/2): the same
    outputs as the logit-routed layer, bit for bit."""
    cfg = wl.LayerConfig("rt1", T=4, H=16, I=8, E=4, top_k=2, ranks=(4,), scalings=(2.0,))
    inp = wl.make_inputs(cfg, seed=2)
    logits = np.zeros((4, 4))
    ids, w = orc.route(logits, 2)
    assert ids.tolist() == [[0, 1]] * 4 and w.tolist() == [[0.5, 0.5]] * 4
    lora = dict(lora_A_gu=np_(inp["lora_A_gu"]), lora_B_gu=np_(inp["lora_B_gu"]),
                lora_A_dn=np_(inp["lora_A_dn"]), lora_B_dn=np_(inp["lora_B_dn"]),
                slot_idx=inp["slot_idx"].numpy(), ranks=inp["ranks"], scalings=inp["scalings"])
    a = orc.moe_lora_forward(np_(inp["hidden"]), logits, np_(inp["w1"]), np_(inp["w2"]), 2, **lora)
    b = orc.moe_lora_forward_routed(np_(inp["hidden"]), orc.pack_topk(ids, w), np_(inp["w1"]), np_(inp["w2"]),
                                    2, num_experts=4, **lora)
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["perm"], b["perm"])


def test_token_subset_rows_equal_full_rows():
    cfg = wl.CONFIGS["tiny"]
    inp = wl.make_inputs(cfg, seed=5)
    full, _, _, _ = _run_both(inp)
    sub = orc.moe_lora_forward(np_(inp["hidden"]), np_(inp["router_logits"]), np_(inp["w1"]),
                               np_(inp["w2"]), cfg.top_k, lora_A_gu=np_(inp["lora_A_gu"]),
                               lora_B_gu=np_(inp["lora_B_gu"]), lora_A_dn=np_(inp["lora_A_dn"]),
                               lora_B_dn=np_(inp["lora_B_dn"]), slot_idx=inp["slot_idx"].numpy(),
                               ranks=inp["ranks"], scalings=inp["scalings"], tokens=[6, 1])
    np.testing.assert_array_equal(sub["out"], full["out"][[6, 1]])


def test_empty_batch():
    res = orc.moe_lora_forward(np.zeros((0, 64)), np.zeros((0, 4)), np.zeros((4, 128, 64)),
                               np.zeros((4, 64, 64)), 2)
    assert res["out"].shape == (0, 64) and res["perm"].size == 0
    assert (res["expert_offsets"] == 0).all()
