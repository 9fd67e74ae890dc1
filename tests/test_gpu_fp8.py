"""Parity of the FP8 block-scale path (through the C ABI) with the CPU oracle, on a GB300.

Bar: the group quantisation's codes and scales bit-exact (both sides take the same
float32 division and round-to-nearest-even conversion); the layer output within
|gpu - ref| <= 3e-2 + 6e-2 |ref| elementwise and relative L2 <= 1.5e-2, three times the
bf16 bounds (tests/gpu_helpers.py gives the reason; the CPU test
test_oracle_fp8.py::test_fp8_tolerance_covers_accumulation_noise derives it).
"""
import numpy as np
import pytest
import torch

import routed_moe_expert_gb300 as pkg
from routed_moe_expert_gb300 import _build
from routed_moe_expert_gb300 import workloads as wl
from oracle import moe_lora_oracle as orc
import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    _build.build()
    torch.cuda.set_device(0)
    h = pkg.Handle(0)
    yield h
    h.close()


def _rows(T, K, seed):
    """bf16 rows with magnitudes spread over many binades, an all-zero group and a group
    holding a single nonzero value."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, K, generator=g) * torch.exp(torch.empty(T, 1).uniform_(-8, 8, generator=g))
    x[0, :128] = 0.0
    if T > 1:
        x[1, 128:256] = 0.0
        x[1, 200] = -3.5
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("T,K,k", [(37, 384, 1), (64, 2048, 8), (5, 7168, 3)])
def test_quant_fp8_bit_exact(handle, T, K, k):
    src = _rows(T, K, T + K)
    src_np = src.float().numpy()
    # plain rows
    codes, scales = pkg.moe_lora_quant_fp8(handle, src.cuda())
    torch.cuda.synchronize()
    q, s = orc.quant_act_fp8(src_np)
    np.testing.assert_array_equal(scales.cpu().numpy(), s.T)
    np.testing.assert_array_equal(orc.e4m3_decode(codes.cpu().numpy()), q)
    # gathered through a permutation of the expanded pairs (the permute + quant)
    perm = torch.randperm(T * k, generator=torch.Generator().manual_seed(K)).to(torch.int32)
    codes, scales = pkg.moe_lora_quant_fp8(handle, src.cuda(), perm.cuda(), k)
    torch.cuda.synchronize()
    rows = src_np[perm.numpy() // k]
    q, s = orc.quant_act_fp8(rows)
    np.testing.assert_array_equal(scales.cpu().numpy(), s.T)
    np.testing.assert_array_equal(orc.e4m3_decode(codes.cpu().numpy()), q)


def _fp8_weights(inp):
    w1q, w1s = wl.quantize_weights_fp8(inp["w1"].cuda())
    w2q, w2s = wl.quantize_weights_fp8(inp["w2"].cuda())
    return w1q, w1s, w2q, w2s


def _forward_fp8(h, g, w8, flags=0, out=None, workspace=None, stream=None, outputs=None):
    w1q, w1s, w2q, w2s = w8
    return pkg.moe_lora_forward_fp8(
        h, g["hidden"], g["router_logits"], w1q, w1s, w2q, w2s, g["top_k"], routing_method=g["method"],
        correction_bias=g["correction_bias"], routed_scaling_factor=g["rsf"], lora_A_gu=g["lora_A_gu"],
        lora_B_gu=g["lora_B_gu"], lora_A_dn=g["lora_A_dn"], lora_B_dn=g["lora_B_dn"], slot_idx=g["slot_idx"],
        ranks=g["ranks"], scalings=g["scalings"], flags=flags, out=out, workspace=workspace, stream=stream,
        outputs=outputs)


def _oracle_fp8(inp, w8, tokens=None, lora_off=False):
    w1q, w1s, w2q, w2s = (t.cpu().numpy() for t in w8)
    np_ = gh.np_
    return orc.moe_lora_forward_fp8(
        np_(inp["hidden"]), np_(inp["router_logits"]), w1q, w1s, w2q, w2s, inp["top_k"], inp["method"],
        np_(inp["correction_bias"]), inp["rsf"], np_(inp["lora_A_gu"]), np_(inp["lora_B_gu"]),
        np_(inp["lora_A_dn"]), np_(inp["lora_B_dn"]), np_(inp["slot_idx"]), inp["ranks"], inp["scalings"],
        lora_off=lora_off, tokens=tokens, shared_outer=bool(inp.get("shared_outer", False)))


FP8_CASES = [
    # several slots of mixed rank, 10% of tokens without an adapter
    wl.LayerConfig("f8_small", T=40, H=256, I=256, E=8, top_k=2, ranks=(8, 16), scalings=(2.0, 0.5),
                   slot_mode="uniform_none10"),
    # DeepSeekV3 routing, K of the down GEMM a single block
    wl.LayerConfig("f8_dsv3", T=70, H=384, I=128, E=16, top_k=4, method=wl.DEEPSEEK_V3, bias_std=0.1, rsf=2.5,
                   ranks=(16,), scalings=(1.0,)),
    # 64-token tiles with a ragged tail (150 pairs per expert), rank not a multiple of 8
    wl.LayerConfig("f8_tiles", T=300, H=256, I=128, E=4, top_k=2, ranks=(4, 12), scalings=(1.0, 2.0),
                   slot_mode="uniform_none10"),
    # the decode workload's shape
    wl.CONFIGS["decode"],
    # shared-outer adapter
    wl.LayerConfig("f8_shared", T=48, H=256, I=256, E=8, top_k=4, ranks=(16, 8), scalings=(2.0, 1.0),
                   slot_mode="uniform_none10", shared_outer=True),
]


@pytest.mark.parametrize("cfg", FP8_CASES, ids=[c.name for c in FP8_CASES])
def test_fp8_layer_matches_oracle(handle, cfg):
    inp = wl.make_inputs(cfg, seed=11)
    g = gh.to_dev(inp)
    w8 = _fp8_weights(inp)
    flags = pkg.FLAG_SHARED_OUTER if cfg.shared_outer else 0
    outs = {n: torch.empty(shape, dtype=dt, device="cuda") for n, shape, dt in
            [("topk_ids", (cfg.T, cfg.top_k), torch.int32), ("expert_offsets", (cfg.E + 1,), torch.int32),
             ("perm", (cfg.P,), torch.int32)]}
    out = _forward_fp8(handle, g, w8, flags=flags, outputs=outs)
    torch.cuda.synchronize()
    ref = _oracle_fp8(inp, w8)
    np.testing.assert_array_equal(outs["topk_ids"].cpu().numpy(), ref["topk_ids"])
    np.testing.assert_array_equal(outs["expert_offsets"].cpu().numpy(), ref["expert_offsets"])
    np.testing.assert_array_equal(outs["perm"].cpu().numpy(), ref["perm"])
    gh.assert_close(out.float().cpu().numpy(), ref["out"], f"{cfg.name} fp8 output", gh.ATOL_FP8, gh.RTOL_FP8,
                    gh.REL_L2_FP8)


# The accumulation model of the FP8 GEMM (gpu_helpers.FP8_ACC_BITS): exact e4m3 products, each
# 128-wide block summed as a tree of depth 7 with at least FP8_ACC_BITS significant bits
# (error <= 7 * 2^-FP8_ACC_BITS * sum of |products|), block sums scaled and added in fp32.
FP8_ACC_BITS = gh.FP8_ACC_BITS


def _fp8_gemm_reference(wq, ws, xq, xs, offsets):
    """Float64 block-scaled product of the FP8 grouped GEMM and its error bound under the
    accumulation model above, from the e4m3 codes (decoded by the oracle's decoder)."""
    E, N, K = wq.shape
    P = xq.shape[0]
    KB = K // 128
    W = orc.e4m3_decode(wq).astype(np.float64)
    X = orc.e4m3_decode(xq).astype(np.float64)
    ref = np.zeros((P, N))
    bnd = np.zeros((P, N))
    for e in range(E):
        q0, q1 = int(offsets[e]), int(offsets[e + 1])
        if q1 == q0:
            continue
        xe = X[q0:q1]
        scaled_abs = np.zeros((q1 - q0, N))
        for b in range(KB):
            kb = slice(128 * b, 128 * b + 128)
            part = xe[:, kb] @ W[e, :, kb].T                              # exact block sums
            absp = np.abs(xe[:, kb]) @ np.abs(W[e, :, kb]).T             # sums of |products|
            sc = xs[b, q0:q1][:, None].astype(np.float64) * np.repeat(ws[e, :, b], 128)[None, :]
            ref[q0:q1] += sc * part
            bnd[q0:q1] += np.abs(sc) * absp * 7.0 * 2.0 ** -FP8_ACC_BITS
            scaled_abs += np.abs(sc * part)
        bnd[q0:q1] += (KB + 2) * 2.0 ** -24 * scaled_abs + 1e-30
    return ref, bnd


def test_fp8_grouped_gemm_within_accumulation_bound(handle):
    """The FP8 grouped GEMM alone (moe_lora_grouped_gemm_fp8), element by element against the
    float64 block-scaled product: random e4m3 codes over the whole finite range (subnormals
    included), random block scales, five experts of ragged sizes with one empty; every output
    within the bound of the accumulation model (FP8_ACC_BITS).  The same data with the weight
    block scales read transposed (a plausible indexing slip) lies far outside that bound."""
    g = torch.Generator().manual_seed(123)
    E, N, K, P = 5, 384, 1024, 130
    offsets = np.array([0, 17, 17, 60, 96, 130], dtype=np.int32)

    def codes(shape):
        c = torch.randint(0, 256, shape, generator=g, dtype=torch.int32)
        c = torch.where((c & 0x7F) == 0x7F, c - 1, c)   # no NaN codes
        return c.to(torch.uint8)

    wq, xq = codes((E, N, K)), codes((P, K))
    ws = torch.exp2(torch.empty((E, N // 128, K // 128)).uniform_(-12, -2, generator=g)).float()
    xs = torch.exp2(torch.empty((K // 128, P)).uniform_(-10, 0, generator=g)).float()
    out = pkg.moe_lora_grouped_gemm_fp8(handle, wq.cuda(), ws.cuda(), xq.cuda(), xs.cuda(),
                                        torch.from_numpy(offsets).cuda())
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    ref, bnd = _fp8_gemm_reference(wq.numpy(), ws.numpy(), xq.numpy(), xs.numpy(), offsets)
    err = np.abs(got - ref)
    worst = float((err / bnd).max())
    assert np.isfinite(got).all()
    assert (err <= bnd).all(), f"{int((err > bnd).sum())} of {err.size} outputs outside the bound, worst {worst:.3g}x"
    # the bound has teeth: a transposed block-scale index is caught
    ws_t = ws.numpy().copy()
    ws_t[:, :, :3] = ws_t[:, :, :3][:, ::-1, :]
    ref_t, _ = _fp8_gemm_reference(wq.numpy(), ws_t, xq.numpy(), xs.numpy(), offsets)
    assert (np.abs(got - ref_t) > bnd).mean() > 0.5


def test_fp8_layer_lora_off(handle):
    cfg = FP8_CASES[0]
    inp = wl.make_inputs(cfg, seed=3)
    w8 = _fp8_weights(inp)
    out = _forward_fp8(handle, gh.to_dev(inp), w8, flags=pkg.FLAG_LORA_OFF)
    torch.cuda.synchronize()
    ref = _oracle_fp8(inp, w8, lora_off=True)
    gh.assert_close(out.float().cpu().numpy(), ref["out"], "fp8 output without LoRA", gh.ATOL_FP8, gh.RTOL_FP8,
                    gh.REL_L2_FP8)


def test_fp8_empty_batch_launches_nothing(handle):
    cfg = wl.LayerConfig("f8_empty", T=0, H=256, I=128, E=4, top_k=2)
    inp = wl.make_inputs(cfg, seed=0)
    n0 = handle.launch_count()
    out = _forward_fp8(handle, gh.to_dev(inp), _fp8_weights(wl.make_inputs(cfg, seed=0, T=1)))
    torch.cuda.synchronize()
    assert out.shape == (0, 256) and handle.launch_count() == n0


def test_fp8_graph_capture_and_replay(handle):
    """One capture, replayed with new hidden states in the captured buffers: each replay
    matches the oracle on those inputs, and an eager forward on them bit for bit."""
    cfg = wl.CONFIGS["decode"]
    inp = wl.make_inputs(cfg, seed=5)
    g = gh.to_dev(inp)
    w8 = _fp8_weights(inp)
    ws = pkg.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.S, cfg.R)
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _forward_fp8(handle, g, w8, out=out, workspace=ws, stream=s)   # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        _forward_fp8(handle, g, w8, out=out, workspace=ws, stream=s)
    for it in range(3):
        # fresh hidden states of the workload's distribution, N(0, 1): the FP8 bounds are
        # derived for it (larger inputs raise the absolute error floor with them)
        g["hidden"].copy_(torch.randn(cfg.T, cfg.H, generator=torch.Generator().manual_seed(it))
                          .to(torch.bfloat16).cuda())
        graph.replay()
        torch.cuda.synchronize()
        ref_inp = dict(inp)
        ref_inp["hidden"] = g["hidden"].cpu()
        gh.assert_close(out.float().cpu().numpy(), _oracle_fp8(ref_inp, w8)["out"], f"replay {it}", gh.ATOL_FP8,
                        gh.RTOL_FP8, gh.REL_L2_FP8)
        eager = _forward_fp8(handle, g, w8)
        torch.cuda.synchronize()
        assert torch.equal(out, eager)


FP8_FUSED_CASES = [
    # four slots of mixed rank, 64-token tiles
    wl.LayerConfig("f8f_four", T=96, H=512, I=256, E=16, top_k=4, ranks=(8, 16, 32, 64),
                   scalings=(2.0, 1.0, 0.5, 0.25), slot_mode="uniform_none10"),
    # shared-outer, 32-token tiles
    wl.LayerConfig("f8f_shared", T=64, H=512, I=256, E=16, top_k=4, ranks=(8, 32), scalings=(2.0, 0.5),
                   slot_mode="uniform_none10", shared_outer=True),
    # a disabled slot and a rank-0 slot; 256-token tiles are capped at 64 on the FP8 path
    wl.LayerConfig("f8f_disabled", T=600, H=256, I=128, E=8, top_k=2, ranks=(16, 24, 0, 8),
                   scalings=(1.0, 0.0, 1.0, 2.0), slot_mode="uniform_none10"),
    # the multi-adapter workload's shape
    wl.CONFIGS["multi_slot"],
]


@pytest.mark.parametrize("cfg", FP8_FUSED_CASES, ids=[c.name for c in FP8_FUSED_CASES])
def test_fp8_fused_lora_with_packed_b_matches_oracle(handle, cfg):
    """With both expand-ready LoRA B copies the FP8 layer runs the fused LoRA placement (the
    tensor-core shrinks and bf16 LoRA K-stages inside the FP8 GEMMs): against the FP8 oracle,
    and against the side-stream placement of the same layer."""
    inp = wl.make_inputs(cfg, seed=13)
    g = gh.to_dev(inp)
    w8 = _fp8_weights(inp)
    flags = pkg.FLAG_SHARED_OUTER if cfg.shared_outer else 0
    bgu = pkg.moe_lora_pack_lora_b(handle, g["lora_B_gu"], g["ranks"], 1)
    bdn = pkg.moe_lora_pack_lora_b(handle, g["lora_B_dn"], g["ranks"], 0)
    ws = pkg.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.S, cfg.R)
    w1q, w1s, w2q, w2s = w8
    kw = dict(routing_method=g["method"], correction_bias=g["correction_bias"], routed_scaling_factor=g["rsf"],
              lora_A_gu=g["lora_A_gu"], lora_B_gu=g["lora_B_gu"], lora_A_dn=g["lora_A_dn"],
              lora_B_dn=g["lora_B_dn"], slot_idx=g["slot_idx"], ranks=g["ranks"], scalings=g["scalings"],
              flags=flags, workspace=ws)
    agu = pkg.moe_lora_pack_lora_a(handle, g["lora_A_gu"], g["ranks"])
    adn = pkg.moe_lora_pack_lora_a(handle, g["lora_A_dn"], g["ranks"])
    n0 = handle.launch_count()
    out = pkg.moe_lora_forward_fp8(handle, g["hidden"], g["router_logits"], w1q, w1s, w2q, w2s, g["top_k"],
                                   lora_B_gu_packed=bgu, lora_B_dn_packed=bdn, lora_A_gu_packed=agu,
                                   lora_A_dn_packed=adn, **kw)
    torch.cuda.synchronize()
    n1 = handle.launch_count()
    st, word = pkg.moe_lora_check_status(ws)
    assert st == 0, f"device status {word:#x}"
    # route, permute + quant, bf16 permute, shrink, gate_up, activation, shrink, quant, down, finalize
    assert n1 - n0 == 10
    ref = _oracle_fp8(inp, w8)
    gh.assert_close(out.float().cpu().numpy(), ref["out"], f"{cfg.name} fused fp8", gh.ATOL_FP8, gh.RTOL_FP8,
                    gh.REL_L2_FP8)
    side = pkg.moe_lora_forward_fp8(handle, g["hidden"], g["router_logits"], w1q, w1s, w2q, w2s, g["top_k"], **kw)
    torch.cuda.synchronize()
    # the two placements share the base GEMMs and differ only in the LoRA sums' order: they
    # agree within the FP8 elementwise bounds and the bf16 relative L2 bound
    gh.assert_close(out.float().cpu().numpy(), side.float().cpu().numpy(), f"{cfg.name} fused vs side-stream",
                    gh.ATOL_FP8, gh.RTOL_FP8, gh.REL_L2)
