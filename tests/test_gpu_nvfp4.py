"""Parity of the NVFP4 path (through the C ABI) with the CPU oracle, on a GB300.

Bar: the row quantisation bit-exact (row scale, block scales, codes and the f16 values the
GEMMs read; both sides take the same float32 divisions and round-to-nearest-even
conversions); the grouped GEMM within the fp32 accumulation bound of exact products; the
layer output within the NVFP4 bounds of tests/gpu_helpers.py (the CPU test
test_oracle_nvfp4.py::test_nvfp4_tolerance_covers_rounding_flips derives them).
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
    """bf16 rows with magnitudes spread over many binades, an all-zero block, a block holding
    a single nonzero value and an all-zero row."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, K, generator=g) * torch.exp(torch.empty(T, 1).uniform_(-8, 8, generator=g))
    x[0, :16] = 0.0
    if T > 2:
        x[1, 16:32] = 0.0
        x[1, 20] = -3.5
        x[2, :] = 0.0
    return x.to(torch.bfloat16)


def _check_quant(got, rows_np):
    g, codes, sf, deq = (t.cpu().numpy() for t in got)
    q, sb, gr = orc.quant_act_nvfp4(rows_np)
    np.testing.assert_array_equal(g, gr)
    np.testing.assert_array_equal(orc.e4m3_decode(sf), sb)
    np.testing.assert_array_equal(orc.e2m1_decode(orc.unpack_nvfp4(codes)), q)
    np.testing.assert_array_equal(deq.astype(np.float64), q * np.repeat(sb, 16, axis=1))


@pytest.mark.parametrize("T,K,k", [(37, 384, 1), (64, 2048, 8), (5, 7168, 3)])
def test_quant_nvfp4_bit_exact(handle, T, K, k):
    src = _rows(T, K, T + K)
    src_np = src.float().numpy()
    _check_quant(pkg.moe_lora_quant_nvfp4(handle, src.cuda()), src_np)
    # gathered through a permutation of the expanded pairs (the permute + quant)
    perm = torch.randperm(T * k, generator=torch.Generator().manual_seed(K)).to(torch.int32)
    got = pkg.moe_lora_quant_nvfp4(handle, src.cuda(), perm.cuda(), k)
    torch.cuda.synchronize()
    _check_quant(got, src_np[perm.numpy() // k])


def _nvfp4_gemm_reference(wq, wsf, wgs, x, xgs, offsets):
    """Float64 product of the NVFP4 grouped GEMM from the packed codes (decoded by the oracle)
    and its bound: the products are exact, the tensor cores sum them in fp32 (relative error
    of a sum of K terms at most K * 2^-24 of its sum of |terms|, with a factor 2 of margin for
    the order of the partial sums), then two fp32 scalings."""
    E, N, K2 = wq.shape
    K = 2 * K2
    P = x.shape[0]
    ref = np.zeros((P, N))
    bnd = np.zeros((P, N))
    X = x.astype(np.float64)
    for e in range(E):
        q0, q1 = int(offsets[e]), int(offsets[e + 1])
        if q1 == q0:
            continue
        W = orc.dequant_weight_nvfp4(wq[e], wsf[e], 1.0)                 # e2m1 * e4m3, exact
        sc = xgs[q0:q1, None].astype(np.float64) * float(wgs[e])
        ref[q0:q1] = sc * (X[q0:q1] @ W.T)
        absp = np.abs(X[q0:q1]) @ np.abs(W).T
        bnd[q0:q1] = np.abs(sc) * absp * 2.0 * K * 2.0 ** -24 + 3 * 2.0 ** -24 * np.abs(ref[q0:q1]) + 1e-30
    return ref, bnd


@pytest.mark.parametrize("offsets", [[0, 17, 17, 60, 96, 130], [0, 20, 20, 27, 35, 40]],
                         ids=["wide-tiles", "narrow-tiles"])
def test_nvfp4_grouped_gemm_within_accumulation_bound(handle, offsets):
    """The NVFP4 grouped GEMM alone, element by element against the float64 product: random
    codes over all 16 values, random e4m3 block scales (subnormals included), five experts of
    ragged sizes with one empty, inputs from the quantiser.  The same data with the two nibbles
    of each byte swapped, or the block scales of neighbouring blocks swapped (plausible slips),
    lies far outside the bound.  130 pairs take the 64-token tcgen05 kernel; 40 pairs (an
    expert of 20: two 16-token tiles) the narrow-tile mma.sync kernel."""
    g = torch.Generator().manual_seed(321)
    E, N, K = 5, 384, 1024
    offsets = np.array(offsets, dtype=np.int32)
    P = int(offsets[-1])
    wq = torch.randint(0, 256, (E, N, K // 2), generator=g, dtype=torch.int32).to(torch.uint8)
    sf = torch.randint(0, 126, (E, N, K // 16), generator=g, dtype=torch.int32).to(torch.uint8)   # finite e4m3
    gs = torch.exp2(torch.empty(E).uniform_(-14, -6, generator=g)).float()
    src = _rows(P, K, 7)
    xgs, _, _, x = pkg.moe_lora_quant_nvfp4(handle, src.cuda())
    out = pkg.moe_lora_grouped_gemm_nvfp4(handle, wq.cuda(), sf.cuda(), gs.cuda(), x, xgs,
                                          torch.from_numpy(offsets).cuda())
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    xn, xgn = x.cpu().numpy(), xgs.cpu().numpy()
    ref, bnd = _nvfp4_gemm_reference(wq.numpy(), sf.numpy(), gs.numpy(), xn, xgn, offsets)
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert (err <= bnd).all(), (f"{int((err > bnd).sum())} of {err.size} outputs outside the bound, "
                                f"worst {float((err / bnd).max()):.3g}x")
    # the bound has teeth: swapped nibbles, swapped neighbouring block scales
    wq_s = ((wq.numpy() >> 4) | (wq.numpy() << 4)).astype(np.uint8)
    ref_s, _ = _nvfp4_gemm_reference(wq_s, sf.numpy(), gs.numpy(), xn, xgn, offsets)
    assert (np.abs(got - ref_s) > bnd).mean() > 0.5
    sf_s = sf.numpy().copy()
    sf_s[..., 0::2], sf_s[..., 1::2] = sf.numpy()[..., 1::2], sf.numpy()[..., 0::2]
    ref_t, _ = _nvfp4_gemm_reference(wq.numpy(), sf_s, gs.numpy(), xn, xgn, offsets)
    assert (np.abs(got - ref_t) > bnd).mean() > 0.5


def _nvfp4_weights(inp):
    w1 = wl.quantize_weights_nvfp4(inp["w1"].cuda())
    w2 = wl.quantize_weights_nvfp4(inp["w2"].cuda())
    return w1 + w2


def _forward_nvfp4(h, g, w4, flags=0, out=None, workspace=None, stream=None, outputs=None):
    w1q, w1s, w1g, w2q, w2s, w2g = w4
    return pkg.moe_lora_forward_nvfp4(
        h, g["hidden"], g["router_logits"], w1q, w1s, w1g, w2q, w2s, w2g, g["top_k"], routing_method=g["method"],
        correction_bias=g["correction_bias"], routed_scaling_factor=g["rsf"], lora_A_gu=g["lora_A_gu"],
        lora_B_gu=g["lora_B_gu"], lora_A_dn=g["lora_A_dn"], lora_B_dn=g["lora_B_dn"], slot_idx=g["slot_idx"],
        ranks=g["ranks"], scalings=g["scalings"], flags=flags, out=out, workspace=workspace, stream=stream,
        outputs=outputs)


def _oracle_nvfp4(inp, w4, tokens=None, lora_off=False):
    w1q, w1s, w1g, w2q, w2s, w2g = (t.cpu().numpy() for t in w4)
    np_ = gh.np_
    return orc.moe_lora_forward_nvfp4(
        np_(inp["hidden"]), np_(inp["router_logits"]), (w1q, w1s, w1g), (w2q, w2s, w2g), inp["top_k"], inp["method"],
        np_(inp["correction_bias"]), inp["rsf"], np_(inp["lora_A_gu"]), np_(inp["lora_B_gu"]),
        np_(inp["lora_A_dn"]), np_(inp["lora_B_dn"]), np_(inp["slot_idx"]), inp["ranks"], inp["scalings"],
        lora_off=lora_off, tokens=tokens, shared_outer=bool(inp.get("shared_outer", False)))


NVFP4_CASES = [
    # several slots of mixed rank, 10% of tokens without an adapter
    wl.LayerConfig("nv4_small", T=40, H=256, I=256, E=8, top_k=2, ranks=(8, 16), scalings=(2.0, 0.5),
                   slot_mode="uniform_none10"),
    # DeepSeekV3 routing, I = 64 (one K block in the down GEMM)
    wl.LayerConfig("nv4_dsv3", T=70, H=384, I=64, E=16, top_k=4, method=wl.DEEPSEEK_V3, bias_std=0.1, rsf=2.5,
                   ranks=(16,), scalings=(1.0,)),
    # 64-token tiles with a ragged tail (150 pairs per expert), rank not a multiple of 8
    wl.LayerConfig("nv4_tiles", T=300, H=256, I=128, E=4, top_k=2, ranks=(4, 12), scalings=(1.0, 2.0),
                   slot_mode="uniform_none10"),
    # the decode workload's shape
    wl.CONFIGS["decode"],
    # shared-outer adapter
    wl.LayerConfig("nv4_shared", T=48, H=256, I=256, E=8, top_k=4, ranks=(16, 8), scalings=(2.0, 1.0),
                   slot_mode="uniform_none10", shared_outer=True),
    # 16-token tiles (the narrow-tile kernel) with a shared-outer adapter of mixed ranks
    wl.LayerConfig("nv4_narrow_shared", T=24, H=256, I=256, E=16, top_k=4, ranks=(16, 8), scalings=(2.0, 1.0),
                   slot_mode="uniform_none10", shared_outer=True),
    # 16-token tiles, down-LoRA rows of 8 values (the expand's one-piece rows)
    wl.LayerConfig("nv4_narrow_r8", T=20, H=512, I=256, E=8, top_k=2, ranks=(8, 4), scalings=(1.0, 2.0),
                   slot_mode="uniform_none10"),
    # 16-token tiles, down-LoRA rows of 12 values (the expand's element-wise rows)
    wl.LayerConfig("nv4_narrow_r12", T=24, H=256, I=256, E=16, top_k=4, ranks=(4, 12), scalings=(2.0, 1.0),
                   slot_mode="uniform_none10"),
]


@pytest.mark.parametrize("cfg", NVFP4_CASES, ids=[c.name for c in NVFP4_CASES])
def test_nvfp4_layer_matches_oracle(handle, cfg):
    inp = wl.make_inputs(cfg, seed=11)
    g = gh.to_dev(inp)
    w4 = _nvfp4_weights(inp)
    flags = pkg.FLAG_SHARED_OUTER if cfg.shared_outer else 0
    outs = {n: torch.empty(shape, dtype=dt, device="cuda") for n, shape, dt in
            [("topk_ids", (cfg.T, cfg.top_k), torch.int32), ("expert_offsets", (cfg.E + 1,), torch.int32),
             ("perm", (cfg.P,), torch.int32)]}
    out = _forward_nvfp4(handle, g, w4, flags=flags, outputs=outs)
    torch.cuda.synchronize()
    ref = _oracle_nvfp4(inp, w4)
    np.testing.assert_array_equal(outs["topk_ids"].cpu().numpy(), ref["topk_ids"])
    np.testing.assert_array_equal(outs["perm"].cpu().numpy(), ref["perm"])
    gh.assert_close(out.float().cpu().numpy(), ref["out"], f"{cfg.name} nvfp4 output", gh.ATOL_NVFP4,
                    gh.RTOL_NVFP4, gh.REL_L2_NVFP4)


def test_nvfp4_layer_lora_off(handle):
    cfg = NVFP4_CASES[0]
    inp = wl.make_inputs(cfg, seed=3)
    w4 = _nvfp4_weights(inp)
    out = _forward_nvfp4(handle, gh.to_dev(inp), w4, flags=pkg.FLAG_LORA_OFF)
    torch.cuda.synchronize()
    ref = _oracle_nvfp4(inp, w4, lora_off=True)
    gh.assert_close(out.float().cpu().numpy(), ref["out"], "nvfp4 output without LoRA", gh.ATOL_NVFP4,
                    gh.RTOL_NVFP4, gh.REL_L2_NVFP4)


def test_nvfp4_empty_batch_launches_nothing(handle):
    cfg = wl.LayerConfig("nv4_empty", T=0, H=256, I=128, E=4, top_k=2)
    inp = wl.make_inputs(cfg, seed=0)
    n0 = handle.launch_count()
    out = _forward_nvfp4(handle, gh.to_dev(inp), _nvfp4_weights(wl.make_inputs(cfg, seed=0, T=1)))
    torch.cuda.synchronize()
    assert out.shape == (0, 256) and handle.launch_count() == n0


def test_nvfp4_graph_capture_and_replay(handle):
    """One capture, replayed with new hidden states in the captured buffers: each replay
    matches the oracle on those inputs, and an eager forward on them bit for bit."""
    cfg = wl.CONFIGS["decode"]
    inp = wl.make_inputs(cfg, seed=5)
    g = gh.to_dev(inp)
    w4 = _nvfp4_weights(inp)
    ws = pkg.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.S, cfg.R)
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _forward_nvfp4(handle, g, w4, out=out, workspace=ws, stream=s)   # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        _forward_nvfp4(handle, g, w4, out=out, workspace=ws, stream=s)
    for it in range(3):
        g["hidden"].copy_(torch.randn(cfg.T, cfg.H, generator=torch.Generator().manual_seed(it))
                          .to(torch.bfloat16).cuda())
        graph.replay()
        torch.cuda.synchronize()
        ref_inp = dict(inp)
        ref_inp["hidden"] = g["hidden"].cpu()
        ref = _oracle_nvfp4(ref_inp, w4)
        gh.assert_close(out.float().cpu().numpy(), ref["out"], f"nvfp4 replay {it}", gh.ATOL_NVFP4,
                        gh.RTOL_NVFP4, gh.REL_L2_NVFP4)
        eager = _forward_nvfp4(handle, g, w4)
        torch.cuda.synchronize()
        assert torch.equal(eager, out)
