"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on a GB300.

Bar: topk_ids, expert_offsets, perm and inv_perm bit-exact; the layer output within
|gpu - ref| <= 1e-2 + 2e-2 |ref| elementwise and relative L2 <= 5e-3.
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


def _check_routing(out, ref, E, T, k):
    ids, w = ref["topk_ids"], ref["topk_weights"]
    np.testing.assert_array_equal(out["topk_ids"].cpu().numpy(), ids)
    np.testing.assert_array_equal(out["expert_offsets"].cpu().numpy(), ref["expert_offsets"])
    np.testing.assert_array_equal(out["perm"].cpu().numpy(), ref["perm"])
    np.testing.assert_array_equal(out["inv_perm"].cpu().numpy(), ref["inv"])
    np.testing.assert_allclose(out["topk_weights"].cpu().numpy(), w, rtol=2e-6, atol=1e-7)


# ------------------------------------------------------------------------ routing

ROUTE_CASES = [
    # T, E, k, method, logit scale (small scale -> many bf16 ties)
    (1, 8, 1, 0, 1.0), (7, 8, 2, 0, 1.0), (64, 128, 8, 0, 1.0), (256, 128, 8, 0, 0.05),
    (300, 100, 5, 0, 1.0), (8192, 128, 8, 0, 1.0), (50, 20, 20, 0, 1.0), (33, 1000, 32, 0, 0.02),
    (128, 384, 8, 1, 1.0), (4096, 384, 8, 1, 1.0), (200, 257, 6, 1, 0.01), (5000, 64, 4, 1, 3.0),
]


@pytest.mark.parametrize("T,E,k,method,scale", ROUTE_CASES)
def test_route_bit_exact(handle, T, E, k, method, scale):
    g = torch.Generator().manual_seed(T * 7 + E)
    logits = (torch.randn(T, E, generator=g) * scale).to(torch.bfloat16)
    logits[0, :] = 0.0                                   # a row of ties
    if T > 2:
        logits[1, E // 2] = float("nan")                 # a NaN logit never wins
    if T > 3:
        logits[2, :] = -0.0                              # -0 and +0 tie: lower ids win
        logits[2, 1::3] = 0.0
    bias = (torch.randn(E, generator=g) * 0.1).float() if method == 1 else None
    rsf = 2.827 if method == 1 else 1.0
    out = pkg.moe_lora_route(handle, logits.cuda(), k, method, None if bias is None else bias.cuda(), rsf)
    torch.cuda.synchronize()
    ids, w = orc.route(logits.float().numpy(), k, method, None if bias is None else bias.numpy(), rsf)
    off, perm, inv = orc.align(ids, E)
    _check_routing(out, dict(topk_ids=ids, topk_weights=w, expert_offsets=off, perm=perm, inv=inv), E, T, k)
    st, word = pkg.moe_lora_check_status(out["workspace"])
    assert st == 0, hex(word)


def test_route_zipf_prefill_bit_exact(handle):
    cfg = wl.CONFIGS["prefill_zipf"]
    inp = wl.make_inputs(cfg, seed=0, device="cuda")
    out = pkg.moe_lora_route(handle, inp["router_logits"], cfg.top_k)
    torch.cuda.synchronize()
    ids, w = orc.route(inp["router_logits"].float().cpu().numpy(), cfg.top_k)
    off, perm, inv = orc.align(ids, cfg.E)
    _check_routing(out, dict(topk_ids=ids, topk_weights=w, expert_offsets=off, perm=perm, inv=inv),
                   cfg.E, cfg.T, cfg.top_k)
    load = np.diff(off)
    assert load.max() > 4 * load.mean()                   # the skew is really there


def test_permute_exact(handle):
    g = torch.Generator().manual_seed(3)
    T, H, k, E = 37, 2048, 4, 16
    hidden = torch.randn(T, H, generator=g).to(torch.bfloat16).cuda()
    logits = torch.randn(T, E, generator=g).to(torch.bfloat16).cuda()
    r = pkg.moe_lora_route(handle, logits, k)
    xp = pkg.moe_lora_permute(handle, hidden, r["perm"], k)
    torch.cuda.synchronize()
    expect = hidden[(r["perm"].long() // k)]
    assert torch.equal(xp, expect)


# ------------------------------------------------------------------------ layer

def _run_and_check(h, cfg, seed=0, device_inputs=False, tokens=None, flags=0, lora_off=False, T=None):
    inp = wl.make_inputs(cfg, seed=seed, device="cuda" if device_inputs else "cpu", T=T)
    return _check_given_inputs(h, cfg, inp, device_inputs, tokens, flags, lora_off)


def _check_given_inputs(h, cfg, inp, device_inputs=False, tokens=None, flags=0, lora_off=False):
    g = gh.to_dev(inp)
    P = g["T"] * cfg.top_k
    outs = dict(topk_ids=torch.empty((g["T"], cfg.top_k), dtype=torch.int32, device="cuda"),
                topk_weights=torch.empty((g["T"], cfg.top_k), dtype=torch.float32, device="cuda"),
                expert_offsets=torch.empty((cfg.E + 1,), dtype=torch.int32, device="cuda"),
                perm=torch.empty((P,), dtype=torch.int32, device="cuda"),
                inv_perm=torch.empty((P,), dtype=torch.int32, device="cuda"))
    ws = pkg.alloc_workspace(g["T"], cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.S, cfg.R)
    out = gh.forward(h, g, flags=flags, outputs=outs, workspace=ws)
    torch.cuda.synchronize()
    st, word = pkg.moe_lora_check_status(ws)
    assert st == 0, f"device status {word:#x}"
    ref = gh.oracle(inp, tokens=tokens, lora_off=lora_off, lazy=device_inputs)
    _check_routing(outs, ref, cfg.E, g["T"], cfg.top_k)
    got = out.float().cpu().numpy()
    if tokens is not None:
        got = got[tokens]
    return gh.assert_close(got, ref["out"], cfg.name), inp, out


def test_tiny_layer(handle):
    _run_and_check(handle, wl.CONFIGS["tiny"])


@pytest.mark.parametrize("seed", range(16))
def test_random_small_layers(handle, seed):
    rng = np.random.default_rng(1000 + seed)
    base = wl.random_small_config(rng, max_T=40, max_E=12)
    H = int(rng.choice([64, 128, 256, 512]))
    I = int(rng.choice([64, 128, 192, 320]))
    cfg = wl.LayerConfig("rand", T=base.T, H=H, I=I, E=base.E, top_k=base.top_k, method=base.method,
                         ranks=tuple(min(r, 16) for r in base.ranks), scalings=base.scalings,
                         slot_mode="uniform_none10", bias_std=0.1, rsf=base.rsf)
    _run_and_check(handle, cfg, seed=seed)


@pytest.mark.parametrize("T,E,k", [(40, 8, 4), (130, 8, 4), (260, 8, 4), (520, 8, 4), (1500, 6, 3)])
def test_token_tile_widths_and_ragged_tails(handle, T, E, k):
    """T*k/E pairs per expert of about 20, 65, 130, 260, 750 select token tiles of
    32, 128, 256, 256 (several per expert) with ragged tails; at 256-token tiles the fused
    gate_up puts each tile's LoRA delta in the idle accumulator; from 128-token tiles on the
    down GEMM hands y to the finalize in bf16."""
    cfg = wl.LayerConfig("tiles", T=T, H=256, I=192, E=E, top_k=k, ranks=(8, 16), scalings=(1.0, 0.5),
                         slot_mode="uniform_none10")
    _run_and_check(handle, cfg, seed=T)


@pytest.mark.parametrize("T,E,k,ranks,flags", [
    (100, 8, 4, (8, 16), 0),                    # 128-token tiles, fused LoRA, two accumulators + two deltas
    (520, 8, 4, (8, 16), 0),                    # 256-token tiles: the delta in the idle accumulator
    (520, 8, 4, (8, 16), pkg.FLAG_LORA_OFF),    # 256-token tiles, activation epilogue, plain down
    (1500, 6, 3, (8, 16, 32, 64), 0),           # several tiles per expert, four slots, ragged tails
])
def test_cta_pair_tiles(handle, T, E, k, ranks, flags):
    """Wide token tiles on CTA pairs (I and H multiples of 128 and 256): each tile's weight
    rows span two CTAs of a cluster, each loading half the token rows."""
    cfg = wl.LayerConfig("pair", T=T, H=512, I=256, E=E, top_k=k, ranks=ranks,
                         scalings=tuple(1.0 / (i + 1) for i in range(len(ranks))), slot_mode="uniform_none10")
    _run_and_check(handle, cfg, seed=T + flags, flags=flags, lora_off=bool(flags & pkg.FLAG_LORA_OFF))


@pytest.mark.parametrize("T,H,I,E,k", [
    (520, 384, 192, 8, 4),    # neither GEMM can pair (2I/128 and H/128 odd): single-CTA wide tiles
    (64, 512, 256, 2, 2),     # pair tiles, far fewer tiles than clusters
    (300, 640, 256, 4, 3),    # gate_up on pairs, down on single CTAs (H/128 = 5 weight tiles)
])
def test_wide_tiles_with_and_without_pairs(handle, T, H, I, E, k):
    """Wide token tiles where the CTA-pair path does not apply (or leaves most clusters
    idle) give the same results as the oracle."""
    for flags in (0, pkg.FLAG_LORA_OFF):
        cfg = wl.LayerConfig("wide", T=T, H=H, I=I, E=E, top_k=k, ranks=(8, 16), scalings=(1.0, 0.5),
                             slot_mode="uniform_none10")
        _run_and_check(handle, cfg, seed=T + H + flags, flags=flags, lora_off=bool(flags & pkg.FLAG_LORA_OFF))


def test_decode_config_full(handle):
    _run_and_check(handle, wl.CONFIGS["decode"], device_inputs=True)


def test_multi_slot_config_full(handle):
    (err, rel), inp, out = _run_and_check(handle, wl.CONFIGS["multi_slot"], device_inputs=True)


def test_prefill_zipf_sampled(handle):
    cfg = wl.CONFIGS["prefill_zipf"]
    inp = wl.make_inputs(cfg, seed=0, device="cuda")
    ids, _ = orc.route(inp["router_logits"].float().cpu().numpy(), cfg.top_k)
    tokens = gh.sample_tokens(ids, cfg.E, every=128, extremes=3, per_expert=16)
    _run_and_check(handle, cfg, device_inputs=True, tokens=tokens)


@pytest.mark.parametrize("name", ["kimi_decode", "kimi_prefill"])
def test_kimi_sampled(handle, name):
    cfg = wl.CONFIGS[name]
    inp = wl.make_inputs(cfg, seed=0, device="cuda")
    ids, _ = orc.route(inp["router_logits"].float().cpu().numpy(), cfg.top_k, 1,
                       inp["correction_bias"].cpu().numpy(), cfg.rsf)
    tokens = gh.sample_tokens(ids, cfg.E, every=max(cfg.T // 12, 1), extremes=1, per_expert=4)
    del inp
    torch.cuda.empty_cache()
    _run_and_check(handle, cfg, device_inputs=True, tokens=tokens)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("flags", [0, 8], ids=["fused", "unfused"])   # 8 = FLAG_UNFUSED_LORA
def test_both_lora_placements_match_oracle(handle, flags):
    """Down-LoRA expand inside the down GEMM (default at ranks that are multiples of 8) and
    in its epilogue, both against the oracle, with four slots of mixed rank, a 10%
    no-adapter share and the NaN-filled rank tails."""
    cfg = wl.LayerConfig("place", T=96, H=512, I=256, E=16, top_k=4, ranks=(8, 16, 32, 64),
                         scalings=(2.0, 1.0, 0.5, 0.25), slot_mode="uniform_none10")
    _run_and_check(handle, cfg, seed=21, flags=flags)


@pytest.mark.parametrize("T,E,k,flags", [(64, 16, 4, 0), (64, 16, 4, 8), (256, 8, 4, 0), (600, 8, 2, 0)],
                         ids=["narrow", "narrow-unfused", "wide-fused", "wide-256"])
def test_shared_outer_lora_matches_oracle(handle, T, E, k, flags):
    """Shared-outer LoRA (one A_gu and one B_dn per slot for every expert) on each LoRA
    placement: the narrow-tile side-stream chain, the unfused placement, and the fused
    tensor-core shrink with LoRA K-stages at 32- and 256-token tiles."""
    cfg = wl.LayerConfig("so", T=T, H=512, I=256, E=E, top_k=k, ranks=(8, 32), scalings=(2.0, 0.5),
                         slot_mode="uniform_none10", shared_outer=True)
    _run_and_check(handle, cfg, seed=T + flags, flags=flags | pkg.FLAG_SHARED_OUTER)


@pytest.mark.parametrize("T,E,k,ranks,shared", [(64, 128, 8, (16,), False), (40, 16, 4, (8, 16, 4), False),
                                                 (64, 32, 4, (16, 8), True)],
                         ids=["decode-shape", "mixed-ranks", "shared-outer"])
def test_down_lora_on_side_stream_matches_oracle(handle, T, E, k, ranks, shared):
    """MOE_LORA_FLAG_DOWN_LORA_SIDE: on the side-stream placement the down LoRA (shrink and
    expand into a bf16 delta per pair) runs beside the down GEMM and the finalize adds it;
    the layer still matches the oracle, eagerly and under CUDA-graph replay."""
    cfg = wl.LayerConfig("dnside", T=T, H=512 if T < 64 else 2048, I=256 if T < 64 else 768, E=E, top_k=k,
                         ranks=ranks, scalings=tuple(1.0 / (i + 1) for i in range(len(ranks))),
                         slot_mode="uniform_none10", shared_outer=shared)
    inp = wl.make_inputs(cfg, seed=T + E)
    g = gh.to_dev(inp)
    flags = pkg.FLAG_DOWN_LORA_SIDE | (pkg.FLAG_SHARED_OUTER if shared else 0)
    ws = pkg.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.S, cfg.R)
    out = gh.forward(handle, g, flags=flags, workspace=ws)
    torch.cuda.synchronize()
    assert pkg.moe_lora_check_status(ws)[0] == 0
    ref = gh.oracle(inp)["out"]
    gh.assert_close(out.float().cpu().numpy(), ref, "down LoRA on the side stream")
    # the same forward captured once and replayed
    out2 = torch.empty_like(out)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gh.forward(handle, g, flags=flags, out=out2, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        gh.forward(handle, g, flags=flags, out=out2, workspace=ws, stream=s)
    out2.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out2, out)


def test_lora_off_matches_oracle_base(handle):
    cfg = wl.LayerConfig("off", T=48, H=256, I=128, E=8, top_k=2, ranks=(8,), scalings=(2.0,))
    _run_and_check(handle, cfg, flags=pkg.FLAG_LORA_OFF, lora_off=True)


def test_no_adapter_tokens_equal_lora_off_bitwise(handle):
    cfg = wl.LayerConfig("none", T=64, H=256, I=128, E=8, top_k=2, ranks=(8, 4), scalings=(2.0, 0.0),
                         slot_mode="uniform_none10")
    g = gh.to_dev(wl.make_inputs(cfg, seed=5))
    base = gh.forward(handle, g, flags=pkg.FLAG_LORA_OFF).clone()
    g["slot_idx"] = torch.full_like(g["slot_idx"], -1)
    none = gh.forward(handle, g).clone()
    g["slot_idx"] = torch.ones_like(g["slot_idx"])       # slot 1 has scaling 0
    zero = gh.forward(handle, g).clone()
    torch.cuda.synchronize()
    assert torch.equal(base, none) and torch.equal(base, zero)


def test_single_and_two_stream_agree_bitwise(handle):
    cfg = wl.CONFIGS["multi_slot"]
    cfg = wl.LayerConfig("ms", T=200, H=512, I=256, E=16, top_k=4, ranks=cfg.ranks, scalings=cfg.scalings,
                         slot_mode="uniform_none10")
    g = gh.to_dev(wl.make_inputs(cfg, seed=9))
    one = gh.forward(handle, g, flags=pkg.FLAG_FORCE_SINGLE_STREAM).clone()
    two = gh.forward(handle, g, flags=pkg.FLAG_FORCE_TWO_STREAM).clone()
    dflt = gh.forward(handle, g).clone()
    torch.cuda.synchronize()
    assert torch.equal(one, two) and torch.equal(one, dflt)


def test_launch_count_per_forward(handle):
    """One forward launches the kernels its placement draws: narrow tiles with LoRA = route,
    side-stream LoRA, permute, gate_up GEMM, activation + down shrink, down GEMM, finalize;
    LoRA off drops the LoRA kernel and fuses nothing else; wide tiles = route, permute with
    the gate_up shrink, gate_up GEMM, tensor-core down shrink, down GEMM, finalize, with the
    gate_up shrink as its own kernel after a plain permute when many ranks are stacked; the
    down LoRA on the side stream replaces the activation + down shrink kernel by a plain
    activation and one side-stream LoRA kernel."""
    narrow = wl.LayerConfig("n", T=64, H=256, I=128, E=32, top_k=4, ranks=(8,), scalings=(1.0,))
    wide = wl.LayerConfig("w", T=256, H=256, I=128, E=8, top_k=4, ranks=(8,), scalings=(1.0,))
    wide_many = wl.LayerConfig("wm", T=256, H=256, I=128, E=8, top_k=4, ranks=(8, 16, 32, 64),
                               scalings=(1.0, 1.0, 1.0, 1.0))
    for cfg, flags, want in ((narrow, 0, 7), (narrow, pkg.FLAG_LORA_OFF, 6), (wide, 0, 6), (wide_many, 0, 7),
                             (narrow, pkg.FLAG_DOWN_LORA_SIDE, 8)):
        g = gh.to_dev(wl.make_inputs(cfg, seed=1))
        n0 = handle.launch_count()
        gh.forward(handle, g, flags=flags)
        torch.cuda.synchronize()
        assert handle.launch_count() - n0 == want, (cfg.name, flags)


def test_slot_out_of_range_reported(handle):
    cfg = wl.LayerConfig("bad", T=16, H=128, I=64, E=4, top_k=2, ranks=(4,), scalings=(1.0,))
    inp = wl.make_inputs(cfg, seed=1)
    g = gh.to_dev(inp)
    g["slot_idx"][3] = 7                                   # S = 1
    ws = pkg.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.S, cfg.R)
    gh.forward(handle, g, workspace=ws)
    st, word = pkg.moe_lora_check_status(ws)
    assert st == 6 and (word & 0xff) == 6
    # the next good call on the same workspace reports OK again
    g["slot_idx"][3] = 0
    gh.forward(handle, g, workspace=ws)
    assert pkg.moe_lora_check_status(ws)[0] == 0


@pytest.mark.parametrize("T,E", [(64, 32), (256, 16)], ids=["narrow-two-stream", "wide-cta-pairs"])
def test_back_to_back_forwards_share_a_workspace(handle, T, E):
    """Three forwards enqueued on one stream and one workspace with no sync between them.
    Each routing cluster starts behind the previous forward's finalize (a programmatic
    launch), so it must not disturb the routing buffers that finalize still reads."""
    cfg = wl.LayerConfig("b2b", T=T, H=512, I=256, E=E, top_k=4, ranks=(8, 16), scalings=(1.0, 0.5),
                         slot_mode="uniform_none10")
    ins = [wl.make_inputs(cfg, seed=s) for s in (31, 32, 33)]
    gs = [gh.to_dev(i) for i in ins]
    ws = pkg.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.S, cfg.R)
    outs = [torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda") for _ in gs]
    for g, o in zip(gs, outs):
        gh.forward(handle, g, out=o, workspace=ws)
    st, word = pkg.moe_lora_check_status(ws)
    assert st == 0, f"device status {word:#x}"
    for i, (inp, o) in enumerate(zip(ins, outs)):
        gh.assert_close(o.float().cpu().numpy(), gh.oracle(inp)["out"], f"forward {i}")


@pytest.mark.parametrize("T,E", [(64, 32), (96, 16), (200, 16), (520, 8), (1024, 8)],
                         ids=["narrow", "wide-32", "wide-cta-pairs", "wide-256", "cooperative-routing"])
def test_programmatic_launches_change_nothing(handle, T, E):
    """The programmatic launch chain only moves kernel start times: with MOE_LORA_FLAG_NO_PDL
    (plain stream order, the header memset before the routing) every output is bitwise the
    same, on every placement and both routing paths."""
    cfg = wl.LayerConfig("pdl", T=T, H=512, I=256, E=E, top_k=4, ranks=(8, 16), scalings=(1.0, 0.5),
                         slot_mode="uniform_none10")
    g = gh.to_dev(wl.make_inputs(cfg, seed=T))
    ws = pkg.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.S, cfg.R)
    a = gh.forward(handle, g, workspace=ws).clone()
    b = gh.forward(handle, g, workspace=ws, flags=pkg.FLAG_NO_PDL).clone()
    c = gh.forward(handle, g, workspace=ws).clone()
    assert pkg.moe_lora_check_status(ws)[0] == 0
    assert torch.equal(a, b) and torch.equal(a, c)


def test_fused_gate_up_tiles_with_and_without_lora(handle):
    """256-token fused gate_up tiles, some of whose pairs all lack an adapter (first half of
    the tokens on slot -1, so an expert's first tile holds no LoRA pair and its last tile
    does): tiles without a delta skip the merge into the idle accumulator, tiles with one
    merge it, in any order on a CTA."""
    cfg = wl.LayerConfig("mixed", T=2048, H=512, I=256, E=4, top_k=2, ranks=(8, 16), scalings=(1.0, 0.5),
                         slot_mode="uniform_none10")
    inp = wl.make_inputs(cfg, seed=21)
    inp["slot_idx"][: cfg.T // 2] = -1
    _check_given_inputs(handle, cfg, inp)


def test_empty_batch(handle):
    cfg = wl.LayerConfig("empty", T=0, H=128, I=64, E=4, top_k=2, ranks=(4,), scalings=(1.0,))
    g = gh.to_dev(wl.make_inputs(cfg, seed=1))
    out = gh.forward(handle, g)
    torch.cuda.synchronize()
    assert out.shape == (0, 128)


@pytest.mark.parametrize("T", [64, 520], ids=["two-stream-narrow", "wide-cta-pairs"])
def test_graph_capture_and_replay(handle, T):
    """Capture the forward once, replay with new inputs and slot maps; every replay must
    match the oracle (regression for the capture-time allocation race of sglang PR #28091,
    Motivation 3).  At 64 tokens the forward forks the side stream; at 520 tokens both GEMMs
    run on CTA pairs (cluster launches) with the fused LoRA stages."""
    cfg = wl.LayerConfig("graph", T=T, H=512, I=256, E=16 if T == 64 else 8, top_k=4, ranks=(8, 16, 32, 4) if T == 64 else (8, 16),
                         scalings=(2.0, 1.0, 0.5, 0.25) if T == 64 else (1.0, 0.5), slot_mode="uniform_none10")
    inp = wl.make_inputs(cfg, seed=11)
    g = gh.to_dev(inp)
    ws = pkg.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.S, cfg.R)
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gh.forward(handle, g, out=out, workspace=ws)          # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gh.forward(handle, g, out=out, workspace=ws)
    for i in range(10 if T == 64 else 3):
        new = wl.make_inputs(cfg, seed=100 + i)
        g["hidden"].copy_(new["hidden"])
        g["router_logits"].copy_(new["router_logits"])
        g["slot_idx"].copy_(new["slot_idx"])
        graph.replay()
        torch.cuda.synchronize()
        ref = dict(inp)
        ref.update(hidden=new["hidden"], router_logits=new["router_logits"], slot_idx=new["slot_idx"])
        gh.assert_close(out.float().cpu().numpy(), gh.oracle(ref)["out"], f"replay {i}")
