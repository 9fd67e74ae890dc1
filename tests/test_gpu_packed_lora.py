"""Expand-ready (packed) LoRA B copies: the pack's layout, bit for bit, against the layout rule
written out in torch; the layer with packed copies and separate shrink kernels against the same
layer with the per-slot LoRA stages (equal outputs: a pair's stacked shrink row is zero outside
its own slot, so the other slots' columns add exact zeros); and the layer with the shrinks run
as tiles of the expert GEMMs against the oracle, with the launches it saves counted."""
import numpy as np
import pytest
import torch

import routed_moe_expert_gb300 as pkg
from routed_moe_expert_gb300 import workloads as wl
import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    h = pkg.Handle(0)
    yield h
    h.close()


def _packed_reference(B: torch.Tensor, ranks, gated: int) -> torch.Tensor:
    """The layout of moe_lora_pack_lora_b, from its definition: row (e * NT + nt) * 128 + r is
    row r of 128-row weight tile nt (gated: gate rows then up rows), slot s's ranks side by side
    from column coff[s], each slot's block rounded up to 16 columns."""
    S, Eb, N, R = B.shape
    NT = N // 128 if gated else (N + 127) // 128
    ru = [(r + 15) // 16 * 16 if r > 0 else 0 for r in ranks]
    coff = np.concatenate([[0], np.cumsum(ru)]).astype(int)
    out = torch.zeros((Eb, NT, 128, int(coff[-1])), dtype=torch.bfloat16)
    rows = torch.arange(128)
    for nt in range(NT):
        n = torch.where(rows < 64, 64 * nt + rows, N // 2 + 64 * nt + rows - 64) if gated else 128 * nt + rows
        ok = n < N
        for s in range(S):
            if ranks[s] > 0:
                out[:, nt, ok, coff[s]:coff[s] + ranks[s]] = B[s][:, n[ok], :ranks[s]]
    return out.reshape(Eb * NT * 128, -1)


@pytest.mark.parametrize("S,Eb,N,R,ranks,gated", [
    (4, 3, 256, 64, (8, 0, 24, 64), 1),     # gate_up layout, a rank-0 slot, a rank not a multiple of 16
    (2, 5, 200, 32, (32, 16), 0),           # down layout, N not a multiple of 128 (zero rows)
    (3, 1, 384, 16, (16, 8, 16), 0),        # shared-outer down B: one expert set
    (1, 2, 128, 128, (128,), 1),            # one slot at the largest rank (two panels)
], ids=["gate_up", "down-ragged", "shared", "rank128"])
def test_pack_lora_b_layout_bit_exact(handle, S, Eb, N, R, ranks, gated):
    g = torch.Generator().manual_seed(N + R)
    B = torch.randn((S, Eb, N, R), generator=g).to(torch.bfloat16)
    for s, r in enumerate(ranks):   # the rank tails must never be read
        B[s, :, :, r:] = float("nan")
    got = pkg.moe_lora_pack_lora_b(handle, B.cuda(), ranks, gated)
    torch.cuda.synchronize()
    ref = _packed_reference(B, ranks, gated)
    assert tuple(got.shape) == tuple(ref.shape) == pkg.packed_lora_b_shape(Eb, N, gated, ranks)
    assert pkg.moe_lora_packed_lora_b_size(S, Eb, N, R, gated, ranks) == ref.numel() * 2
    assert torch.equal(got.cpu().view(torch.int16), ref.view(torch.int16))


def _packed_a_reference(A: torch.Tensor, ranks) -> torch.Tensor:
    """The layout of moe_lora_pack_lora_a, from its definition: for each expert, every slot's
    rank rows one after another, each slot's block rounded up to 8 rows of zeros."""
    S, Ea, R, K = A.shape
    ro = [(r + 7) // 8 * 8 if r > 0 else 0 for r in ranks]
    aoff = np.concatenate([[0], np.cumsum(ro)]).astype(int)
    out = torch.zeros((Ea, int(aoff[-1]), K), dtype=torch.bfloat16)
    for s in range(S):
        if ranks[s] > 0:
            out[:, aoff[s]:aoff[s] + ranks[s], :] = A[s, :, :ranks[s], :]
    return out.reshape(Ea * int(aoff[-1]), K)


@pytest.mark.parametrize("S,Ea,R,K,ranks", [
    (4, 3, 64, 256, (8, 16, 32, 64)),   # the multi-slot ranks
    (4, 2, 24, 128, (16, 24, 0, 5)),    # a rank-0 slot and ranks that are not multiples of 8
    (2, 1, 16, 384, (16, 8)),           # shared-outer A: one expert set
], ids=["four", "ragged", "shared"])
def test_pack_lora_a_layout_bit_exact(handle, S, Ea, R, K, ranks):
    g = torch.Generator().manual_seed(K + R)
    A = torch.randn((S, Ea, R, K), generator=g).to(torch.bfloat16)
    for s, r in enumerate(ranks):   # the rank tails must never be read
        A[s, :, r:, :] = float("nan")
    got = pkg.moe_lora_pack_lora_a(handle, A.cuda(), ranks)
    torch.cuda.synchronize()
    ref = _packed_a_reference(A, ranks)
    assert tuple(got.shape) == tuple(ref.shape) == pkg.packed_lora_a_shape(Ea, K, ranks)
    assert pkg.moe_lora_packed_lora_a_size(S, Ea, K, R, ranks) == ref.numel() * 2
    assert torch.equal(got.cpu().view(torch.int16), ref.view(torch.int16))


def _run_pair(h, cfg, seed, flags=0, device_inputs=False, saved_launches=None):
    """The layer on the same inputs with per-slot LoRA stages, with packed stages and separate
    shrink kernels (equal to the first), and with packed stages and the shrinks as tiles of the
    GEMMs where they fit (the shrink's products are then accumulated with the operands'
    roles swapped, so it is held to the oracle's tolerance); returns the first and the last."""
    inp = wl.make_inputs(cfg, seed=seed, device="cuda" if device_inputs else "cpu")
    g = gh.to_dev(inp)
    ws = pkg.alloc_workspace(g["T"], cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.S, cfg.R)
    base = gh.forward(h, g, flags=flags, workspace=ws)
    torch.cuda.synchronize()
    st, word = pkg.moe_lora_check_status(ws)
    assert st == 0, f"device status {word:#x}"
    so = bool(flags & pkg.FLAG_SHARED_OUTER)
    bgu = pkg.moe_lora_pack_lora_b(h, g["lora_B_gu"], g["ranks"], 1)
    bdn = pkg.moe_lora_pack_lora_b(h, g["lora_B_dn"], g["ranks"], 0)
    assert bdn.shape[0] == (1 if so else cfg.E) * ((cfg.H + 127) // 128) * 128
    agu = pkg.moe_lora_pack_lora_a(h, g["lora_A_gu"], g["ranks"])
    adn = pkg.moe_lora_pack_lora_a(h, g["lora_A_dn"], g["ranks"])

    def packed(extra, with_a=False):
        more = dict(lora_A_gu_packed=agu, lora_A_dn_packed=adn) if with_a else {}
        o = pkg.moe_lora_forward(
            h, g["hidden"], g["router_logits"], g["w1"], g["w2"], g["top_k"], routing_method=g["method"],
            correction_bias=g["correction_bias"], routed_scaling_factor=g["rsf"],
            lora_A_gu=g["lora_A_gu"], lora_B_gu=g["lora_B_gu"], lora_A_dn=g["lora_A_dn"],
            lora_B_dn=g["lora_B_dn"], slot_idx=g["slot_idx"], ranks=g["ranks"], scalings=g["scalings"],
            flags=flags | extra, workspace=ws, lora_B_gu_packed=bgu, lora_B_dn_packed=bdn, **more)
        torch.cuda.synchronize()
        st, word = pkg.moe_lora_check_status(ws)
        assert st == 0, f"device status {word:#x}"
        return o

    n0 = h.launch_count()
    sep = packed(pkg.FLAG_SEPARATE_SHRINK)
    n1 = h.launch_count()
    assert torch.equal(sep, base), f"packed and per-slot LoRA stages differ: {int((sep != base).sum())} elements"
    out = packed(0)
    n2 = h.launch_count()
    if saved_launches is not None:   # shrink kernels that ran as GEMM tiles instead
        assert (n1 - n0) - (n2 - n1) == saved_launches, ((n1 - n0), (n2 - n1))
    ref = gh.oracle(inp, lazy=device_inputs)
    gh.assert_close(out.float().cpu().numpy(), ref["out"], cfg.name)
    gh.assert_close(out.float().cpu().numpy(), base.float().cpu().numpy(), cfg.name + " vs per-slot")
    # the shrink-ready A copies change only where each rank row comes from (one copy per K step)
    sep_a = packed(pkg.FLAG_SEPARATE_SHRINK, with_a=True)
    assert torch.equal(sep_a, base), f"shrink-ready A, shrink kernels: {int((sep_a != base).sum())} elements differ"
    out_a = packed(0, with_a=True)
    assert torch.equal(out_a, out), f"shrink-ready A, shrink tiles: {int((out_a != out).sum())} elements differ"
    return base, out


@pytest.mark.parametrize("T,E,k,ranks,scalings,shared,saved", [
    (96, 16, 4, (8, 16, 32, 64), (2.0, 1.0, 0.5, 0.25), False, 2),   # 64-token tiles: both shrinks in the GEMMs
    (96, 16, 4, (8, 16), (2.0, 0.5), False, 1),                      # <= 32 stacked ranks: permute + shrink
    (64, 16, 4, (8, 32), (2.0, 0.5), True, 2),                       # shared-outer, 32-token tiles
    (96, 16, 4, (16, 24, 0, 8), (1.0, 0.0, 1.0, 2.0), False, 1),     # a disabled slot and a rank-0 slot
    (600, 8, 2, (8, 16, 32, 64), (2.0, 1.0, 0.5, 0.25), False, 0),   # 256-token CTA-pair tiles
    (96, 16, 4, (64, 64, 8), (1.0, 0.5, 2.0), False, 0),             # 136 active rank rows: too many
], ids=["four-slots", "few-ranks", "shared-outer", "disabled-slots", "pair-tiles", "many-ranks"])
def test_packed_lora_b_equals_per_slot_stages(handle, T, E, k, ranks, scalings, shared, saved):
    cfg = wl.LayerConfig("pk", T=T, H=512, I=256, E=E, top_k=k, ranks=ranks, scalings=scalings,
                         slot_mode="uniform_none10", shared_outer=shared)
    _run_pair(handle, cfg, seed=T + len(ranks), flags=pkg.FLAG_SHARED_OUTER if shared else 0,
              saved_launches=saved)


def test_packed_lora_b_multi_slot_config(handle):
    _run_pair(handle, wl.CONFIGS["multi_slot"], seed=0, device_inputs=True, saved_launches=2)


def test_packed_lora_b_graph_replay(handle):
    """Captured once, replayed: the packed stages read only buffers that exist before capture."""
    cfg = wl.LayerConfig("pkg", T=96, H=512, I=256, E=16, top_k=4, ranks=(8, 16, 32, 64),
                         scalings=(2.0, 1.0, 0.5, 0.25), slot_mode="uniform_none10")
    base, _ = _run_pair(handle, cfg, seed=5)
    inp = wl.make_inputs(cfg, seed=5)
    g = gh.to_dev(inp)
    ws = pkg.alloc_workspace(g["T"], cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.S, cfg.R)
    bgu = pkg.moe_lora_pack_lora_b(handle, g["lora_B_gu"], g["ranks"], 1)
    bdn = pkg.moe_lora_pack_lora_b(handle, g["lora_B_dn"], g["ranks"], 0)
    out = torch.empty_like(base)
    kw = dict(routing_method=g["method"], correction_bias=g["correction_bias"], routed_scaling_factor=g["rsf"],
              lora_A_gu=g["lora_A_gu"], lora_B_gu=g["lora_B_gu"], lora_A_dn=g["lora_A_dn"],
              lora_B_dn=g["lora_B_dn"], slot_idx=g["slot_idx"], ranks=g["ranks"], scalings=g["scalings"],
              workspace=ws, out=out, lora_B_gu_packed=bgu, lora_B_dn_packed=bdn)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkg.moe_lora_forward(handle, g["hidden"], g["router_logits"], g["w1"], g["w2"], g["top_k"], stream=s, **kw)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        pkg.moe_lora_forward(handle, g["hidden"], g["router_logits"], g["w1"], g["w2"], g["top_k"], stream=s, **kw)
    eager = out.clone()   # the warm-up forward's output (the shrinks ran inside the GEMMs)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    gh.assert_close(eager.float().cpu().numpy(), base.float().cpu().numpy(), "graph vs per-slot")
