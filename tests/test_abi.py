"""C-ABI checks that need no GPU: the library loads, exports every declared entry
point, and its host-side argument checks accept and reject what the header says."""
import ctypes
import os
import re

import pytest

from routed_moe_expert_gb300 import binding as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe_lora.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_lora_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_lora_route", "moe_lora_permute", "moe_lora_forward", "moe_lora_create",
              "moe_lora_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(built_lib):
    for name in declared_functions():
        assert hasattr(built_lib, name), name
    assert sorted(declared_functions()) == sorted(B.EXPORTED)


def test_status_strings(built_lib):
    for s in range(7):
        assert B.moe_lora_status_string(s)
    assert "invalid" in B.moe_lora_status_string(1)


def test_workspace_size_host_only(built_lib):
    small = B.moe_lora_workspace_size(8, 128, 64, 8, 2, 1, 4)
    big = B.moe_lora_workspace_size(64, 2048, 768, 128, 8, 1, 16)
    assert 0 < small < big
    # the permuted activations alone need T*k*H*2 bytes
    assert big >= 64 * 8 * 2048 * 2
    with pytest.raises(B.MoELoRAError):
        B.moe_lora_workspace_size(8, 128, 64, 8, 9)     # top_k > E
    with pytest.raises(B.MoELoRAError):
        B.moe_lora_workspace_size(8, 128, 64, 0, 1)     # no experts
    assert B.moe_lora_workspace_size(0, 128, 64, 8, 2) > 0


def test_packed_lora_b_size_host_only(built_lib):
    """The expand-ready LoRA B copy's size follows its layout rule (rows: experts x 128-row
    tiles; columns: every slot's rank rounded up to 16), the Python shape helper agrees, and
    the host checks reject what the header says they reject."""
    # gate_up: 4 experts, N = 2I = 512 (4 tiles), ranks 8, 16, 32, 64 -> 16+16+32+64 columns
    assert B.moe_lora_packed_lora_b_size(4, 4, 512, 64, 1, (8, 16, 32, 64)) == 4 * 4 * 128 * 128 * 2
    assert B.packed_lora_b_shape(4, 512, 1, (8, 16, 32, 64)) == (4 * 4 * 128, 128)
    # down, N = 200 (2 tiles, zero rows past N), a rank-0 slot and a rank of 24
    assert B.moe_lora_packed_lora_b_size(3, 2, 200, 24, 0, (24, 0, 8)) == 2 * 2 * 128 * 48 * 2
    assert B.packed_lora_b_shape(2, 200, 0, (24, 0, 8)) == (2 * 2 * 128, 48)
    for bad in (dict(ranks=(0, 0)),                  # no stacked column at all
                dict(ranks=(8, 40)),                 # a rank above R
                dict(N=200, gated=1),                # gated needs whole 128-row tiles of gate+up rows
                dict(S=0, ranks=())):
        kw = dict(S=2, Eb=2, N=256, R=32, gated=1, ranks=(8, 16))
        kw.update(bad)
        with pytest.raises(B.MoELoRAError):
            B.moe_lora_packed_lora_b_size(kw["S"], kw["Eb"], kw["N"], kw["R"], kw["gated"], kw["ranks"])


def test_packed_lora_a_size_host_only(built_lib):
    """The shrink-ready LoRA A copy: rows are experts x every slot's rank rounded up to 8."""
    assert B.moe_lora_packed_lora_a_size(4, 3, 2048, 64, (8, 16, 32, 64)) == 3 * 120 * 2048 * 2
    assert B.packed_lora_a_shape(3, 2048, (8, 16, 32, 64)) == (3 * 120, 2048)
    assert B.moe_lora_packed_lora_a_size(3, 2, 256, 24, (5, 0, 24)) == 2 * 32 * 256 * 2
    assert B.packed_lora_a_shape(2, 256, (5, 0, 24)) == (2 * 32, 256)
    for bad in (dict(ranks=(0, 0)), dict(ranks=(8, 40)), dict(K=100), dict(S=0, ranks=())):
        kw = dict(S=2, Ea=2, K=256, R=32, ranks=(8, 16))
        kw.update(bad)
        with pytest.raises(B.MoELoRAError):
            B.moe_lora_packed_lora_a_size(kw["S"], kw["Ea"], kw["K"], kw["R"], kw["ranks"])


FAKE = 0x7f0000000000          # 16-byte aligned fake device address (never dereferenced)


def _args(**over):
    ranks = (ctypes.c_int32 * 2)(4, 2)
    scal = (ctypes.c_float * 2)(2.0, 1.0)
    a = B.Args()
    vals = dict(T=8, H=128, I=64, E=8, top_k=2, S=2, R=4, routing_method=0, routed_scaling_factor=1.0,
                n_group=1, topk_group=1, hidden=FAKE, router_logits=FAKE, correction_bias=None, w1=FAKE,
                w2=FAKE, lora_A_gu=FAKE, lora_B_gu=FAKE, lora_A_dn=FAKE, lora_B_dn=FAKE, slot_idx=FAKE,
                h_ranks=ranks, h_scalings=scal, flags=0)
    vals.update(over)
    for k, v in vals.items():
        setattr(a, k, v)
    return a, (ranks, scal)


def _validate(**over):
    a, keep = _args(**over)
    return B.lib().moe_lora_validate(ctypes.byref(a))


def test_validate_accepts_a_good_call(built_lib):
    assert _validate() == 0
    assert _validate(T=0, hidden=None, w1=None) == 0                  # empty batch
    assert _validate(routing_method=1, correction_bias=FAKE, routed_scaling_factor=2.5) == 0
    assert _validate(flags=B.FLAG_LORA_OFF, lora_A_gu=None, lora_B_gu=None, lora_A_dn=None,
                     lora_B_dn=None, slot_idx=None) == 0
    assert _validate(S=0, R=0, lora_A_gu=None) == 0


@pytest.mark.parametrize("over,code", [
    (dict(H=96), 1), (dict(H=0), 1), (dict(I=32), 1), (dict(E=0), 1), (dict(E=2000), 1),
    (dict(top_k=9), 1), (dict(top_k=0), 1), (dict(T=-1), 1), (dict(routing_method=3), 1),
    (dict(routing_method=1), 1),                       # DeepSeekV3 needs the correction bias
    (dict(n_group=2), 2), (dict(topk_group=4), 2),     # grouped DeepSeekV3 not supported
    (dict(hidden=None), 1), (dict(w2=None), 1), (dict(hidden=FAKE + 8), 1),
    (dict(lora_A_gu=None), 1), (dict(slot_idx=None), 1), (dict(S=65), 1), (dict(R=129), 1),
    (dict(R=3), 1),                                    # ranks[0] = 4 > R
])
def test_validate_rejects(built_lib, over, code):
    assert _validate(**over) == code


def test_validate_rejects_nan_scaling(built_lib):
    a, keep = _args()
    scal = (ctypes.c_float * 2)(float("nan"), 1.0)
    a.h_scalings = scal
    assert B.lib().moe_lora_validate(ctypes.byref(a)) == 1


def test_forward_rejects_null_handle_without_launching(built_lib):
    a, keep = _args()
    st = B.lib().moe_lora_forward(None, ctypes.byref(a), FAKE, FAKE, 1 << 30, None)
    assert st == 1


@pytest.mark.parametrize("over,rover", [
    (dict(), dict(num_experts=8, local_expert_offset=1)),          # local range [1, 9) past 8 experts
    (dict(), dict(num_experts=0)),
    (dict(), dict(do_finalize=2)),
    (dict(), dict(packed_topk_ids=None)),
    (dict(), dict(do_finalize=0, gemm2_output=None)),
    (dict(), dict(do_finalize=0, expanded_idx_to_permuted_idx=None)),
    (dict(E=1024), dict(num_experts=2048)),                        # E + 1 routing buckets > 1024
    (dict(H=96), dict()),                                          # the forward's own shape checks
])
def test_forward_routed_rejects_without_launching(built_lib, over, rover):
    """Host checks of moe_lora_forward_routed return INVALID_ARG before any device work (the
    handle and device addresses passed here are never dereferenced)."""
    a, keep = _args(router_logits=None, **over)
    r = B.Routed()
    vals = dict(packed_topk_ids=FAKE, num_experts=16, local_expert_offset=0, do_finalize=1,
                gemm2_output=FAKE, activation_output=None, expert_weights=None, expanded_idx_to_permuted_idx=FAKE)
    vals.update(rover)
    for k, v in vals.items():
        setattr(r, k, v)
    st = B.lib().moe_lora_forward_routed(ctypes.c_void_p(FAKE), ctypes.byref(a), ctypes.byref(r),
                                         ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 1 << 30, None)
    assert st == 1


def test_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", "/nonexistent/libmoelora.so")
    with pytest.raises(B.MoELoRAError):
        B.lib()


def _shape_args(E=4, T=3, H=64, I=32, S=2, R=8, shared=False):
    import torch
    Eo = 1 if shared else E
    return dict(hidden=torch.zeros(T, H), router_logits=torch.zeros(T, E), w1=torch.zeros(E, 2 * I, H),
                w2=torch.zeros(E, H, I), lora_A_gu=torch.zeros(S, Eo, R, H), lora_B_gu=torch.zeros(S, E, 2 * I, R),
                lora_A_dn=torch.zeros(S, E, R, I), lora_B_dn=torch.zeros(S, Eo, H, R),
                slot_idx=torch.zeros(T, dtype=torch.int32), ranks=(8, 4), scalings=(1.0, 0.5),
                flags=B.FLAG_SHARED_OUTER if shared else 0)


def test_binding_checks_shapes_before_taking_pointers():
    """The library reads every tensor through a raw pointer at the size the shape arguments
    imply, so the binding rejects any tensor whose shape disagrees (host only, no launch)."""
    import torch
    B.check_shapes(**_shape_args())
    B.check_shapes(**_shape_args(shared=True))
    bad = [
        ("lora_A_gu", torch.zeros(2, 1, 8, 64)),     # shared-outer layout without the flag
        ("lora_B_dn", torch.zeros(2, 1, 64, 8)),
        ("lora_B_gu", torch.zeros(2, 4, 64, 4)),     # rank dimension disagrees with A
        ("lora_A_dn", torch.zeros(2, 4, 8, 64)),     # K of the down shrink is I, not H
        ("w2", torch.zeros(4, 32, 64)),              # transposed
        ("router_logits", torch.zeros(3, 5)),
        ("slot_idx", torch.zeros(4, dtype=torch.int32)),
    ]
    for name, t in bad:
        kw = _shape_args()
        kw[name] = t
        with pytest.raises(ValueError, match=name):
            B.check_shapes(**kw)
    kw = _shape_args(shared=True)
    kw["flags"] = 0                                  # per-expert flag with shared-outer tensors
    with pytest.raises(ValueError, match="lora_A_gu"):
        B.check_shapes(**kw)
    kw = _shape_args()
    kw["ranks"] = (8, 16)                            # a rank above R
    with pytest.raises(ValueError, match="rank"):
        B.check_shapes(**kw)
    kw = _shape_args()
    kw["scalings"] = (1.0,)
    with pytest.raises(ValueError, match="same length"):
        B.check_shapes(**kw)
    kw = _shape_args()
    kw["correction_bias"] = torch.zeros(4)           # [E]
    B.check_shapes(**kw)
    kw["correction_bias"] = torch.zeros(5)
    with pytest.raises(ValueError, match="correction_bias"):
        B.check_shapes(**kw)


@pytest.mark.parametrize("over,wover", [
    (dict(H=192), dict()),                                         # H not a multiple of 128
    (dict(I=64), dict()),                                          # I not a multiple of 128
    (dict(), dict(w1_scale=None)),
    (dict(), dict(w2_scale=FAKE + 2)),                             # misaligned scales
    (dict(), dict(w1=None)),
    (dict(top_k=9), dict()),                                       # the forward's own checks
])
def test_forward_fp8_rejects_without_launching(built_lib, over, wover):
    """Host checks of moe_lora_forward_fp8 return INVALID_ARG before any device work (the
    handle and device addresses passed here are never dereferenced)."""
    a, keep = _args(**{**dict(H=256, I=128), **over})
    w = B.Fp8Weights()
    vals = dict(w1=FAKE, w1_scale=FAKE, w2=FAKE, w2_scale=FAKE)
    vals.update(wover)
    for k, v in vals.items():
        setattr(w, k, v)
    st = B.lib().moe_lora_forward_fp8(ctypes.c_void_p(FAKE), ctypes.byref(a), ctypes.byref(w),
                                      ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 1 << 30, None)
    assert st == 1


def test_quant_fp8_host_checks(built_lib):
    L = B.lib()
    h = ctypes.c_void_p(FAKE)
    assert L.moe_lora_quant_fp8(None, FAKE, None, 4, 256, 1, FAKE, FAKE, None) == 1        # no handle
    assert L.moe_lora_quant_fp8(h, FAKE, None, 4, 192, 1, FAKE, FAKE, None) == 1           # K % 128
    assert L.moe_lora_quant_fp8(h, FAKE, None, -1, 256, 1, FAKE, FAKE, None) == 1          # rows < 0
    assert L.moe_lora_quant_fp8(h, FAKE, FAKE, 4, 256, 0, FAKE, FAKE, None) == 1           # top_k with perm
    assert L.moe_lora_quant_fp8(h, FAKE + 8, None, 4, 256, 1, FAKE, FAKE, None) == 1       # misaligned rows
    assert L.moe_lora_quant_fp8(h, None, None, 0, 256, 1, None, None, None) == 0           # nothing to do


def test_grouped_gemm_fp8_host_checks(built_lib):
    """Host checks of the FP8 grouped GEMM return INVALID_ARG before any device work."""
    L = B.lib()
    h = ctypes.c_void_p(FAKE)
    ok = dict(w=FAKE, ws=FAKE, x=FAKE, xs=FAKE, off=FAKE, E=4, N=256, K=384, P=32, out=FAKE)

    def call(**over):
        v = {**ok, **over}
        return L.moe_lora_grouped_gemm_fp8(over.get("h", h), v["w"], v["ws"], v["x"], v["xs"], v["off"], v["E"],
                                           v["N"], v["K"], v["P"], v["out"], None)
    assert call(h=None) == 1                  # no handle
    assert call(N=192) == 1                   # N % 128
    assert call(K=64) == 1                    # K % 128
    assert call(E=0) == 1 and call(E=1025) == 1
    assert call(P=-1) == 1
    assert call(x=FAKE + 8) == 1              # misaligned codes
    assert call(out=FAKE + 4) == 1            # misaligned output
    assert call(off=None) == 1
    assert call(P=0, w=None, x=None, out=None) == 0   # nothing to do


def test_binding_checks_fp8_weight_shapes():
    import torch
    E, H, I = 3, 256, 128
    good = dict(w1_q=torch.zeros(E, 2 * I, H, dtype=torch.uint8), w1_scale=torch.zeros(E, 2, 2),
                w2_q=torch.zeros(E, H, I, dtype=torch.uint8), w2_scale=torch.zeros(E, 2, 1))
    B.check_fp8_weights(**good)
    for name, t in [("w2_q", torch.zeros(E, I, H, dtype=torch.uint8)), ("w1_scale", torch.zeros(E, 2, 1)),
                    ("w2_scale", torch.zeros(E, 1, 2))]:
        kw = dict(good)
        kw[name] = t
        with pytest.raises(ValueError, match=name):
            B.check_fp8_weights(**kw)
    with pytest.raises(ValueError, match="multiples of 128"):
        B.check_fp8_weights(torch.zeros(E, 128, 192, dtype=torch.uint8), torch.zeros(E, 1, 1),
                            torch.zeros(E, 192, 64, dtype=torch.uint8), torch.zeros(E, 1, 1))


def test_validate_accepts_every_stated_maximum(built_lib):
    """The header's limits are inclusive: E 1024, top_k 32, S 64, R 128, H and I 16384."""
    ranks = (ctypes.c_int32 * 64)(*([128] * 64))
    scal = (ctypes.c_float * 64)(*([0.5] * 64))
    a, keep = _args(E=1024, top_k=32, S=64, R=128, H=16384, I=16384)
    a.h_ranks, a.h_scalings = ranks, scal
    assert B.lib().moe_lora_validate(ctypes.byref(a)) == 0
    for name, bad in (("top_k", 33), ("E", 1025), ("S", 65), ("R", 129), ("H", 16384 + 64), ("I", 16384 + 64)):
        setattr(a, name, bad)
        assert B.lib().moe_lora_validate(ctypes.byref(a)) == 1, name
        setattr(a, name, dict(top_k=32, E=1024, S=64, R=128, H=16384, I=16384)[name])
