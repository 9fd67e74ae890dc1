"""GPU parity of the externally routed entry (moe_lora_forward_routed): routing given as
packed (expert << 16 | bf16 weight) words, a local expert range with the other pairs
dropped, and the do_finalize=False outputs -- against the oracle's
moe_lora_forward_routed on the same seeded inputs."""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
import routed_moe_expert_gb300 as pkg
from oracle import moe_lora_oracle as orc
from routed_moe_expert_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    return pkg.Handle(0)


def _case(T, H, I, E_loc, E_glob, k, ranks=(8, 16), scalings=(2.0, 0.5), seed=0, shared_outer=False):
    cfg = wl.LayerConfig("routed", T=T, H=H, I=I, E=E_loc, top_k=k, ranks=ranks, scalings=scalings,
                         slot_mode="uniform_none10", shared_outer=shared_outer)
    inp = wl.make_inputs(cfg, seed=seed)
    ids, w = wl.make_routing(T, E_glob, k, seed=seed + 1)
    packed = orc.pack_topk(ids.numpy(), w.numpy())
    return inp, packed


def _run(h, inp, packed, E_glob, offset, do_finalize, flags=0, tokens=None):
    g = gh.to_dev(inp)
    ws = pkg.alloc_workspace(g["T"], inp["hidden"].shape[1], inp["w1"].shape[1] // 2, inp["w1"].shape[0],
                             inp["top_k"], len(inp["ranks"]), int(inp["lora_A_gu"].shape[2]))
    res = pkg.moe_lora_forward_routed(
        h, g["hidden"], torch.from_numpy(packed).cuda(), g["w1"], g["w2"], inp["top_k"], E_glob,
        local_expert_offset=offset, do_finalize=do_finalize, lora_A_gu=g["lora_A_gu"], lora_B_gu=g["lora_B_gu"],
        lora_A_dn=g["lora_A_dn"], lora_B_dn=g["lora_B_dn"], slot_idx=g["slot_idx"], ranks=inp["ranks"],
        scalings=inp["scalings"], flags=flags | (pkg.FLAG_SHARED_OUTER if inp["shared_outer"] else 0), workspace=ws)
    torch.cuda.synchronize()
    st, word = pkg.moe_lora_check_status(ws)
    ref = orc.moe_lora_forward_routed(
        gh.np_(inp["hidden"]), packed, gh.np_(inp["w1"]), gh.np_(inp["w2"]), inp["top_k"], E_glob,
        local_expert_offset=offset, lora_A_gu=gh.np_(inp["lora_A_gu"]), lora_B_gu=gh.np_(inp["lora_B_gu"]),
        lora_A_dn=gh.np_(inp["lora_A_dn"]), lora_B_dn=gh.np_(inp["lora_B_dn"]), slot_idx=gh.np_(inp["slot_idx"]),
        ranks=inp["ranks"], scalings=inp["scalings"], do_finalize=do_finalize, tokens=tokens,
        shared_outer=inp["shared_outer"])
    return res, ref, st


@pytest.mark.parametrize("T,E_loc,E_glob,offset,k", [(40, 8, 24, 8, 4), (64, 128, 128, 0, 8), (600, 16, 32, 16, 4)],
                         ids=["ep-third", "decode-all-local", "wide-tiles-upper-half"])
def test_routed_finalized_matches_oracle(handle, T, E_loc, E_glob, offset, k):
    H, I = (512, 256) if E_loc <= 16 else (2048, 768)
    inp, packed = _case(T, H, I, E_loc, E_glob, k, seed=T)
    out, ref, st = _run(handle, inp, packed, E_glob, offset, True)
    assert st == 0
    gh.assert_close(out.float().cpu().numpy(), ref["out"], "routed out")


def test_routed_shared_outer_matches_oracle(handle):
    inp, packed = _case(96, 512, 256, 8, 16, 4, seed=11, shared_outer=True)
    out, ref, st = _run(handle, inp, packed, 16, 8, True)
    assert st == 0
    gh.assert_close(out.float().cpu().numpy(), ref["out"], "routed shared-outer out")


def test_routed_unfinalized_outputs_match_oracle(handle):
    inp, packed = _case(48, 512, 256, 8, 20, 4, seed=5)
    res, ref, st = _run(handle, inp, packed, 20, 6, False)
    assert st == 0
    idx = res["expanded_idx_to_permuted_idx"].cpu().numpy()
    np.testing.assert_array_equal(idx, ref["expanded_idx_to_permuted_idx"])
    np.testing.assert_array_equal(res["expert_weights"].cpu().numpy(), ref["expert_weights"])
    q = idx[idx >= 0]
    gh.assert_close(res["gemm2_output"].cpu().numpy()[q], ref["gemm2_output"][q], "gemm2_output")
    gh.assert_close(res["activation_output"].float().cpu().numpy()[q], ref["activation"][q], "activation")


def test_routed_all_local_equals_logit_routing_bitwise(handle):
    """Constant logits route every token to experts 0..k-1 with weight 1/k, which bf16 holds
    exactly: the packed entry with every expert local gives the logit-routed bits."""
    cfg = wl.LayerConfig("eq", T=96, H=512, I=256, E=16, top_k=4, ranks=(8, 16), scalings=(2.0, 0.5),
                         slot_mode="uniform_none10")
    inp = wl.make_inputs(cfg, seed=3)
    inp["router_logits"] = torch.zeros_like(inp["router_logits"])
    g = gh.to_dev(inp)
    a = gh.forward(handle, g).clone()
    ids, w = orc.route(np.zeros((96, 16)), 4)
    packed = torch.from_numpy(orc.pack_topk(ids, w)).cuda()
    b = pkg.moe_lora_forward_routed(handle, g["hidden"], packed, g["w1"], g["w2"], 4, 16, lora_A_gu=g["lora_A_gu"],
                                    lora_B_gu=g["lora_B_gu"], lora_A_dn=g["lora_A_dn"], lora_B_dn=g["lora_B_dn"],
                                    slot_idx=g["slot_idx"], ranks=inp["ranks"], scalings=inp["scalings"])
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_routed_expert_id_out_of_range_reported(handle):
    """An expert id past num_experts is reported as a device check and its pair dropped."""
    inp, packed = _case(16, 256, 128, 4, 8, 2, seed=9)
    packed = packed.copy()
    packed[3, 1] = np.int32((9 << 16) | 0x3F00)      # expert 9 of 8
    g = gh.to_dev(inp)
    ws = pkg.alloc_workspace(16, 256, 128, 4, 2, 2, 16)
    pkg.moe_lora_forward_routed(handle, g["hidden"], torch.from_numpy(packed).cuda(), g["w1"], g["w2"], 2, 8,
                                lora_A_gu=g["lora_A_gu"], lora_B_gu=g["lora_B_gu"], lora_A_dn=g["lora_A_dn"],
                                lora_B_dn=g["lora_B_dn"], slot_idx=g["slot_idx"], ranks=inp["ranks"],
                                scalings=inp["scalings"], workspace=ws)
    st, word = pkg.moe_lora_check_status(ws)
    assert st == 6 and (word & 0xff) == 6
