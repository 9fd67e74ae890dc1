"""The allocation-free routing entry point, checked against the regular one.

moe_lora_route_noalloc serves callers that cannot allocate device memory or hand the
library a workspace (a plug-in whose host framework owns all device memory, or a
real-time path that must not touch an allocator once it runs).  Its routing scratch
lives in a fixed array inside the library, shared by every call.  This test calls it
through the C ABI twice in a row, on different inputs, and requires the same results as
moe_lora_route: identical expert ids, offsets and permutations, and routing weights
within the tolerance the other routing tests use.  The second call also shows that the
scratch left behind by the first does not leak into the next result.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _noalloc(lib, logits, bias, k, method, rsf):
    T, E = logits.shape
    P = T * k
    out = dict(topk_ids=torch.empty((T, k), dtype=torch.int32, device="cuda"),
               topk_weights=torch.empty((T, k), dtype=torch.float32, device="cuda"),
               expert_offsets=torch.empty((E + 1,), dtype=torch.int32, device="cuda"),
               perm=torch.empty((P,), dtype=torch.int32, device="cuda"),
               inv_perm=torch.empty((P,), dtype=torch.int32, device="cuda"))
    f = lib.moe_lora_route_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_float, ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 6
    st = f(logits.data_ptr(), None if bias is None else bias.data_ptr(), T, E, k, method, rsf, 1, 1,
           out["topk_ids"].data_ptr(), out["topk_weights"].data_ptr(), out["expert_offsets"].data_ptr(),
           out["perm"].data_ptr(), out["inv_perm"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, f"moe_lora_route_noalloc returned {st}"
    return out


# (8192, 1024, 8): the routing grid (128 CTAs of 64 tokens) is cut to the 63 CTAs whose
# scratch fits the fixed array, so each CTA routes 131 tokens.
@pytest.mark.parametrize("T,E,k,method", [(64, 128, 8, 0), (4096, 384, 8, 1), (8192, 1024, 8, 0)])
def test_noalloc_route_matches_route_twice(T, E, k, method):
    import routed_moe_expert_gb300 as pkg
    from routed_moe_expert_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    lib = pkg.lib()
    h = pkg.Handle(0)
    rsf = 2.827 if method == 1 else 1.0
    for call in range(2):
        g = torch.Generator().manual_seed(1000 * call + T + E)
        logits = torch.randn(T, E, generator=g).to(torch.bfloat16).cuda()
        bias = (torch.randn(E, generator=g) * 0.1).float().cuda() if method == 1 else None
        got = _noalloc(lib, logits, bias, k, method, rsf)
        ref = pkg.moe_lora_route(h, logits, k, method, bias, rsf)
        torch.cuda.synchronize()
        for key in ("topk_ids", "expert_offsets", "perm", "inv_perm"):
            assert torch.equal(got[key], ref[key]), f"call {call}: {key} differs"
        np.testing.assert_allclose(got["topk_weights"].cpu().numpy(), ref["topk_weights"].cpu().numpy(),
                                   rtol=2e-6, atol=1e-7)
    h.close()
