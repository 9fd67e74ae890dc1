"""Helpers for the GPU parity tests: move seeded inputs to the device, run the CUDA
path through the C ABI, run the CPU oracle on the same inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import routed_moe_expert_gb300 as pkg
from oracle import moe_lora_oracle as orc

# Float tolerance of the layer output: |gpu - ref| <= ATOL + RTOL * |ref| elementwise,
# and relative L2 error <= REL_L2.
ATOL, RTOL, REL_L2 = 1e-2, 2e-2, 5e-3
# The FP8 path: three times the bf16 relative L2 bound, ten times its elementwise bounds.
# Its activation is quantised to e4m3 after the bf16 rounding, so a rounding difference
# upstream (the e4m3 tensor-core accumulation of the gate_up GEMM) comes out about three
# times larger than in the bf16 layer in relative L2; on single elements more: a change of
# a 128-value group's largest activation changes the group's scale (amax / 448) and every
# code in it, which with one group per row (I = 128) moves a token's whole output row.  The
# derivation is pinned on the CPU by
# tests/test_oracle_fp8.py::test_fp8_tolerance_covers_accumulation_noise, from the
# accumulation model below, over the shapes of the GPU tests and several inputs.
ATOL_FP8, RTOL_FP8, REL_L2_FP8 = 1e-1, 2e-1, 1.5e-2
# Accumulation model of the block-scaled FP8 GEMM behind those bounds: every product of two
# e4m3 values is exact (4 x 4 significant bits); the tensor cores sum a 128-wide K block's
# products as a tree of depth 7 whose adders keep at least FP8_ACC_BITS significant bits, so
# a block sum is off by at most 7 * 2^-FP8_ACC_BITS times the block's sum of |products|; the
# block sums are scaled and added in fp32.  tests/test_gpu_fp8.py holds the GPU GEMM to this
# bound element by element; tests/test_oracle_fp8.py propagates errors of this size through
# the layer and shows the FP8 bounds above cover them.
FP8_ACC_BITS = 16
# The NVFP4 path: ten times the bf16 elementwise bounds, five times its relative L2 bound.
# Its GEMM products are exact and summed in fp32, but both of its GEMM inputs are re-quantised
# to e2m1 (steps of a third to a half of the value): a one-ulp bf16 change of the gate_up
# output, or of a row's largest activation (the row scale), moves codes by a whole e2m1 step.
# Model of the fp32 sums: the probabilistic rounding-error bound of a K-term sum,
# NVFP4_LAMBDA * sqrt(K) * 2^-24 times its sum of |terms| (Higham and Mary, "A new approach to
# probabilistic rounding error analysis", SIAM J. Sci. Comput. 41(5), 2019, with lambda = 3).
# tests/test_oracle_nvfp4.py::test_nvfp4_tolerance_covers_rounding_flips plants errors of that
# size in the oracle's gate_up sums and shows these bounds cover the resulting flips while the
# bf16 bounds do not; tests/test_gpu_nvfp4.py holds the GPU GEMM to its fp32 bound.
ATOL_NVFP4, RTOL_NVFP4, REL_L2_NVFP4 = 1e-1, 2e-1, 2.5e-2
NVFP4_LAMBDA = 3.0


def to_dev(inp: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def forward(h, g: dict, flags=0, outputs=None, out=None, workspace=None, stream=None, prof_events=None):
    return pkg.moe_lora_forward(
        h, g["hidden"], g["router_logits"], g["w1"], g["w2"], g["top_k"], routing_method=g["method"],
        correction_bias=g["correction_bias"], routed_scaling_factor=g["rsf"],
        lora_A_gu=g["lora_A_gu"], lora_B_gu=g["lora_B_gu"], lora_A_dn=g["lora_A_dn"], lora_B_dn=g["lora_B_dn"],
        slot_idx=g["slot_idx"], ranks=g["ranks"], scalings=g["scalings"], flags=flags, outputs=outputs,
        out=out, workspace=workspace, stream=stream, prof_events=prof_events)


class _ByExpert:
    """Expert-indexed view of a (possibly device-resident) weight tensor, for the oracle:
    [e] / [s, e] returns that slice as a float32 numpy array, copied when asked."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, idx):
        return self.t[idx].float().cpu().numpy()

    def __len__(self):
        return self.t.shape[0]


def np_(t):
    if t is None:
        return None
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()


def oracle(inp: dict, tokens=None, lora_off=False, lazy=False):
    W = (lambda t: None if t is None else _ByExpert(t)) if lazy else np_
    return orc.moe_lora_forward(
        np_(inp["hidden"]), np_(inp["router_logits"]), W(inp["w1"]), W(inp["w2"]), inp["top_k"], inp["method"],
        np_(inp["correction_bias"]), inp["rsf"], W(inp["lora_A_gu"]), W(inp["lora_B_gu"]), W(inp["lora_A_dn"]),
        W(inp["lora_B_dn"]), np_(inp["slot_idx"]), inp["ranks"], inp["scalings"], lora_off=lora_off, tokens=tokens,
        shared_outer=bool(inp.get("shared_outer", False)))


def assert_close(got, ref, what="output", atol=ATOL, rtol=RTOL, rel_l2=REL_L2):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance, "
                           f"max err {err.max():.4g}, rel L2 {rel:.3g}")
    assert rel <= rel_l2, f"{what}: relative L2 error {rel:.4g} > {rel_l2}"
    return float(err.max()), float(rel)


def sample_tokens(ids: np.ndarray, E: int, every: int, extremes: int = 3, per_expert: int = 64) -> np.ndarray:
    """Every `every`-th token plus up to `per_expert` tokens routed to each of the
    `extremes` most and least loaded (non-empty) experts."""
    T = ids.shape[0]
    load = np.bincount(ids.reshape(-1), minlength=E)
    nz = np.nonzero(load)[0]
    order = nz[np.argsort(load[nz], kind="stable")]
    pick = set(order[:extremes].tolist()) | set(order[-extremes:].tolist())
    toks = set(range(0, T, every))
    for e in pick:
        toks |= set(np.nonzero((ids == e).any(axis=1))[0][:per_expert].tolist())
    return np.array(sorted(toks), dtype=np.int64)
