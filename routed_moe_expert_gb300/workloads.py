"""Seeded synthetic workloads for the routed MoE-LoRA expert layer.

This module only draws inputs.  It holds none of the layer's arithmetic, so both
the CUDA path (through the binding) and the CPU oracle can consume what it makes
without sharing any code with each other.

Shapes and value distributions follow the layer configurations the MoE-LoRA pages
describe (sglang PR #28466 "bf16 MoE-LoRA for trtllm backend", Verification:
Qwen3-30B-A3B-class experts, rank-16 adapter; sglang PR #28091 "Fix experimental
fast-path multi-adapter correctness", Accuracy Tests: four resident adapters of
ranks 16/32 with mixed traffic; sglang PR #27329 "Experimental fast LoRA path",
Tests done: Kimi-K2.5, a DeepSeekV3-routed 384-expert model):

  hidden ~ N(0, 1), router_logits ~ N(0, 1) (rounded to bf16),
  w1, w2, LoRA A ~ N(0, 1/sqrt(K)) with K the contraction length,
  LoRA B ~ N(0, 0.02).

Rank tails (rows r >= ranks[s] of A, columns r >= ranks[s] of B) are filled with
NaN so that any read past a slot's rank poisons the result.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

RENORMALIZE = 0
DEEPSEEK_V3 = 1


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    top_k: int
    method: int = RENORMALIZE
    ranks: tuple = (16,)
    scalings: tuple = (2.0,)
    slot_mode: str = "all0"          # "all0" | "uniform_none10"
    zipf_bias: bool = False          # per-expert bias 1.5*log(1/rank_e) on the logits
    bias_std: float = 0.0            # DeepSeekV3 correction bias ~ N(0, bias_std)
    rsf: float = 1.0                 # routed_scaling_factor (DeepSeekV3)
    shared_outer: bool = False       # one A_gu and one B_dn per slot ([S, 1, ...]) for all experts

    @property
    def S(self) -> int:
        return len(self.ranks)

    @property
    def R(self) -> int:
        return max(self.ranks) if self.ranks else 0

    @property
    def P(self) -> int:
        return self.T * self.top_k

    def describe(self) -> str:
        rk = "/".join(str(r) for r in self.ranks)
        meth = "DeepSeekV3" if self.method == DEEPSEEK_V3 else "Renormalize"
        return (f"{self.name}: T{self.T} H{self.H} I{self.I} E{self.E} k{self.top_k} "
                f"{meth} r{rk}")


CONFIGS = {
    # tiny parity case: one adapter rank 4, scaling 2
    "tiny": LayerConfig("tiny", T=8, H=128, I=64, E=8, top_k=2, ranks=(4,), scalings=(2.0,)),
    # decode, Qwen3-30B-A3B-like expert shape, one rank-16 adapter
    "decode": LayerConfig("decode", T=64, H=2048, I=768, E=128, top_k=8),
    # multi-adapter decode: four resident slots of mixed rank, 10% of tokens without adapter
    "multi_slot": LayerConfig("multi_slot", T=256, H=2048, I=768, E=128, top_k=8,
                              ranks=(8, 16, 32, 64), scalings=(2.0, 1.0, 0.5, 0.25),
                              slot_mode="uniform_none10"),
    # prefill with Zipf-skewed expert load
    "prefill_zipf": LayerConfig("prefill_zipf", T=8192, H=2048, I=768, E=128, top_k=8,
                                zipf_bias=True),
    # Kimi-K2-like expert shape with DeepSeekV3 routing, decode and prefill token counts
    "kimi_decode": LayerConfig("kimi_decode", T=128, H=7168, I=2048, E=384, top_k=8,
                               method=DEEPSEEK_V3, bias_std=0.1, rsf=2.827),
    "kimi_prefill": LayerConfig("kimi_prefill", T=4096, H=7168, I=2048, E=384, top_k=8,
                                method=DEEPSEEK_V3, bias_std=0.1, rsf=2.827),
    # the Kimi-like expert shape with 32 experts (2.8 GB of weights): the same GEMM shapes
    # at a size an ncu capture of every counter can hold
    "kimi_prefill_e32": LayerConfig("kimi_prefill_e32", T=512, H=7168, I=2048, E=32, top_k=8,
                                    method=DEEPSEEK_V3, bias_std=0.1, rsf=2.827),
    # decode with a shared-outer adapter of rank 32 (one A on gate_up, one B on down)
    "shared_outer_decode": LayerConfig("shared_outer_decode", T=64, H=2048, I=768, E=128, top_k=8,
                                       ranks=(32,), scalings=(2.0,), shared_outer=True),
}


def _randn(shape, std, gen, device, dtype=torch.bfloat16):
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=gen)
    return t.to(dtype)


def make_inputs(cfg: LayerConfig, seed: int = 0, device: str = "cpu",
                nan_rank_tail: bool = True, T: Optional[int] = None) -> dict:
    """Draw one seeded instance of `cfg` on `device`.

    The draw order is fixed: logits, hidden, w1, w2, LoRA A_gu, B_gu, A_dn, B_dn,
    correction bias, slot indices.  `T` overrides the token count (the weights do
    not depend on it, so a smaller T with the same seed gives the same weights).
    """
    T = cfg.T if T is None else T
    H, I, E, k, S, R = cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.S, cfg.R
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    logits = torch.empty((T, E), dtype=torch.float32, device=device).normal_(0.0, 1.0, generator=gen)
    if cfg.zipf_bias:
        # Zipf-ranked experts: expert e gets rank 1 + pi(e) for a seeded permutation pi,
        # and a logit bias of 1.5*log(1/rank).
        pgen = torch.Generator(device="cpu")
        pgen.manual_seed(seed)
        rank_of = torch.randperm(E, generator=pgen).to(torch.float64) + 1.0
        bias = (-1.5 * torch.log(rank_of)).to(torch.float32).to(device)
        logits = logits + bias[None, :]
    logits = logits.to(torch.bfloat16)
    hidden = _randn((T, H), 1.0, gen, device)
    w1 = _randn((E, 2 * I, H), 1.0 / math.sqrt(H), gen, device)
    w2 = _randn((E, H, I), 1.0 / math.sqrt(I), gen, device)
    if S > 0:
        Eo = 1 if cfg.shared_outer else E   # experts of the shared-outer weights (A_gu, B_dn)
        A_gu = _randn((S, Eo, R, H), 1.0 / math.sqrt(H), gen, device)
        B_gu = _randn((S, E, 2 * I, R), 0.02, gen, device)
        A_dn = _randn((S, E, R, I), 1.0 / math.sqrt(I), gen, device)
        B_dn = _randn((S, Eo, H, R), 0.02, gen, device)
        if nan_rank_tail:
            for s, r in enumerate(cfg.ranks):
                if r < R:
                    A_gu[s, :, r:, :] = float("nan")
                    B_gu[s, :, :, r:] = float("nan")
                    A_dn[s, :, r:, :] = float("nan")
                    B_dn[s, :, :, r:] = float("nan")
    else:
        A_gu = B_gu = A_dn = B_dn = None
    if cfg.method == DEEPSEEK_V3:
        corr = torch.empty((E,), dtype=torch.float32, device=device).normal_(0.0, cfg.bias_std, generator=gen)
    else:
        corr = None
    slot_idx = make_slot_idx(cfg, T, seed)
    return dict(
        hidden=hidden, router_logits=logits, w1=w1, w2=w2,
        lora_A_gu=A_gu, lora_B_gu=B_gu, lora_A_dn=A_dn, lora_B_dn=B_dn,
        correction_bias=corr, slot_idx=slot_idx.to(device),
        ranks=list(cfg.ranks), scalings=[float(s) for s in cfg.scalings],
        T=T, H=H, I=I, E=E, top_k=k, S=S, R=R, method=cfg.method, rsf=cfg.rsf,
        shared_outer=cfg.shared_outer,
    )


def make_slot_idx(cfg: LayerConfig, T: int, seed: int) -> torch.Tensor:
    """Per-token adapter slot: all slot 0, or uniform over the slots with 10% set to -1."""
    if cfg.S == 0:
        return torch.full((T,), -1, dtype=torch.int32)
    if cfg.slot_mode == "all0":
        return torch.zeros((T,), dtype=torch.int32)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 1)
    s = torch.randint(0, cfg.S, (T,), generator=g, dtype=torch.int64)
    none = torch.rand((T,), generator=g) < 0.10
    s[none] = -1
    return s.to(torch.int32)


def random_small_config(rng, max_T=12, max_E=8) -> LayerConfig:
    """A random tiny layer for property tests (H, I multiples of 64 as the kernels need)."""
    E = int(rng.integers(1, max_E + 1))
    k = int(rng.integers(1, min(E, 3) + 1))
    S = int(rng.integers(1, 4))
    ranks = tuple(int(rng.choice([1, 2, 4, 8, 16])) for _ in range(S))
    scal = tuple(float(rng.choice([0.0, 0.5, 1.0, 2.0])) for _ in range(S))
    return LayerConfig("random", T=int(rng.integers(1, max_T + 1)), H=64 * int(rng.integers(1, 3)),
                       I=64, E=E, top_k=k, ranks=ranks, scalings=scal,
                       slot_mode="uniform_none10",
                       method=int(rng.integers(0, 2)), bias_std=0.1, rsf=float(rng.choice([1.0, 2.5])))


def make_routing(T: int, num_experts: int, top_k: int, seed: int = 0):
    """Routing drawn from outside the layer, for the externally-routed entry: per token
    top_k distinct global expert ids (uniform, seeded) and positive weights uniform in
    [0.05, 1).  Returns (ids int32 [T, k], weights float32 [T, k]) on the CPU."""
    gen = torch.Generator().manual_seed(seed)
    ids = torch.stack([torch.randperm(num_experts, generator=gen)[:top_k] for _ in range(T)]) if T > 0 \
        else torch.zeros((0, top_k), dtype=torch.int64)
    w = torch.rand((T, top_k), generator=gen) * 0.95 + 0.05
    return ids.to(torch.int32), w.to(torch.float32)


def packed_routing_words(ids: torch.Tensor, weights: torch.Tensor) -> torch.Tensor:
    """The routed entry's input encoding of a given routing: int32 words with the expert id
    in the high 16 bits and the weight's bfloat16 bit pattern (torch's round-to-nearest
    conversion) in the low 16 bits."""
    bits = weights.to(torch.bfloat16).view(torch.int16).to(torch.int64) & 0xFFFF
    v = (ids.to(torch.int64) << 16) | bits
    v = torch.where(v >= 2 ** 31, v - 2 ** 32, v)      # the same 32 bits as a signed int32
    return v.to(torch.int32)


def quantize_weights_fp8(w: torch.Tensor, block: int = 128):
    """Block-FP8 copy of expert weights w [E, N, K] (N, K multiples of `block`), as an FP8
    block-quantised checkpoint stores them: per block x block tile a float32 scale
    amax / 448 and e4m3 codes of w / scale (torch's float8_e4m3fn conversion).  Returns
    (codes [E, N, K] uint8 bit patterns, scales [E, N/block, K/block] float32) on w's
    device, one expert at a time so the float32 temporaries stay small."""
    E, N, K = w.shape
    if N % block or K % block:
        raise ValueError("N and K must be multiples of the block size")
    codes = torch.empty((E, N, K), dtype=torch.uint8, device=w.device)
    scales = torch.empty((E, N // block, K // block), dtype=torch.float32, device=w.device)
    for e in range(E):
        wb = w[e].float().reshape(N // block, block, K // block, block)
        amax = wb.abs().amax(dim=(1, 3)).clamp(min=1e-12)
        s = amax / 448.0
        q = (wb / s[:, None, :, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
        codes[e] = q.reshape(N, K).view(torch.uint8)
        scales[e] = s
    return codes, scales


def quantize_weights_nvfp4(w: torch.Tensor, block: int = 16):
    """NVFP4 copy of expert weights w [E, N, K] (K a multiple of `block`), as
    an NVFP4 checkpoint stores them: per expert a float32 tensor scale gs = amax / (6 * 448),
    per block of 16 values along K an e4m3 scale of amax_block / (6 * gs) (torch's
    float8_e4m3fn conversion), and e2m1 codes of w / (scale * gs), the nearest of
    0, 0.5, 1, 1.5, 2, 3, 4, 6, packed two per byte (element 2i in the low nibble).
    Returns (packed [E, N, K/2] uint8, scale codes [E, N, K/block] uint8, tensor scales [E]
    float32) on w's device, one expert at a time."""
    E, N, K = w.shape
    if K % block or block % 2:
        raise ValueError("K must be a multiple of the (even) block size")
    dev = w.device
    grid = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], device=dev)
    packed = torch.empty((E, N, K // 2), dtype=torch.uint8, device=dev)
    scodes = torch.empty((E, N, K // block), dtype=torch.uint8, device=dev)
    gscale = torch.empty((E,), dtype=torch.float32, device=dev)
    for e in range(E):
        wf = w[e].float()
        gs = (wf.abs().max() / 2688.0).clamp(min=1e-12)
        blk = wf.reshape(N, K // block, block)
        sb = (blk.abs().amax(dim=2) / (6.0 * gs)).clamp(max=448.0).to(torch.float8_e4m3fn)
        eff = (sb.float() * gs).clamp(min=1e-30)
        q = blk / eff[:, :, None]
        idx = (q.abs().clamp(max=6.0)[..., None] - grid).abs().argmin(dim=-1)   # nearest magnitude
        code = (idx | ((q < 0).to(torch.int64) << 3)).to(torch.uint8).reshape(N, K)
        packed[e] = code[:, 0::2] | (code[:, 1::2] << 4)
        scodes[e] = sb.view(torch.uint8)
        gscale[e] = gs
    return packed, scodes, gscale
