"""CPU oracle for the routed MoE expert layer with per-expert LoRA (test infrastructure).

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain definition of what the
layer computes.  Only the test suite, the smoke check and the CPU-baseline leg of
the benchmark may import it; the product path (the CUDA library and its Python
binding) never does.  It shares no code with the CUDA path.

Arithmetic: float64 accumulation with bfloat16 rounding exactly at the stage
boundaries the pages fix -- the gate_up GEMM output and the gate_up LoRA delta are
bf16 tensors (sglang PR #28466 "bf16 MoE-LoRA for trtllm backend", Files changed,
launcher row: bf16 Gemm2 gate_up output, bf16 activation; vLLM API page
"fused_moe/experts/trtllm_lora_moe", TrtLlmBf16LoRAExperts.apply step 1: the
gemm1_lora_delta tensor is bf16), the activation output is bf16 (same launcher
row: "bf16 out, no quant"), and the layer output is bf16.  Everything between
those points (LoRA shrink, down GEMM, down LoRA, finalize sum) stays float64.

The one exception is the DeepSeekV3 selection key: floating point decides an
integer there (which experts are chosen), so the oracle computes that key in the
same float32 arithmetic the kernel uses, step by step (see `sigmoid_f32`).

Readings of points the pages leave open (each also listed in the design notes):
  * w1 rows [0, I) are the gate projection and rows [I, 2I) the up projection
    (vLLM page, apply step 1: "vLLM's w13 order (gate=w1 first, up=w3 second)").
  * `scaling[s]` multiplies the whole B.A.x product (standard LoRA alpha/r).
  * The gate_up delta is not multiplied by the routing weight; the down delta is
    (vLLM page, apply step 1 comment "do NOT multiply by the routing weight (it is
    a pre-SwiGLU bias)"; _finalize_with_w2_lora docstring "already-weighted w2_delta").
  * A token with slot -1, or a slot with scaling 0 or rank 0, gets no delta
    (sglang PR #28466, §2 routed-expert LoRA bullet: "-1 sentinel" for tokens with
    no adapter).
  * Only rows r < ranks[s] of A and columns r < ranks[s] of B are read.
  * Ties in top-k selection go to the lower expert id; a token's selected experts
    are listed in selection order (higher key first, lower id first on ties).
  * The permutation lists pairs expert by expert, ascending expanded index
    p = t*top_k + j inside each expert (vLLM page, _unpermute_activation
    docstring: "expanded_idx = token*top_k + k").
  * Renormalize: weights = softmax over the k selected logits (vLLM page,
    _supports_routing_method lists Renormalize and RenormalizeNaive; softmax of all
    logits followed by renormalising the top k gives the same numbers).
  * DeepSeekV3 with n_group = topk_group = 1: scores s = sigmoid(logit), select on
    s + correction_bias, weights = s_sel / sum(s_sel) * routed_scaling_factor.
  * Shared-outer LoRA (sglang PR #28466 section 2: "shared A on gate_up / shared B on
    down", one weight set for every expert): lora_A_gu is [S, 1, R, H] and lora_B_dn
    [S, 1, H, R]; the gate_up expand (B_gu) and the down shrink (A_dn) stay per expert, and
    every other rule (slots, ranks, scaling, rounding) is that of the per-expert mode.
  * Externally routed entry (moe_lora_forward_routed): the packed word is the expert id
    in the high 16 bits and the bf16 bits of the routing weight (nearest even) in the low
    16 bits; pairs of experts outside the local range are dropped (they add nothing and
    map to permuted index -1) and are aligned after the last local expert; with
    do_finalize=False the returned per-pair down output already holds the down-LoRA
    delta, unweighted (what the vLLM page's _finalize_with_w2_lora adds back).
  * FP8 path (moe_lora_forward_fp8): e4m3 codes without infinities (largest finite
    value 448); one float32 weight scale per 128 x 128 block; the gate_up and down GEMM
    inputs quantised per token in groups of 128 along K with scale
    max(amax, 1e-10) / 448 and codes e4m3(v / s), both float32 operations, rounded to
    nearest even and saturated at +-448; the down GEMM's input is the bf16 activation;
    the LoRA chain reads the unquantised bf16 x and a; the LoRA weights stay bf16.
  * NVFP4 path (moe_lora_forward_nvfp4): e2m1 values in blocks of 16 along K with an e4m3
    block scale and one float32 tensor scale (per expert for the weights, per token for
    the activations); the token scale is max(amax, 1e-10) / (6 * 448), the block scale
    e4m3(amax_block / (6 * token scale)), the codes e2m1(v / (block scale * token scale)),
    every step a float32 operation, roundings to nearest even with saturation; packed
    codes hold element 2i in the low nibble; the quant points and the LoRA chain are those
    of the FP8 path.
"""
from __future__ import annotations

import numpy as np

RENORMALIZE = 0
DEEPSEEK_V3 = 1

# ----------------------------------------------------------------------------
# bf16 rounding of float64 values
# ----------------------------------------------------------------------------

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (8 significant bits,
    ties to even), returned as float64.  One rounding, straight from float64."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        _, e = np.frexp(x)                    # x = m * 2**e with 0.5 <= |m| < 1
        e = np.maximum(e, -125)               # below 2**-126 the bf16 grid is fixed at 2**-133
        q = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)
        q = np.where(np.abs(q) > _BF16_MAX, np.copysign(np.inf, x), q)
    return np.where(np.isfinite(x), q, x)


# ----------------------------------------------------------------------------
# the float32 sigmoid used for the DeepSeekV3 selection key
# ----------------------------------------------------------------------------
# sigma(z) = 1 / (1 + E(-z)), E = exp evaluated by Cody-Waite range reduction
# (W. J. Cody and W. Waite, "Software Manual for the Elementary Functions", 1980):
#   n = rint(x * log2(e)),  r = (x - n*C1) - n*C2  with C1 + C2 = ln 2 and C1 short
#   enough that n*C1 is exact,  exp(x) = 2**n * exp(r),
# and exp(r) from its degree-7 Taylor polynomial in Horner form.  Every operation
# is one IEEE float32 operation rounded to nearest (no fused multiply-add), so the
# CUDA kernel, which spells out the same operations, gets the same bits.

_F = np.float32
_LOG2E = _F(1.4426950408889634)
_LN2_HI = _F(0.693359375)                # 355/512: 9 significant bits
_LN2_LO = _F(-2.12194440054690583e-4)    # ln 2 - 355/512
_TAYLOR = [_F(1.0) / _F(f) for f in (1.0, 1.0, 2.0, 6.0, 24.0, 120.0, 720.0, 5040.0)]  # 1/k!, k=0..7


def exp_f32(x) -> np.ndarray:
    """exp(x) in float32 by the Cody-Waite scheme above; x clamped to [-86, 88]."""
    x = np.asarray(x, dtype=np.float32)
    x = np.minimum(np.maximum(x, _F(-86.0)), _F(88.0))
    n = np.rint(x * _LOG2E).astype(np.float32)
    r = (x - n * _LN2_HI).astype(np.float32)
    r = (r - n * _LN2_LO).astype(np.float32)
    p = np.full_like(r, _TAYLOR[7])
    for c in reversed(_TAYLOR[:7]):
        p = (p * r).astype(np.float32)
        p = (p + c).astype(np.float32)
    two_n = np.ldexp(np.ones_like(p), n.astype(np.int32)).astype(np.float32)
    return (p * two_n).astype(np.float32)


def sigmoid_f32(z) -> np.ndarray:
    """sigma(z) = 1 / (1 + exp(-z)) in float32 (one rounding per operation)."""
    z = np.asarray(z, dtype=np.float32)
    e = exp_f32(-z)
    return (_F(1.0) / (_F(1.0) + e).astype(np.float32)).astype(np.float32)


# ----------------------------------------------------------------------------
# routing
# ----------------------------------------------------------------------------

def _select_topk(keys: np.ndarray, top_k: int) -> np.ndarray:
    """Indices of the top_k largest keys per row, larger key first, lower id first
    on equal keys (a stable sort of -key keeps ids ascending among ties)."""
    order = np.argsort(-keys, axis=1, kind="stable")
    return order[:, :top_k].astype(np.int32)


def route(router_logits, top_k: int, method: int = RENORMALIZE, correction_bias=None,
          routed_scaling_factor: float = 1.0, n_group: int = 1, topk_group: int = 1):
    """Top-k routing of each token (vLLM API page "fused_moe/experts/trtllm_lora_moe",
    TrtLlmBf16LoRAExperts._supports_routing_method: Renormalize, DeepSeekV3).

    router_logits: [T, E] bf16 values (any float dtype holding them exactly).
    Returns topk_ids [T, k] int32 and topk_weights [T, k] float64.
    """
    if n_group != 1 or topk_group != 1:
        raise NotImplementedError("only n_group = topk_group = 1")
    logit = np.asarray(router_logits, dtype=np.float32)
    logit = np.where(np.isnan(logit), np.float32(-np.inf), logit)   # NaN logits never win
    T, E = logit.shape
    if not 1 <= top_k <= E:
        raise ValueError("need 1 <= top_k <= E")
    if method == RENORMALIZE:
        ids = _select_topk(logit.astype(np.float64), top_k)
        sel = np.take_along_axis(logit.astype(np.float64), ids, axis=1)
        ex = np.exp(sel - sel[:, :1])
        w = ex / ex.sum(axis=1, keepdims=True)
    elif method == DEEPSEEK_V3:
        bias = np.asarray(correction_bias, dtype=np.float32)
        s = sigmoid_f32(logit)                                   # [T, E] float32
        key = (s + bias[None, :]).astype(np.float32)             # float32 add, as the kernel
        ids = _select_topk(key, top_k)
        sel = np.take_along_axis(s, ids, axis=1).astype(np.float64)
        w = sel / sel.sum(axis=1, keepdims=True) * float(routed_scaling_factor)
    else:
        raise ValueError("unknown routing method")
    return ids, w


def align(topk_ids, E: int):
    """Group routed pairs by expert.

    Returns expert_offsets [E+1] (exclusive prefix of per-expert counts),
    perm [P] (permuted position -> expanded index p = t*k + j) and inv [P]
    (expanded index -> permuted position; the expanded_idx_to_permuted_idx map of
    the vLLM page, _unpermute_activation docstring).
    """
    flat = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    counts = np.bincount(flat, minlength=E)[:E]
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(flat, kind="stable").astype(np.int32)   # by expert, p ascending within
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int32)
    return offsets, perm, inv


# ----------------------------------------------------------------------------
# the layer
# ----------------------------------------------------------------------------

def silu(z):
    """SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)), float64."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def _experts(x, ids, w, top_k, tok, w1, w2, lora_A_gu, lora_B_gu, lora_A_dn, lora_B_dn, slots,
             ranks, scalings, lora_off, inter, local=None, shared_outer=False, act_quant=None):
    """Per-pair expert math for the pairs of tokens `tok` (see moe_lora_forward).  With
    `local` (a bool mask [T, k]) only those pairs are evaluated.  With `act_quant` (the
    FP8 path) the two base GEMMs read act_quant(x) and act_quant(a) instead of x and a;
    the LoRA shrinks still read x and a.  Returns {(t, j): (y + dd, a)} in float64 (a
    holds bf16 values)."""
    S = len(ranks)
    eo = (lambda e: 0) if shared_outer else (lambda e: e)   # expert index of A_gu and B_dn
    res = {}
    pair_t = np.repeat(tok, top_k)
    pair_j = np.tile(np.arange(top_k), tok.size)
    if local is not None:
        keep = local[pair_t, pair_j]
        pair_t, pair_j = pair_t[keep], pair_j[keep]
    pair_e = ids[pair_t, pair_j]
    # pairs grouped by expert: one matrix product per expert evaluates every pair routed
    # to that expert; pairs are independent
    for e in np.unique(pair_e):
        sel = np.nonzero(pair_e == e)[0]
        ts, js = pair_t[sel], pair_j[sel]
        xe = x[ts]                                               # [n, H]
        W1 = _f64(w1[e])                                         # [2I, H]
        W2 = _f64(w2[e])                                         # [H, I]
        I = W1.shape[0] // 2
        xg = xe if act_quant is None else act_quant(xe)          # the gate_up GEMM's input
        g = round_bf16(xg @ W1.T)                                # [n, 2I]
        d = np.zeros_like(g)
        lora_rows = []
        if not lora_off and S > 0:
            for s in range(S):
                r = int(ranks[s])
                sc = float(scalings[s])
                m = np.nonzero(slots[ts] == s)[0]
                if m.size == 0 or r == 0 or sc == 0.0:
                    continue
                A = _f64(lora_A_gu[s, eo(e)])[:r]                # [r, H]
                B = _f64(lora_B_gu[s, e])[:, :r]                 # [2I, r]
                u = xe[m] @ A.T                                  # [m, r]
                d[m] = round_bf16(sc * (u @ B.T))
                lora_rows.append((s, r, sc, m))
        a = round_bf16(silu(g[:, :I] + d[:, :I]) * (g[:, I:] + d[:, I:]))   # [n, I]
        ag = a if act_quant is None else act_quant(a)            # the down GEMM's input
        y = ag @ W2.T                                            # [n, H]
        dd = np.zeros_like(y)
        for s, r, sc, m in lora_rows:
            A = _f64(lora_A_dn[s, e])[:r]                        # [r, I]
            B = _f64(lora_B_dn[s, eo(e)])[:, :r]                 # [H, r]
            v = a[m] @ A.T                                       # [m, r]
            dd[m] = sc * (v @ B.T)
        for i in range(sel.size):
            res[(int(ts[i]), int(js[i]))] = (y[i] + dd[i], a[i])
            if inter is not None:
                inter[int(ts[i]) * top_k + int(js[i])] = dict(g=g[i], d=d[i], a=a[i], y=y[i], dd=dd[i])
    return res


def _finalize(tok, top_k, H, w, rows, local=None):
    """out_acc[t] = sum over j = 0..k-1, in that order, of w[t,j] * (y + dd) (float64),
    skipping pairs outside `local`."""
    out_acc = np.zeros((tok.size, H), dtype=np.float64)
    for i, t in enumerate(tok):
        acc = np.zeros(H, dtype=np.float64)
        for j in range(top_k):
            if local is not None and not local[t, j]:
                continue
            acc = acc + w[t, j] * rows[(int(t), j)][0]
        out_acc[i] = acc
    return out_acc


def moe_lora_forward(hidden, router_logits, w1, w2, top_k, method=RENORMALIZE,
                     correction_bias=None, routed_scaling_factor=1.0,
                     lora_A_gu=None, lora_B_gu=None, lora_A_dn=None, lora_B_dn=None,
                     slot_idx=None, ranks=(), scalings=(), lora_off=False,
                     tokens=None, keep_intermediates=False, shared_outer=False):
    """Forward of the routed MoE expert layer with per-expert LoRA.

    The stages are those of sglang PR #28466 ("Files changed", launcher row, and
    §1 flow (A)): routing -> permute -> gate_up GEMM (N = 2I) -> LoRA delta added
    before SwiGLU -> down GEMM (+ down LoRA delta) -> weighted top-k finalize; the
    finalize formula is the vLLM page's _finalize_with_w2_lora: for each token, the
    routing-weighted sum over its top-k pairs of the down output plus the
    (routing-weighted) down LoRA delta.

    Per pair p = (t, j) with expert e = topk_ids[t, j] and slot s = slot_idx[t]
    (L = s >= 0 and scalings[s] != 0 and ranks[s] > 0, and not lora_off):
      g  = bf16(w1[e] @ x_t)                                       [2I]
      d  = bf16(scaling_s * B_gu[s,e][:, :r] @ (A_gu[s,e][:r] @ x_t))  if L else 0
      a  = bf16(silu(g[:I] + d[:I]) * (g[I:] + d[I:]))             [I]
      y  = w2[e] @ a                                               [H]
      dd = scaling_s * B_dn[s,e][:, :r] @ (A_dn[s,e][:r] @ a)       if L else 0
      out[t] = bf16(sum_j w[t,j] * (y + dd))

    Arguments are arrays holding bf16 values (w1/w2/LoRA weights may also be any
    object whose [e] / [s, e] indexing returns such an array, so large weights can
    be streamed expert by expert).  `tokens` restricts the layer output to those
    token rows (routing and the permutation are always computed for all tokens;
    tokens are independent given the routing).

    Returns a dict with out [n_tok, H] (float64 holding bf16 values), topk_ids,
    topk_weights, expert_offsets, perm, inv and, if keep_intermediates, the
    per-pair g, d, a, y, dd keyed by expanded index.
    """
    x = _f64(hidden)
    T, H = x.shape
    ids, w = route(router_logits, top_k, method, correction_bias, routed_scaling_factor)
    E = np.asarray(router_logits).shape[1]
    offsets, perm, inv = align(ids, E)
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    slots = np.full(T, -1, dtype=np.int64) if slot_idx is None else np.asarray(slot_idx, dtype=np.int64)
    inter = {} if keep_intermediates else None
    rows = _experts(x, ids, w, top_k, tok, w1, w2, lora_A_gu, lora_B_gu, lora_A_dn, lora_B_dn, slots,
                    ranks, scalings, lora_off, inter, shared_outer=shared_outer)
    # finalize: out[t] = bf16(sum over j = 0..k-1, in that order, of w[t,j] * (y + dd))
    out_acc = _finalize(tok, top_k, H, w, rows)
    res = dict(out=round_bf16(out_acc), topk_ids=ids, topk_weights=w,
               expert_offsets=offsets, perm=perm, inv=inv, tokens=tok)
    if inter is not None:
        res["pairs"] = inter
    return res


# ----------------------------------------------------------------------------
# externally routed entry (routing computed outside the layer)
# ----------------------------------------------------------------------------

def pack_topk(topk_ids, topk_weights):
    """Packed top-k words of the externally-routed API (vLLM API page
    "fused_moe/experts/trtllm_lora_moe", TrtLlmBf16LoRAExperts.apply: "pack it into the
    (eid<<16)|w.bf16 format the routed API expects"): the expert id in the high 16 bits
    and the bf16 bit pattern of the routing weight (rounded to nearest even) in the low
    16 bits, as an int32."""
    ids = np.asarray(topk_ids, dtype=np.int64)
    w = round_bf16(np.asarray(topk_weights, dtype=np.float64)).astype(np.float32)
    bits = (w.view(np.uint32) >> 16).astype(np.int64)
    return ((ids << 16) | bits).astype(np.uint32).view(np.int32)


def unpack_topk(packed):
    """Inverse of pack_topk: expert ids [T, k] int64 and routing weights [T, k] float64."""
    u = np.asarray(packed).astype(np.int32).view(np.uint32).astype(np.int64)
    ids = u >> 16
    w = ((u & 0xFFFF) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    return ids, w


def moe_lora_forward_routed(hidden, packed_topk_ids, w1, w2, top_k, num_experts, local_expert_offset=0,
                            lora_A_gu=None, lora_B_gu=None, lora_A_dn=None, lora_B_dn=None,
                            slot_idx=None, ranks=(), scalings=(), lora_off=False, do_finalize=True,
                            tokens=None, shared_outer=False):
    """The layer with routing given from outside (vLLM API page "fused_moe/experts/
    trtllm_lora_moe": invoke_routed_moe / trtllm_bf16_routed_moe with packed_topk_ids,
    local_expert_offset, local_num_experts and do_finalize).

    packed_topk_ids [T, k]: (global expert id << 16) | bf16 bits of the weight.  w1/w2 and
    the LoRA weights hold the E_loc = len(w1) local experts, global ids
    [local_expert_offset, local_expert_offset + E_loc).  A pair routed to any other expert
    is dropped here: it contributes nothing and its expanded_idx_to_permuted_idx is -1
    (another rank owns that expert; the ranks' partial outputs are summed outside).

    The local pairs are aligned exactly as in moe_lora_forward (by local expert, then
    expanded index); the dropped ones follow after the last local expert.

    do_finalize=True: out[t] = bf16(sum over local j, in j order, of w[t,j] * (y + dd)).
    do_finalize=False: the unfinalized tuple of the page's invoke_routed_moe --
    gemm2_output [P, H] (row q = y + dd of the pair at permuted position q, unweighted;
    the down-LoRA delta is already inside, which is what the page's
    _finalize_with_w2_lora adds), expert_weights [T, k], expanded_idx_to_permuted_idx
    [T*k] (-1 for dropped pairs) and activation [P, I] (rows of dropped pairs are zero).
    `tokens` restricts the evaluated pairs to those tokens' rows (the others are zero).
    """
    x = _f64(hidden)
    T, H = x.shape
    E_loc = len(w1)
    gid, w = unpack_topk(packed_topk_ids)
    if np.any((gid < 0) | (gid >= num_experts)):
        raise ValueError("expert id outside [0, num_experts)")
    lid = gid - int(local_expert_offset)
    local = (lid >= 0) & (lid < E_loc)
    bucket = np.where(local, lid, E_loc)                          # dropped pairs after the local ones
    offsets, perm, inv = align(bucket, E_loc + 1)
    idx_map = np.where(local.reshape(-1), inv, -1).astype(np.int32)
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    slots = np.full(T, -1, dtype=np.int64) if slot_idx is None else np.asarray(slot_idx, dtype=np.int64)
    rows = _experts(x, np.where(local, lid, 0), w, top_k, tok, w1, w2, lora_A_gu, lora_B_gu, lora_A_dn,
                    lora_B_dn, slots, ranks, scalings, lora_off, None, local=local, shared_outer=shared_outer)
    res = dict(topk_ids=gid, topk_weights=w, expert_offsets=offsets[:E_loc + 1], perm=perm,
               expanded_idx_to_permuted_idx=idx_map, local=local, tokens=tok)
    if do_finalize:
        out_acc = _finalize(tok, top_k, H, w, rows, local=local)
        res["out"] = round_bf16(out_acc)
        res["out_acc"] = out_acc
        return res
    P = T * top_k
    I = _f64(w1[0]).shape[0] // 2 if E_loc > 0 else 0
    gemm2 = np.zeros((P, H), dtype=np.float64)
    act = np.zeros((P, I), dtype=np.float64)
    for (t, j), (yd, a) in rows.items():
        q = int(idx_map[t * top_k + j])
        gemm2[q] = yd
        act[q] = a
    res.update(gemm2_output=gemm2, activation=act, expert_weights=w)
    return res



# ----------------------------------------------------------------------------
# FP8 block-scale path: e4m3 weights with one float32 scale per 128 x 128 block, and
# the two GEMM inputs quantised per token in groups of 128 along K
# ----------------------------------------------------------------------------
# The pages' FP8 flow (sglang PR #28466, section 1 flow (A) diagram: the FP8 flow has a
# per_token_group_quant_fp8 step before the MoE op and a post-activation quant before
# the down GEMM; its summary: the FP8 path works on block-quantised checkpoints; sglang PR #27329
# "Experimental fast LoRA path", Optimizations: the FP8 target checkpoint
# Qwen3.5-35B-A3B-FP8).  The LoRA chain of that flow runs on the bf16 hidden states and
# on the bf16 activation (the activation kernel hands the down LoRA its input before
# the quant), so only the base GEMMs see quantised inputs.

E4M3_MAX = 448.0          # largest finite e4m3 value
FP8_BLOCK = 128           # weight blocks are 128 x 128; activation groups are 128 wide
FP8_EPS = np.float32(1e-10)


def e4m3_decode(codes) -> np.ndarray:
    """Value of each e4m3 code byte (the OCP 8-bit floating point format E4M3: a sign bit,
    4 exponent bits with bias 7 and 3 mantissa bits; exponent field 0 holds the
    subnormals m * 2**-9; there are no infinities and S.1111.111 is NaN), float64."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where((c >> 7) != 0, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(ex == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(ex - 7.0))
    mag = np.where((ex == 15) & (m == 7), np.nan, mag)
    return sign * mag


def round_e4m3(x) -> np.ndarray:
    """Nearest e4m3 value of each float64 value, ties to the even mantissa, saturating at
    +-448 (a "satfinite" conversion); NaN stays NaN."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    with np.errstate(invalid="ignore", over="ignore"):
        _, e = np.frexp(ax)             # ax = f * 2**e with 0.5 <= f < 1
        e = np.maximum(e - 1, -6)       # leading-bit exponent; below 2**-6 the step is 2**-9
        quantum = np.exp2(e - 3.0)      # 3 mantissa bits
        q = np.rint(ax / quantum) * quantum
    q = np.minimum(q, E4M3_MAX)
    q = np.where(np.isnan(x), np.nan, q)
    return np.copysign(q, x)


def quant_act_fp8(v, group: int = FP8_BLOCK):
    """Quantise rows of activations per token in groups of `group` consecutive values.

    For a group with largest magnitude amax, the scale is s = max(amax, 1e-10) / 448, and
    the code of a value v is e4m3(v / s).  The scale and the quotient are float32
    operations rounded to nearest, so the codes are a function of the float32 inputs.
    Returns (q [n, K] float64 values on the e4m3 grid, s [n, K / group] float32).
    """
    v32 = np.asarray(v, dtype=np.float32)
    n, K = v32.shape
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    g = v32.reshape(n, K // group, group)
    amax = np.abs(g).max(axis=2)
    s = (np.maximum(amax, FP8_EPS) / np.float32(E4M3_MAX)).astype(np.float32)
    quot = (g / s[:, :, None]).astype(np.float32)
    q = round_e4m3(quot.astype(np.float64))
    return q.reshape(n, K), s


def dequant_act_fp8(q, s, group: int = FP8_BLOCK) -> np.ndarray:
    """q * s with each value's group scale (float64; the products are exact)."""
    q = np.asarray(q, dtype=np.float64)
    n, K = q.shape
    return (q.reshape(n, K // group, group) * np.asarray(s, np.float64)[:, :, None]).reshape(n, K)


def fake_quant_act_fp8(v, group: int = FP8_BLOCK) -> np.ndarray:
    """The values a base GEMM of the FP8 path reads for activations v: dequant(quant(v))."""
    q, s = quant_act_fp8(v, group)
    return dequant_act_fp8(q, s, group)


def dequant_weight_fp8(codes, scale, block: int = FP8_BLOCK) -> np.ndarray:
    """W[n, k] = e4m3(codes[n, k]) * scale[n // block, k // block], float64."""
    w = e4m3_decode(codes)
    N, K = w.shape
    sc = np.asarray(scale, dtype=np.float64)
    rows = np.arange(N) // block
    cols = np.arange(K) // block
    return w * sc[rows[:, None], cols[None, :]]


class Fp8Experts:
    """w[e] -> the dequantised float64 weight of expert e, from codes [E, N, K] (uint8
    e4m3 bit patterns) and scales [E, N/128, K/128] (any arrays or CPU tensors indexable
    by expert, so large weights can be streamed expert by expert)."""

    def __init__(self, codes, scales):
        self.codes, self.scales = codes, scales

    def __getitem__(self, e):
        return dequant_weight_fp8(np.asarray(self.codes[e]), np.asarray(self.scales[e]))

    def __len__(self):
        return len(self.codes)


def moe_lora_forward_fp8(hidden, router_logits, w1_q, w1_scale, w2_q, w2_scale, top_k, method=RENORMALIZE,
                         correction_bias=None, routed_scaling_factor=1.0,
                         lora_A_gu=None, lora_B_gu=None, lora_A_dn=None, lora_B_dn=None,
                         slot_idx=None, ranks=(), scalings=(), lora_off=False, tokens=None,
                         shared_outer=False):
    """The layer of moe_lora_forward with FP8 block-scale expert weights.

    w1_q [E, 2I, H] and w2_q [E, H, I] hold e4m3 codes, w1_scale [E, 2I/128, H/128] and
    w2_scale [E, H/128, I/128] their block scales.  Per pair, with every other step as in
    moe_lora_forward:
      g  = bf16(W1[e] @ fq(x_t))      W1 = dequant(w1_q[e], w1_scale[e]), fq = fake_quant_act_fp8
      y  = W2[e] @ fq(a)              W2 = dequant(w2_q[e], w2_scale[e])
    The LoRA shrinks read the bf16 x_t and a.  Since sum_b s_x[b] s_w[b] sum_{k in b} q_x q_w
    equals the product of the two dequantised operands, the block-scaled GEMM is written as
    that product.
    """
    x = _f64(hidden)
    T, H = x.shape
    ids, w = route(router_logits, top_k, method, correction_bias, routed_scaling_factor)
    E = np.asarray(router_logits).shape[1]
    offsets, perm, inv = align(ids, E)
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    slots = np.full(T, -1, dtype=np.int64) if slot_idx is None else np.asarray(slot_idx, dtype=np.int64)
    rows = _experts(x, ids, w, top_k, tok, Fp8Experts(w1_q, w1_scale), Fp8Experts(w2_q, w2_scale), lora_A_gu,
                    lora_B_gu, lora_A_dn, lora_B_dn, slots, ranks, scalings, lora_off, None,
                    shared_outer=shared_outer, act_quant=fake_quant_act_fp8)
    out_acc = _finalize(tok, top_k, H, w, rows)
    return dict(out=round_bf16(out_acc), topk_ids=ids, topk_weights=w, expert_offsets=offsets, perm=perm,
                inv=inv, tokens=tok)


# ----------------------------------------------------------------------------
# NVFP4 path: e2m1 values in blocks of 16 along K, each block with an e4m3 scale, and one
# float32 scale per tensor (per expert weight; per token for the activations)
# ----------------------------------------------------------------------------
# The pages' other target checkpoint is NVFP4 (sglang PR #27329, Optimizations: the
# Kimi-K2.5-NVFP4 target, "modelopt_fp4" quantisation in its launch commands, with
# activations quantised per token under the per-token activation switch; for NVFP4 the
# permute and the down quantisation are fused with their neighbours).  The pages fix the
# format only by name: NVIDIA's NVFP4, whose element is the OCP FP4 E2M1 value (sign,
# 2 exponent bits with bias 1, 1 mantissa bit: 0, 0.5, 1, 1.5, 2, 3, 4, 6), grouped in
# blocks of 16 that share an e4m3 scale, times one float32 scale per tensor.

E2M1_MAX = 6.0
NVFP4_BLOCK = 16
_NVFP4_RANGE = np.float32(E2M1_MAX * E4M3_MAX)   # 2688: what one tensor scale spans


def e2m1_decode(codes) -> np.ndarray:
    """Value of each 4-bit e2m1 code (bit 3 sign, bits 2-1 exponent with bias 1, bit 0
    mantissa; exponent field 0 holds the subnormals 0 and 0.5), float64."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    sign = np.where((c >> 3) != 0, -1.0, 1.0)
    ex = (c >> 1) & 0x3
    m = (c & 0x1).astype(np.float64)
    mag = np.where(ex == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(ex - 1.0))
    return sign * mag


def unpack_nvfp4(packed) -> np.ndarray:
    """Codes of a packed NVFP4 tensor [..., K/2] (uint8): element 2i is the low nibble of
    byte i and element 2i+1 its high nibble.  Returns codes [..., K]."""
    b = np.asarray(packed).astype(np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out


def round_e2m1(x) -> np.ndarray:
    """Nearest e2m1 value of each float64 value, ties to the even mantissa, saturating at
    +-6 (below 1 the step is 0.5, in [2^e, 2^(e+1)) it is 2^(e-1))."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        _, e = np.frexp(ax)              # ax = f * 2**e with 0.5 <= f < 1
        e = np.maximum(e - 1, 0)         # leading-bit exponent; below 1 the step is 0.5
        quantum = np.exp2(e - 1.0)       # 1 mantissa bit
        q = np.rint(ax / quantum) * quantum
    q = np.minimum(q, E2M1_MAX)
    return np.copysign(q, x)


def quant_act_nvfp4(v, block: int = NVFP4_BLOCK):
    """Quantise rows of activations to NVFP4 with one tensor scale per row (per token).

    With amax_t the row's largest magnitude and amax_b a block's, all float32 operations
    rounded to nearest:
      g   = max(amax_t, 1e-10) / 2688                       (the token's scale, 2688 = 6 * 448)
      s_b = e4m3(amax_b / (6 * g))                          (the block's scale, rounded to nearest
                                                              even and saturated at 448)
      q   = e2m1(v / (s_b * g))  (0 where s_b is 0)         (rounded to nearest even, saturated at 6)
    Returns (q [n, K] float64 e2m1 values, s_b [n, K/block] float64 e4m3 values, g [n] float32).
    """
    v32 = np.asarray(v, dtype=np.float32)
    n, K = v32.shape
    if K % block:
        raise ValueError("K must be a multiple of the block size")
    amax_t = np.abs(v32).max(axis=1)
    g = (np.maximum(amax_t, FP8_EPS) / _NVFP4_RANGE).astype(np.float32)            # [n]
    blk = v32.reshape(n, K // block, block)
    amax_b = np.abs(blk).max(axis=2)                                                # [n, K/block]
    six_g = (np.float32(E2M1_MAX) * g).astype(np.float32)
    sb = round_e4m3((amax_b / six_g[:, None]).astype(np.float32).astype(np.float64))  # e4m3 values
    eff = (sb.astype(np.float32) * g[:, None]).astype(np.float32)                  # [n, K/block]
    with np.errstate(invalid="ignore", divide="ignore"):
        quot = (blk / eff[:, :, None]).astype(np.float32)
    q = np.where(eff[:, :, None] > 0, round_e2m1(quot.astype(np.float64)), 0.0)
    return q.reshape(n, K), sb, g


def dequant_act_nvfp4(q, sb, g, block: int = NVFP4_BLOCK) -> np.ndarray:
    """q * s_b * g for every value (float64; the products are exact)."""
    q = np.asarray(q, dtype=np.float64)
    n, K = q.shape
    s = np.asarray(sb, np.float64)[:, :, None] * np.asarray(g, np.float64)[:, None, None]
    return (q.reshape(n, K // block, block) * s).reshape(n, K)


def fake_quant_act_nvfp4(v, block: int = NVFP4_BLOCK) -> np.ndarray:
    """The values a base GEMM of the NVFP4 path reads for activations v."""
    return dequant_act_nvfp4(*quant_act_nvfp4(v, block), block=block)


def dequant_weight_nvfp4(packed, scale_codes, global_scale, block: int = NVFP4_BLOCK) -> np.ndarray:
    """W[n, k] = e2m1(code[n, k]) * e4m3(scale_codes[n, k // 16]) * global_scale, float64,
    from the packed codes [N, K/2] (uint8), the block scales' e4m3 bit patterns
    [N, K/16] (uint8) and the expert's float32 tensor scale."""
    w = e2m1_decode(unpack_nvfp4(packed))
    N, K = w.shape
    sb = e4m3_decode(scale_codes)
    return w * np.repeat(sb, block, axis=1)[:, :K] * float(np.float32(global_scale))


class Nvfp4Experts:
    """w[e] -> the dequantised float64 weight of expert e, from packed codes [E, N, K/2],
    block scale codes [E, N, K/16] and tensor scales [E]."""

    def __init__(self, packed, scale_codes, global_scales):
        self.packed, self.scale_codes, self.global_scales = packed, scale_codes, global_scales

    def __getitem__(self, e):
        return dequant_weight_nvfp4(np.asarray(self.packed[e]), np.asarray(self.scale_codes[e]),
                                    np.asarray(self.global_scales)[e])

    def __len__(self):
        return len(self.packed)


def moe_lora_forward_nvfp4(hidden, router_logits, w1, w2, top_k, method=RENORMALIZE, correction_bias=None,
                           routed_scaling_factor=1.0, lora_A_gu=None, lora_B_gu=None, lora_A_dn=None,
                           lora_B_dn=None, slot_idx=None, ranks=(), scalings=(), lora_off=False, tokens=None,
                           shared_outer=False):
    """The layer of moe_lora_forward with NVFP4 expert weights.

    w1 and w2 are (packed codes, block scale codes, tensor scales) triples: w1 packed
    [E, 2I, H/2], scales [E, 2I, H/16], tensor scales [E]; w2 the same with [E, H, I/2],
    [E, H, I/16].  The two base GEMMs read NVFP4-quantised inputs (quant_act_nvfp4 per
    token: the permuted hidden rows and the bf16 activation); the LoRA chain reads the
    bf16 values, and every other rule is that of moe_lora_forward.
    """
    x = _f64(hidden)
    T, H = x.shape
    ids, w = route(router_logits, top_k, method, correction_bias, routed_scaling_factor)
    E = np.asarray(router_logits).shape[1]
    offsets, perm, inv = align(ids, E)
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    slots = np.full(T, -1, dtype=np.int64) if slot_idx is None else np.asarray(slot_idx, dtype=np.int64)
    rows = _experts(x, ids, w, top_k, tok, Nvfp4Experts(*w1), Nvfp4Experts(*w2), lora_A_gu, lora_B_gu,
                    lora_A_dn, lora_B_dn, slots, ranks, scalings, lora_off, None, shared_outer=shared_outer,
                    act_quant=fake_quant_act_nvfp4)
    out_acc = _finalize(tok, top_k, H, w, rows)
    return dict(out=round_bf16(out_acc), topk_ids=ids, topk_weights=w, expert_offsets=offsets, perm=perm,
                inv=inv, tokens=tok)
