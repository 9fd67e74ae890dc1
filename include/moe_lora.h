/*
 * moe_lora.h -- C ABI of the routed MoE expert layer with per-expert LoRA (sm_103a): bf16
 * expert weights (moe_lora_forward) or FP8 block-scale ones (moe_lora_forward_fp8).
 *
 * The layer (sglang PR #28466 "[LoRA] bf16 MoE-LoRA for trtllm backend with two-stream
 * overlap + routing opts", section "Files changed", launcher row, and section 1 flow (A);
 * vLLM API page "vllm.model_executor.layers.fused_moe.experts.trtllm_lora_moe",
 * TrtLlmBf16LoRAExperts.apply):
 *
 *   route      top-k experts per token from the router logits (Renormalize or DeepSeekV3)
 *   permute    gather token rows into expert-sorted order
 *   gate_up    per expert  g = x . w1[e]^T                    (N = 2I, bf16 out)
 *   LoRA gu    d = scaling[s] * B_gu[s,e] (A_gu[s,e] x)       (bf16, NOT routing-weighted)
 *   activation a = silu(g_gate + d_gate) * (g_up + d_up)        (bf16)
 *   down       y = a . w2[e]^T, plus dd = scaling[s] * B_dn[s,e] (A_dn[s,e] a)
 *   finalize   out[t] = sum_j w[t,j] * (y_j + dd_j)             (bf16)
 *
 * Conventions for every call below:
 *   - Pointers are DEVICE pointers unless the name starts with h_ (host memory).
 *   - bf16 tensors are raw bfloat16 bit patterns (uint16_t), row-major, densely packed,
 *     16-byte aligned (router_logits: 2-byte).  int32/float tensors are 4-byte aligned,
 *     densely packed.
 *   - The caller owns every buffer, including the workspace.  No call allocates device
 *     memory after moe_lora_create, so moe_lora_route/permute/forward can be captured
 *     in a CUDA graph on `stream` (the side stream is forked from and joined back to it).
 *   - Calls are asynchronous on `stream`; they return after enqueueing work.
 *   - Host-side argument checks run before any launch: a bad argument returns
 *     MOE_LORA_ERR_INVALID_ARG (or MOE_LORA_ERR_UNSUPPORTED) and launches nothing.
 *   - Conditions only the device can see (a slot index outside [-1, S), a bounded wait
 *     that ran out) are recorded in a status word inside the workspace and reported by
 *     moe_lora_check_status; the kernels never trap.
 *   - A handle serves one stream at a time (its side stream and events are shared).
 */
#ifndef MOE_LORA_H
#define MOE_LORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_lora_bf16;              /* raw bfloat16 bits */
typedef struct CUstream_st* moe_lora_stream; /* identical to cudaStream_t */
typedef struct moe_lora_handle moe_lora_handle;

typedef enum {
  MOE_LORA_OK = 0,
  MOE_LORA_ERR_INVALID_ARG = 1,        /* shape, pointer or value rejected on the host */
  MOE_LORA_ERR_UNSUPPORTED = 2,        /* valid request outside what the kernels cover */
  MOE_LORA_ERR_WORKSPACE_TOO_SMALL = 3,
  MOE_LORA_ERR_CUDA = 4,               /* a CUDA runtime call failed (see moe_lora_last_cuda_error) */
  MOE_LORA_ERR_TIMEOUT = 5,            /* a bounded device-side wait ran out */
  MOE_LORA_ERR_DEVICE_CHECK = 6        /* device saw a bad value: a slot index outside [-1, S) or a given expert id >= num_experts */
} moe_lora_status;

/* Routing methods (vLLM page, TrtLlmBf16LoRAExperts._supports_routing_method). */
typedef enum {
  MOE_LORA_ROUTE_RENORMALIZE = 0,      /* weights = softmax over the k selected logits */
  MOE_LORA_ROUTE_DEEPSEEK_V3 = 1       /* s = sigmoid(logit); select on s + bias; w = s/sum(s)*rsf */
} moe_lora_routing;

/* moe_lora_args.flags */
#define MOE_LORA_FLAG_LORA_OFF            1u /* base layer only: no LoRA work at all */
#define MOE_LORA_FLAG_FORCE_SINGLE_STREAM 2u /* never fork the LoRA chain to the side stream */
#define MOE_LORA_FLAG_FORCE_TWO_STREAM    4u /* fork even above 256 tokens */
#define MOE_LORA_FLAG_UNFUSED_LORA        8u /* down-LoRA expand in the epilogue (see forward) */
#define MOE_LORA_FLAG_NO_PDL             16u /* launch every kernel fully behind its predecessor */
#define MOE_LORA_FLAG_SHARED_OUTER       32u /* shared-outer LoRA: lora_A_gu [S,1,R,H], lora_B_dn [S,1,H,R] */
#define MOE_LORA_FLAG_DOWN_LORA_SIDE     64u /* narrow placement, two streams: the down LoRA on the side
                                                 stream beside the down GEMM (see forward) */
#define MOE_LORA_FLAG_SEPARATE_SHRINK   128u /* fused placement with packed B: run the LoRA shrinks as
                                                 their own kernels, not as tiles of the GEMMs */

/* Stages that moe_lora_args.prof_events can bracket (two events per stage). */
enum {
  MOE_LORA_STAGE_ROUTE = 0, MOE_LORA_STAGE_PERMUTE = 1, MOE_LORA_STAGE_GATE_UP_GEMM = 2,
  MOE_LORA_STAGE_LORA_GATE_UP = 3, MOE_LORA_STAGE_ACTIVATION = 4, MOE_LORA_STAGE_DOWN_GEMM = 5,
  MOE_LORA_STAGE_LORA_DOWN = 6, MOE_LORA_STAGE_FINALIZE = 7, MOE_LORA_NUM_STAGES = 8
};

/* Sizes that determine the workspace.  S = resident LoRA slots (0 allowed), R = max rank. */
typedef struct {
  int T, H, I, E, top_k, S, R;
} moe_lora_shape;

/* Arguments of moe_lora_forward. */
typedef struct {
  int T;                 /* tokens (0 allowed: nothing is launched)                        */
  int H;                 /* hidden size, multiple of 64, <= 16384                          */
  int I;                 /* per-expert intermediate size, multiple of 64, <= 16384         */
  int E;                 /* experts, 1..1024                                               */
  int top_k;             /* 1..min(E, 32)                                                  */
  int S;                 /* resident LoRA slots, 0..64                                     */
  int R;                 /* max LoRA rank (leading size of the stacked adapters), 0..128   */
  int routing_method;    /* moe_lora_routing                                               */
  float routed_scaling_factor; /* DeepSeekV3 only (applied once, in the routing weights)   */
  int n_group, topk_group;     /* DeepSeekV3 grouping; only 1/1 is supported                */
  const moe_lora_bf16* hidden;        /* [T, H]                                            */
  const moe_lora_bf16* router_logits; /* [T, E]                                            */
  const float* correction_bias;       /* [E], DeepSeekV3 only, else NULL                   */
  const moe_lora_bf16* w1;            /* [E, 2I, H]: rows [0,I) gate, [I,2I) up            */
  const moe_lora_bf16* w2;            /* [E, H, I]                                         */
  const moe_lora_bf16* lora_A_gu;     /* [S, E, R, H] ([S, 1, R, H] shared-outer); rows r < ranks[s] read */
  const moe_lora_bf16* lora_B_gu;     /* [S, E, 2I, R] cols r < ranks[s] are read          */
  const moe_lora_bf16* lora_A_dn;     /* [S, E, R, I]                                      */
  const moe_lora_bf16* lora_B_dn;     /* [S, E, H, R] ([S, 1, H, R] shared-outer)            */
  const int32_t* slot_idx;            /* [T], slot of each token, -1 = no adapter          */
  const int32_t* h_ranks;             /* [S] host, 0 <= ranks[s] <= R                      */
  const float* h_scalings;            /* [S] host, 0 disables the slot                     */
  unsigned flags;                     /* MOE_LORA_FLAG_*                                   */
  /* Optional device outputs (NULL: kept in the workspace). */
  int32_t* topk_ids;                  /* [T, top_k]                                        */
  float* topk_weights;                /* [T, top_k]                                        */
  int32_t* expert_offsets;            /* [E + 1]                                           */
  int32_t* perm;                      /* [T*top_k] permuted position -> expanded index     */
  int32_t* inv_perm;                  /* [T*top_k] expanded index -> permuted position     */
  /* Optional profiling: 2*MOE_LORA_NUM_STAGES cudaEvent_t handles (entries may be NULL);
     events 2i and 2i+1 are recorded around stage i on the stream that runs it. */
  void* const* prof_events;
  /* Optional expand-ready copies of lora_B_gu and lora_B_dn made by moe_lora_pack_lora_b
     (gated = 1 for lora_B_gu, 0 for lora_B_dn, E_b = 1 for a shared-outer lora_B_dn) from
     the SAME h_ranks as this call's (a copy made for other ranks gives wrong results); NULL:
     not given.  Used by the fused LoRA placement (see moe_lora_forward), 16-byte aligned. */
  const moe_lora_bf16* lora_B_gu_packed;
  const moe_lora_bf16* lora_B_dn_packed;
  /* Optional shrink-ready copies of lora_A_gu and lora_A_dn made by moe_lora_pack_lora_a
     (E_a = 1 for a shared-outer lora_A_gu) from the SAME h_ranks; NULL: not given.  Read by
     the tensor-core shrinks (kernels or GEMM tiles) of the fused placement, 16-byte aligned. */
  const moe_lora_bf16* lora_A_gu_packed;
  const moe_lora_bf16* lora_A_dn_packed;
} moe_lora_args;

/* Create a handle on `device`: queries the device, creates the LoRA side stream and the
   fork/join events, resolves the tensor-map encoder.  Call OUTSIDE stream capture.
   Errors: MOE_LORA_ERR_INVALID_ARG (null h), MOE_LORA_ERR_UNSUPPORTED (not sm_103),
   MOE_LORA_ERR_CUDA. */
moe_lora_status moe_lora_create(moe_lora_handle** h, int device);

/* Destroy a handle (synchronizes its side stream first).  NULL is accepted. */
moe_lora_status moe_lora_destroy(moe_lora_handle* h);

/* Static text for a status code. */
const char* moe_lora_status_string(moe_lora_status s);

/* Text of the last CUDA error seen by this library on the calling thread ("" if none). */
const char* moe_lora_last_cuda_error(void);

/* Host-only: bytes of workspace moe_lora_forward needs for `shape`.  No GPU needed.
   Errors: MOE_LORA_ERR_INVALID_ARG. */
moe_lora_status moe_lora_workspace_size(const moe_lora_shape* shape, size_t* bytes);

/* Host-only: the host-side argument checks of moe_lora_forward, without launching.
   Returns MOE_LORA_OK or the code forward would return. */
moe_lora_status moe_lora_validate(const moe_lora_args* a);

/* Routing + expert alignment in one launch (sglang PR #27329 "Experimental fast LoRA
   path", Optimizations: "topk + FlashInfer routed-pack in a single launch", "JIT
   MoE-align"; vLLM page, _unpermute_activation docstring for the expanded index).
   Writes topk_ids/topk_weights [T, top_k] in selection order (higher key first, lower
   expert id first on ties), expert_offsets [E+1] (exclusive prefix of per-expert pair
   counts), perm [T*top_k] (pairs grouped by expert, ascending expanded index
   p = t*top_k + j inside an expert) and inv_perm (its inverse).  correction_bias: [E]
   for DeepSeekV3, else NULL.  `workspace` must hold moe_lora_workspace_size() bytes
   for this T, E, top_k (H, I, S, R may be 0 there).  Errors: INVALID_ARG, UNSUPPORTED
   (n_group/topk_group != 1), WORKSPACE_TOO_SMALL, CUDA. */
moe_lora_status moe_lora_route(moe_lora_handle* h, const moe_lora_bf16* router_logits,
                               const float* correction_bias, int T, int E, int top_k,
                               int routing_method, float routed_scaling_factor,
                               int n_group, int topk_group,
                               int32_t* topk_ids, float* topk_weights, int32_t* expert_offsets,
                               int32_t* perm, int32_t* inv_perm,
                               void* workspace, size_t workspace_bytes, moe_lora_stream stream);

/* Token permute (sglang PR #28466, Files changed, launcher row: "moe::dev::permute (bf16
   gather)"): permuted[q, :] = hidden[perm[q] / top_k, :] for q < T*top_k.
   H multiple of 8.  Errors: INVALID_ARG, CUDA. */
moe_lora_status moe_lora_permute(moe_lora_handle* h, const moe_lora_bf16* hidden,
                                 const int32_t* perm, int T, int H, int top_k,
                                 moe_lora_bf16* permuted, moe_lora_stream stream);

/* Expand-ready copy of a stacked LoRA B for the fused LoRA K-stages of the expert GEMMs
   (sglang PR #28466 section 1, the expand half of merged_experts_fused_moe_lora_add; the
   pages keep B as [S, E, N, R] and reach it per slot).  B: [S, E_b, N, R] bf16 (lora_B_gu
   with N = 2I and gated = 1, or lora_B_dn with N = H and gated = 0; E_b = E, or 1 for a
   shared-outer lora_B_dn).  packed: [E_b * NT * 128, Rs] bf16, caller-owned, 16-byte
   aligned, moe_lora_packed_lora_b_size() bytes, NT = N/128 (gated) or ceil(N/128); row
   (e * NT + nt) * 128 + r is the weight row that row r of the GEMM's 128-row tile nt
   multiplies (gated: gate row 64 nt + r for r < 64, up row N/2 + 64 nt + r - 64 above;
   otherwise row 128 nt + r, zero past N), and its columns hold every slot side by side:
   slot s's B[s, e, n, 0 .. ranks[s]) at columns [coff[s], coff[s] + ranks[s]), zero up to
   coff[s+1] = coff[s] + ranks[s] rounded up to 16; Rs = coff[S].  Columns r >= ranks[s] of
   B are never read.  A weight-load step: call it once when the adapters in the slots
   change, with the ranks every later forward passes; the copy is then read by each forward
   as full 128-byte rows (two per slot and row otherwise).  Enqueued on `stream`.
   Errors: INVALID_ARG (sizes, ranks outside [0, R], all ranks 0, N not a multiple of 128
   when gated, null or misaligned pointers), CUDA. */
moe_lora_status moe_lora_packed_lora_b_size(int S, int E_b, int N, int R, int gated, const int32_t* h_ranks,
                                            size_t* bytes);
moe_lora_status moe_lora_pack_lora_b(moe_lora_handle* h, const moe_lora_bf16* B, int S, int E_b, int N, int R,
                                     int gated, const int32_t* h_ranks, moe_lora_bf16* packed,
                                     moe_lora_stream stream);

/* Shrink-ready copy of a stacked LoRA A for the tensor-core shrinks (sglang PR #28466 section 1,
   the shrink half of merged_experts_fused_moe_lora_add).  A: [S, E_a, R, K] bf16 (lora_A_gu
   with K = H, E_a = E or 1 when shared-outer; lora_A_dn with K = I, E_a = E).  packed:
   [E_a * RS, K] bf16, caller-owned, 16-byte aligned, moe_lora_packed_lora_a_size() bytes:
   row e * RS + aoff[s] + r is A[s, e, r, :] for r < ranks[s], zero up to aoff[s+1] =
   aoff[s] + ranks[s] rounded up to 8; RS = aoff[S].  Every slot's rank rows of an expert are
   then one block, which a shrink copies in one piece per K step instead of one piece per slot
   (used when RS <= 128 by the shrink tiles of the GEMMs, RS <= 256 by the shrink kernel).
   Rows r >= ranks[s] of A are never read.  A weight-load step, as moe_lora_pack_lora_b.
   K a multiple of 8.  Errors: INVALID_ARG (sizes, ranks outside [0, R], all ranks 0, null or
   misaligned pointers), CUDA. */
moe_lora_status moe_lora_packed_lora_a_size(int S, int E_a, int K, int R, const int32_t* h_ranks, size_t* bytes);
moe_lora_status moe_lora_pack_lora_a(moe_lora_handle* h, const moe_lora_bf16* A, int S, int E_a, int K, int R,
                                     const int32_t* h_ranks, moe_lora_bf16* packed, moe_lora_stream stream);

/* The whole layer: out [T, H] bf16.  `workspace` holds moe_lora_workspace_size() bytes;
   its contents on entry do not matter.
   LoRA placement follows the GEMMs' token tile BN (twice the mean pairs per expert,
   rounded up to 16..256):
   - BN >= 32, R a multiple of 8, S <= 8 and S*R <= 256 (unless MOE_LORA_FLAG_UNFUSED_LORA):
     both LoRA shrinks run on the tensor cores over every active slot at once, both
     expands run inside the expert GEMMs as extra tensor-core K-stages (the gate_up delta
     in its own accumulator, so the GEMM output and the delta are rounded to bf16
     separately, as the pages do), and the activation runs in the gate_up GEMM's epilogue.
     With lora_B_dn_packed the down expand's K-stages read the packed copy, one stage per 64
     stacked rank columns; with lora_B_gu_packed so does the gate_up expand when the gate_up
     shrink is the tensor-core kernel (more than 32 stacked active ranks).  The results equal
     those of the per-slot stages.  With a packed B, single-CTA token tiles (BN <= 128) and
     at most 128 active rank rows (each active rank a multiple of 8), the shrink itself runs
     as the first tiles of that GEMM (one per expert token tile; a GEMM tile waits for its
     own shrink tile before its LoRA stages) instead of a kernel of its own, unless
     MOE_LORA_FLAG_SEPARATE_SHRINK.
   - otherwise: the gate_up LoRA chain (shrink + expand into a bf16 delta) runs on the side
     stream beside the permute and gate_up GEMM and joins before the activation (sglang PR
     #28466 section 1 flow (B)).  When the down expand cannot be K-stages (BN 16, R not a
     multiple of 8, S > 8, or MOE_LORA_FLAG_UNFUSED_LORA) the activation and the down
     shrink run as one kernel and the expand runs in the down GEMM's epilogue on the CUDA
     cores; else the down shrink runs after the activation and its expand inside the down
     GEMM.  The side stream is used when T <= 256 unless FORCE_SINGLE_STREAM (sglang PR
     #28466, "Which diagram applies when": decode-shaped batches only).
   With MOE_LORA_FLAG_DOWN_LORA_SIDE on the side-stream placement (bf16 weights), the down
   LoRA (shrink and expand, one kernel, into a bf16 delta per pair) runs on the side stream
   beside the down GEMM and joins before the finalize, which adds it (sglang PR #28466
   section 1 flow (B), the gemm2_done_event overlap the pages left unwired); without the
   flag it stays in the activation kernel and the down GEMM's epilogue.  Elsewhere the flag
   is ignored.
   Kernels after the routing start as programmatic dependents of the previous kernel on
   the stream unless MOE_LORA_FLAG_NO_PDL.
   Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA. */
moe_lora_status moe_lora_forward(moe_lora_handle* h, const moe_lora_args* a, moe_lora_bf16* out,
                                 void* workspace, size_t workspace_bytes, moe_lora_stream stream);

/* Routing given from outside the layer (the vLLM API page "fused_moe/experts/
   trtllm_lora_moe": TrtLlmBf16LoRAExperts.apply packs the top-k as (eid << 16) | w.bf16
   and calls invoke_routed_moe / trtllm_bf16_routed_moe with local_expert_offset,
   local_num_experts and do_finalize).  All pointers are device pointers owned by the
   caller. */
typedef struct {
  const int32_t* packed_topk_ids;   /* [T, top_k]: (global expert id << 16) | bf16 bits of the
                                       routing weight (the id in the high 16 bits, unsigned) */
  int num_experts;                  /* global expert count: ids must lie in [0, num_experts) */
  int local_expert_offset;          /* global id of local expert 0; moe_lora_args.E experts are local */
  int do_finalize;                  /* 1: write `out`; 0: write the unfinalized outputs below */
  float* gemm2_output;              /* [T*top_k, H] fp32 (do_finalize = 0, required): row q = the
                                       down output of the pair at permuted position q, unweighted,
                                       down-LoRA delta included; rows of dropped pairs undefined */
  moe_lora_bf16* activation_output; /* [T*top_k, I] bf16 (do_finalize = 0, optional, 16-byte
                                       aligned): the SwiGLU output of each permuted pair */
  float* expert_weights;            /* [T, top_k] fp32 routing weights (optional) */
  int32_t* expanded_idx_to_permuted_idx; /* [T*top_k] (required for do_finalize = 0): permuted
                                       position of expanded pair t*top_k + j, or -1 when its
                                       expert is not local */
} moe_lora_routed;

/* The layer with the routing given (see moe_lora_routed).  `a` is used as for
   moe_lora_forward except that router_logits, correction_bias, routing_method,
   routed_scaling_factor, n_group, topk_group and the optional routing outputs (topk_ids,
   topk_weights, expert_offsets, perm, inv_perm) are ignored; a->E counts the local experts
   (w1, w2 and the LoRA weights hold those only) and a->E + 1 <= 1024.  A pair whose expert
   is not local is dropped: it adds nothing to `out` (the caller sums the ranks' outputs)
   and maps to -1.  Local pairs are permuted by local expert, then expanded index; the
   dropped pairs follow.  An expert id >= num_experts is reported as
   MOE_LORA_ERR_DEVICE_CHECK by moe_lora_check_status and treated as not local.  The
   workspace size is moe_lora_workspace_size() of the same shape.
   Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA. */
moe_lora_status moe_lora_forward_routed(moe_lora_handle* h, const moe_lora_args* a, const moe_lora_routed* r,
                                        moe_lora_bf16* out, void* workspace, size_t workspace_bytes,
                                        moe_lora_stream stream);

/* FP8 block-scale expert weights, as FP8 block-quantised checkpoints store them (the pages'
   FP8 path: sglang PR #28466, summary, where the FP8 path needs block-quantised weights; section 1
   flow (A) diagram, the FP8 flow's per_token_group_quant_fp8 before the MoE op and its
   post-activation quant before the down GEMM).  e4m3 codes are the OCP 8-bit float E4M3
   bit patterns (no infinities, largest finite value 448).  Device pointers owned by the
   caller; codes 16-byte aligned, scales 4-byte aligned. */
typedef struct {
  const uint8_t* w1;        /* [E, 2I, H] e4m3 codes: rows [0,I) gate, [I,2I) up              */
  const float* w1_scale;    /* [E, 2I/128, H/128]: w1 = code * scale of its 128 x 128 block   */
  const uint8_t* w2;        /* [E, H, I] e4m3 codes                                           */
  const float* w2_scale;    /* [E, H/128, I/128]                                              */
} moe_lora_fp8_weights;

/* The layer of moe_lora_forward with FP8 block-scale expert weights `w` (a->w1 and a->w2
   are not read).  The two base GEMMs read their inputs quantised per token in groups of
   128 along K (s = max(amax, 1e-10) / 448 per group, codes e4m3(v / s) rounded to nearest
   even and saturated, both float32 operations): the permuted hidden rows for the gate_up
   GEMM and the bf16 activation for the down GEMM; each GEMM sums, per 128-wide K block,
   the e4m3 products times the two block scales, in fp32.  The LoRA weights and the LoRA
   chain stay bf16 and read the unquantised hidden rows and activation, as in the pages'
   FP8 flow.  Every other rule (routing, rounding points, slots, ranks, scalings, flags) is
   that of moe_lora_forward, with token tiles of at most 64.  LoRA placement: with both
   expand-ready B copies (lora_B_gu_packed, lora_B_dn_packed) and the fused conditions of
   moe_lora_forward (32-token tiles or wider, R a multiple of 8, S <= 8, S*R <= 256, no
   MOE_LORA_FLAG_UNFUSED_LORA), the fused one: tensor-core shrinks on the bf16 permuted
   rows and activation, the expands as bf16 K-stages inside the FP8 GEMMs (the gate_up
   delta kept in its own accumulator and written as its own bf16 tensor, which the
   activation adds, as the pages do); otherwise the narrow one (side-stream gate_up LoRA,
   down expand in the down GEMM's epilogue).  H and I must be multiples of 128.  The workspace is moe_lora_workspace_size() of the same shape.
   Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA. */
moe_lora_status moe_lora_forward_fp8(moe_lora_handle* h, const moe_lora_args* a, const moe_lora_fp8_weights* w,
                                     moe_lora_bf16* out, void* workspace, size_t workspace_bytes,
                                     moe_lora_stream stream);

/* The FP8 group quantisation of moe_lora_forward_fp8 on its own: codes [rows, K] (e4m3,
   16-byte aligned) and scales [K/128, rows] float32 (scales[g * rows + q] is the scale of
   group g of output row q) of bf16 rows src (16-byte aligned).  With perm (the routing's
   permuted -> expanded map) output row q quantises src row perm[q] / top_k, the permute and
   quant of the gate_up GEMM's input; with perm NULL it quantises src row q.  K a multiple
   of 128.  Errors: INVALID_ARG, CUDA. */
moe_lora_status moe_lora_quant_fp8(moe_lora_handle* h, const moe_lora_bf16* src, const int32_t* perm, int rows,
                                   int K, int top_k, uint8_t* codes, float* scales, moe_lora_stream stream);

/* The FP8 grouped GEMM of moe_lora_forward_fp8 on its own (its down GEMM: fp32 output, no
   LoRA): for every expert e and its rows q in [expert_offsets[e], expert_offsets[e+1]),
     out[q, n] = sum over 128-wide K blocks b of  x_scale[b * P + q] * w_scale[e, n/128, b]
                 * sum_{k in b} e4m3(x[q, k]) * e4m3(w[e*N + n, k])
   (the block-scaled product of FP8 block-quantised checkpoints, sglang PR #28466 summary;
   the tensor cores sum each 128-wide block of e4m3 products, the scales are applied in fp32).
   w [E, N, K] and x [P, K] are e4m3 codes (16-byte aligned), w_scale [E, N/128, K/128] and
   x_scale [K/128, P] float32, expert_offsets [E + 1] int32 (non-decreasing, offsets[E] = P),
   out [P, N] float32 (16-byte aligned).  N and K multiples of 128, P >= 0.  Rows of no
   expert are not written.  Errors: INVALID_ARG, CUDA. */
moe_lora_status moe_lora_grouped_gemm_fp8(moe_lora_handle* h, const uint8_t* w, const float* w_scale,
                                          const uint8_t* x, const float* x_scale, const int32_t* expert_offsets,
                                          int E, int N, int K, int P, float* out, moe_lora_stream stream);

/* NVFP4 expert weights, as NVFP4 checkpoints store them (the pages' other target checkpoint:
   sglang PR #27329, Optimizations, the Kimi-K2.5-NVFP4 target and its "modelopt_fp4"
   quantisation).  Each weight is e2m1(code) * e4m3(block scale) * tensor scale: e2m1 codes
   are the OCP FP4 E2M1 values (sign, 2 exponent bits with bias 1, 1 mantissa bit: 0, 0.5, 1,
   1.5, 2, 3, 4, 6), two per byte with element 2i in the low nibble of byte i; one e4m3 block
   scale (OCP E4M3 bit pattern) per 16 consecutive values along K; one float32 tensor scale
   per expert.  Device pointers owned by the caller; codes 16-byte aligned, block scales and
   tensor scales 4-byte aligned. */
typedef struct {
  const uint8_t* w1;        /* [E, 2I, H/2] packed codes: rows [0,I) gate, [I,2I) up          */
  const uint8_t* w1_sf;     /* [E, 2I, H/16] e4m3 block scales                                */
  const float* w1_gs;       /* [E] tensor scales                                              */
  const uint8_t* w2;        /* [E, H, I/2] packed codes                                       */
  const uint8_t* w2_sf;     /* [E, H, I/16]                                                   */
  const float* w2_gs;       /* [E]                                                            */
} moe_lora_nvfp4_weights;

/* The layer of moe_lora_forward with NVFP4 expert weights `w` (a->w1 and a->w2 are not read).
   The two base GEMMs read their inputs quantised to NVFP4 per row (per token: the permuted
   hidden rows for the gate_up GEMM, the bf16 activation for the down GEMM), all float32
   operations rounded to nearest:
     g = max(amax_row, 1e-10) / 2688;  per 16 values s = e4m3(amax_16 / (6 g)) (nearest even,
     saturated at 448);  q = e2m1(v / (s g)) (nearest even on the e2m1 grid, saturated at 6;
     0 where s g is 0),
   and each GEMM sums, in fp32, the exact products (q s) * (weight code * block scale), then
   multiplies by g and the expert's tensor scale.  The LoRA weights and chain stay bf16 and read
   the unquantised hidden rows and activation.  Every other rule (routing, rounding points,
   slots, ranks, scalings, flags except MOE_LORA_FLAG_UNFUSED_LORA, which is implied) is that of
   moe_lora_forward; the LoRA placement is the narrow one at every token count, with token
   tiles of at most 64.  H must be a multiple of 128 and I of 64.  The workspace is
   moe_lora_workspace_size() of the same shape.  Errors: INVALID_ARG, UNSUPPORTED,
   WORKSPACE_TOO_SMALL, CUDA. */
moe_lora_status moe_lora_forward_nvfp4(moe_lora_handle* h, const moe_lora_args* a, const moe_lora_nvfp4_weights* w,
                                       moe_lora_bf16* out, void* workspace, size_t workspace_bytes,
                                       moe_lora_stream stream);

/* The NVFP4 row quantisation of moe_lora_forward_nvfp4 on its own, for bf16 rows src (16-byte
   aligned): row scales g [rows] float32, and any of the packed codes [rows, K/2] (element 2i
   in the low nibble of byte i), the e4m3 block scales [rows, K/16] and the exact f16 values
   q * s [rows, K] that the GEMMs read (each NULL to skip; codes and f16 values 16-byte aligned,
   g 4-byte aligned).  With perm (the routing's permuted -> expanded map) output row q
   quantises src row perm[q] / top_k, the permute and quant of the gate_up GEMM's input; with
   perm NULL it quantises src row q.  K a multiple of 16 (of 32 with codes).  Errors:
   INVALID_ARG, CUDA. */
moe_lora_status moe_lora_quant_nvfp4(moe_lora_handle* h, const moe_lora_bf16* src, const int32_t* perm, int rows,
                                     int K, int top_k, float* g, uint8_t* codes, uint8_t* block_scales,
                                     uint16_t* deq_f16, moe_lora_stream stream);

/* The NVFP4 grouped GEMM of moe_lora_forward_nvfp4 on its own (its down GEMM: fp32 output, no
   LoRA): for every expert e and its rows q in [expert_offsets[e], expert_offsets[e+1]),
     out[q, n] = x_gs[q] * w_gs[e] * sum_k x[q, k] * e2m1(w[e*N + n, k]) * e4m3(w_sf[e*N + n, k/16])
   with x [P, K] the f16 values of moe_lora_quant_nvfp4 (16-byte aligned), w [E, N, K/2] packed
   codes (16-byte aligned), w_sf [E, N, K/16] e4m3 block scales and w_gs [E], x_gs [P] float32
   (4-byte aligned), expert_offsets [E + 1] int32 (non-decreasing, offsets[E] = P), out [P, N]
   float32 (16-byte aligned).  The products are exact; the tensor cores sum them in fp32.  N a
   multiple of 128, K of 64, P >= 0.  Rows of no expert are not written.  With a few rows per
   expert, K a multiple of 256 and w_sf 16-byte aligned, a kernel for narrow token tiles runs
   (same results up to the order of the fp32 sums).  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
moe_lora_status moe_lora_grouped_gemm_nvfp4(moe_lora_handle* h, const uint8_t* w, const uint8_t* w_sf,
                                            const float* w_gs, const uint16_t* x, const float* x_gs,
                                            const int32_t* expert_offsets, int E, int N, int K, int P, float* out,
                                            moe_lora_stream stream);

/* Routing + expert alignment that allocates nothing and takes no workspace or handle.
   The pages have no counterpart to this call; it exists for callers that cannot call
   cudaMalloc or supply a workspace (plug-ins inside a host framework that owns all device
   memory, allocation-free real-time paths).  Same arguments, outputs and results as
   moe_lora_route.  The kernel's scratch lives in a 512 KiB array inside the library's
   device image, held by every GPU that loads the library until the process exits.  Up to
   512 tokens the routing runs as one thread-block cluster and uses only the array's
   header; above that the routing grid shrinks until its scratch fits (8*E bytes per
   routing CTA), and a shape that cannot fit is rejected with MOE_LORA_ERR_UNSUPPORTED.  The first call on a device
   resolves the array's address on the current device (cudaGetSymbolAddress), so make
   that first call before any stream capture.  All calls share the array: each call
   clears its status word and barrier counter on `stream`, and calls that overlap on the
   GPU race.  A device-side wait that runs out (which such a race can cause) is recorded
   only in the shared array, which no call reads back: the outputs of that call are then
   wrong and nothing reports it.  The array's address is looked up once per device and
   kept for the life of the process, so do not call this on a device after
   cudaDeviceReset (or another reset of its primary context) in the same process.
   Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
moe_lora_status moe_lora_route_noalloc(const moe_lora_bf16* router_logits, const float* correction_bias,
                                       int T, int E, int top_k, int routing_method,
                                       float routed_scaling_factor, int n_group, int topk_group,
                                       int32_t* topk_ids, float* topk_weights, int32_t* expert_offsets,
                                       int32_t* perm, int32_t* inv_perm, moe_lora_stream stream);

/* Cumulative number of this library's kernels launched through `h` (each route, permute,
   forward or routed forward adds the kernels it enqueued; a memset is not counted).  For
   measurement; the pages have no counterpart.  Host-only.  Errors: INVALID_ARG. */
moe_lora_status moe_lora_launch_count(const moe_lora_handle* h, uint64_t* count);

/* Synchronizes `stream`, then reads the device status word the last route/forward on this
   workspace left: MOE_LORA_OK, MOE_LORA_ERR_TIMEOUT or MOE_LORA_ERR_DEVICE_CHECK.
   *detail (optional) receives the raw word (code in the low byte, where in the high bytes). */
moe_lora_status moe_lora_check_status(const void* workspace, moe_lora_stream stream,
                                      uint32_t* detail);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LORA_H */
