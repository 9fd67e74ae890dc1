// Internal launch interface between the C-ABI layer (moe_lora.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace mlk {

constexpr int kMaxSlots = 64;
constexpr int kMaxRank = 128;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kMaxRouteCtas = 256;
constexpr int kMaxFusedSlots = 8;   // slots the GEMMs can take as extra LoRA MMA stages
constexpr int kMaxLoraPanels = 8;   // 64-column panels of the stacked ranks of a packed LoRA B

// "where" tags of the device status word (bits 8 and up; the low byte is the code)
enum : uint32_t {
  kWhereRouteBarrier = 1, kWhereGemmProducer = 2, kWhereGemmMma = 3, kWhereGemmEpilogue = 4,
  kWhereLoraShrinkGu = 5, kWhereLoraExpandGu = 6, kWhereLoraShrinkDn = 7, kWhereFinalize = 8,
  kWhereLoraShrinkTc = 9, kWhereRouteExpert = 10,
};

struct LoraSlots {
  int S, E, R;
  int ranks[kMaxSlots];
  float scal[kMaxSlots];
};

// ---------------------------------------------------------------- routing + align
struct RouteParams {
  const __nv_bfloat16* logits;   // [T, E]
  const float* bias;             // [E] (DeepSeekV3) or null
  int T, E, k, method;
  float rsf;
  int tokens_per_cta;
  int32_t* ids;                  // [T, k]
  float* weights;                // [T, k]
  int32_t* offsets;              // [E + 1]
  int32_t* perm;                 // [T * k]
  int32_t* inv;                  // [T * k]
  int32_t* hist;                 // [grid, E] scratch
  int32_t* base;                 // [grid, E] scratch
  int32_t* total;                // [E] scratch
  uint32_t* barrier;             // zeroed before the launch
  uint32_t* status;
  // method 2 (routing given from outside): packed[t*k + j] = (global expert << 16) | bf16
  // weight bits.  Experts [local_offset, local_offset + E - 1) map to buckets 0..E-2; every
  // other pair goes to the last bucket E - 1 and gets inv = -1.
  const int32_t* packed;         // [T, k]
  int ext_experts;               // global expert ids must lie in [0, ext_experts)
  int local_offset;
};
cudaError_t launch_route_align(const RouteParams& p, int grid, cudaStream_t stream);
// Routing as one thread-block cluster of route_cluster_ctas(T) CTAs (no global scratch,
// no grid barrier); 0 when T is too large and the cooperative grid is used instead.
int route_cluster_ctas(int T);
// One thread-block cluster (<= 512 tokens).  It writes the status word once (0 or the first
// routing error), so with pdl it may start behind the previous forward without a memset.
cudaError_t launch_route_cluster(const RouteParams& p, int ctas, cudaStream_t stream, bool pdl = false);
int route_max_coop_ctas(int E);

// ---------------------------------------------------------------- grouped GEMM
// out[q, col] = sum_k X[q, k] * W[e*N + row(col), k] for the pairs q of expert e.
// gated = 1: the 128-row weight tile n holds gate rows [64n, 64n+64) and up rows
// [N/2 + 64n, N/2 + 64n + 64); the output row is written interleaved in 64-column
// halves (gate block then up block), i.e. column 128n + j.
// gated = 2: same tiles; the epilogue applies the activation (plus the LoRA delta of the
// fused stages, rounded separately) and writes a [P, N/2] bf16.
struct GemmParams {
  CUtensorMap tmap_w;            // weights [E*N rows, K cols], box {64, 64}
  CUtensorMap tmap_x;            // activations [P rows, K cols], box {64, BN / cta_pair}
  __nv_bfloat16* out;            // [P, N] bf16 output, or
  float* out_f32;                //   fp32 output when non-null
  CUtensorMap tmap_y;            // the output [P rows, N cols]: fp32 with box {32, 16}, or bf16 (out_f32
                                 // null) with box {32, 32}; whole chunks leave by TMA (y_tma = 1)
  int y_tma;
  const int32_t* offsets;        // [E + 1]
  uint32_t* status;
  int E, N, K, gated, stages;
  int cta_pair;                  // 2: CTA pairs share each tile (M = 256; N/128 even); else 1
  // Optional LoRA expand as extra MMA K-stages of every tile (fused LoRA): for each slot
  // s present among the tile's pairs, A' = rows of lora B of slot s (tmap_lb[s], inner
  // extent ranks[s], so the stacked rank tail reads as zero) and B' = the tile's rows of
  // ub = scaling[s] * bf16(shrink), zero for pairs of other slots (tmap_lu, rows s*P + q).
  CUtensorMap tmap_lb[kMaxFusedSlots];
  CUtensorMap tmap_lu;           // [S*P rows, RU cols] bf16, box {64, BN / cta_pair}
  int lora_fused;                // 1: use the extra stages (pair_slot gives the slots)
  int lora_kb;                   // 64-wide K blocks per slot: ceil(R / 64)
  int P;
  // Optional LoRA expand added in the epilogue before the store (down GEMM, when the
  // fused stages are not usable):
  // out[q, h] += sum_{r<ranks[s]} lora_B[s, e, h, r] * lora_v[q, r]   (s = pair_slot[q])
  // lora_v holds scaling[s] * (down-LoRA shrink), written with pair_slot by the shrink.
  const float* lora_v;           // [P, R] or null
  const __nv_bfloat16* lora_B;   // [S, E, N, R], or [S, 1, N, R] with lora_b_e1
  int lora_b_e1;                 // 1: the LoRA B (epilogue or fused stages) is one set per slot
  const int32_t* pair_slot;      // [P], -1 = no LoRA for the pair
  LoraSlots slots;
  // Fused LoRA from the expand-ready copy of B (lora_packed = 1, replaces the per-slot stages):
  // A' = the tile's 128 rows of the packed B (tmap_lbp: [Eb*NT*128 rows, Rs cols], rows in the
  // tile's own order, slot s's ranks in columns [coff[s], coff[s] + ranks[s]), zero up to
  // coff[s+1]), B' = the tile's rows of the stacked ub (tmap_lup: [P rows, Rs cols], zero
  // outside the pair's own slot).  One stage per 64-column panel j, issued when a slot of
  // lora_panel_slots[j] is present among the tile's pairs.
  CUtensorMap tmap_lbp;          // box {64, 64}
  CUtensorMap tmap_lup;          // box {64, BN / cta_pair}
  int lora_packed;
  int lora_rs;                   // Rs, a multiple of 16
  uint32_t lora_panel_slots[kMaxLoraPanels];
  // The LoRA shrink as tiles of this GEMM (shrink_in_gemm = 1; packed B, single-CTA tiles):
  // one shrink tile per (expert, token tile), all of them in front of the GEMM tiles in the
  // schedule.  Its stages hold every active slot's rank rows of A for the expert (tmap_sa[s],
  // box rows = ranks[s], at row sa_row_off[s] of the weight half; at most 128 rows) and the
  // tile's token rows of X (tmap_x, as the GEMM tiles); its epilogue writes the tile's
  // stacked ub rows (ub_out [P, lora_rs], columns coff), then counts
  // shrink_ready[shrink tile] up (release).  A GEMM tile's producer waits for its own shrink
  // tile (acquire) before it issues the LoRA stages that read those ub rows.  pair_slot
  // then holds each pair's token slot as the permute gathered it (checked where it is read).
  int shrink_in_gemm;
  CUtensorMap tmap_sa[kMaxFusedSlots];
  int sa_row_off[kMaxFusedSlots + 1];
  int sa_packed;                 // 1: tmap_sa[0] is the shrink-ready A [Ea*RS rows, K] (box RS rows), one
                                 //    copy per stage; sa_row_off its slot offsets, sa_R = RS
  int sa_e1;                     // A is [S, 1, R, K]: one set per slot
  int sa_R;                      // rank stride of A's rows: (s * Ea + e) * sa_R
  int coff[kMaxFusedSlots + 1];  // stacked ub columns of slot s
  __nv_bfloat16* ub_out;         // [P, lora_rs]
  const int32_t* perm;           // [P]
  const int32_t* slot_idx;       // [T]
  int k;
  int* shrink_ready;             // [shrink tiles], zero when the kernel starts
};
constexpr int kMaxGemmSmem = 227 * 1024;   // dynamic shared memory a CTA may have
int gemm_smem_bytes(int bn, int cg, int stages, int E, int lora_R, int act_fused, int y_tma);
int gemm_stage_bytes(int rows);   // one stage: 128 weight rows + `rows` token rows, 64 wide
cudaError_t launch_grouped_gemm(const GemmParams& p, int bn, int grid, cudaStream_t stream, bool pdl = false);

// ---------------------------------------------------------------- FP8 grouped GEMM
// out[q, col] = sum_b x_scale[b*P + q] * w_scale[e, n/128, b] * sum_{k in block b}
// X8[q, k] * W8[e*N + n, k] over the 128-wide K blocks b, n = row(col) (gated as in
// GemmParams).  N and K multiples of 128; token tiles of 16, 32 or 64.
struct GemmF8Params {
  CUtensorMap tmap_w;            // e4m3 weights [E*N rows, K cols] (bytes), box {128, 64}
  CUtensorMap tmap_x;            // e4m3 activations [P rows, K cols], box {128, BN}
  const float* w_scale;          // [E, N/128, K/128]
  const float* x_scale;          // [K/128, P]
  __nv_bfloat16* out;            // [P, N] bf16 output, or
  float* out_f32;                //   fp32 output when non-null
  const int32_t* offsets;        // [E + 1]
  uint32_t* status;
  int E, N, K, P, gated, stages;
  // Optional down-LoRA expand in the epilogue (as GemmParams' lora_v path):
  // out[q, n] += sum_{r<ranks[s]} lora_B[s, e, n, r] * lora_v[q, r]   (s = pair_slot[q])
  const float* lora_v;           // [P, R] or null
  const __nv_bfloat16* lora_B;   // [S, E, N, R], or [S, 1, N, R] with lora_b_e1
  int lora_b_e1;
  const int32_t* pair_slot;      // [P], -1 = no LoRA for the pair
  LoraSlots slots;
  // Fused LoRA expand from the expand-ready B (lora_packed = 1, replaces lora_v): after a
  // tile's main K blocks, one bf16 stage per 64-column panel of the stacked ranks (A' = the
  // tile's rows of the packed B, tmap_lbp; B' = the tile's stacked ub rows, tmap_lup), issued
  // when a slot of lora_panel_slots[j] is among the tile's pairs (pair_slot), as tcgen05
  // kind::f16 MMAs into a delta accumulator.  The epilogue adds the delta to the fp32 sum
  // (gated = 0), or stores it rounded to bf16 as d_out [P, N] in the logical column order,
  // zero for pairs without an adapter (gated = 1: the gate_up delta the activation adds).
  CUtensorMap tmap_lbp;          // [Eb*NT*128 rows, Rs cols] bf16, box {64, 64}
  CUtensorMap tmap_lup;          // [P rows, Rs cols] bf16, box {64, BN}
  int lora_packed;
  int lora_rs;
  uint32_t lora_panel_slots[kMaxLoraPanels];
  __nv_bfloat16* d_out;
};
int gemm_fp8_smem_bytes(int bn, int stages, int E, int lora_R, int lora_packed = 0);
int gemm_fp8_stage_bytes(int bn);
cudaError_t launch_grouped_gemm_fp8(const GemmF8Params& p, int bn, int grid, cudaStream_t stream, bool pdl = false);

// ---------------------------------------------------------------- elementwise
cudaError_t launch_permute(const __nv_bfloat16* x, const int32_t* perm, int P, int k, int H,
                           __nv_bfloat16* xp, cudaStream_t stream, bool pdl = false,
                           const int32_t* slot_idx = nullptr, int32_t* slot_out = nullptr,
                           int* zero_out = nullptr, int zero_n = 0);
cudaError_t launch_activation(const __nv_bfloat16* g, const __nv_bfloat16* d, int P, int I,
                              __nv_bfloat16* a, cudaStream_t stream, bool pdl = false);
// FP8 group quantisation of rows (gathered through perm[q] / k when perm is set):
// codes [P, K] e4m3, scale [K/128, P]; K a multiple of 128.
cudaError_t launch_quant_fp8(const __nv_bfloat16* src, const int32_t* perm, int k, int P, int K, uint8_t* codes,
                             float* scale, cudaStream_t stream, bool pdl = false,
                             const int32_t* slot_idx = nullptr, int32_t* slot_out = nullptr);

// ---------------------------------------------------------------- NVFP4 path
// NVFP4 grouped GEMM: the weights are e2m1 codes (two per byte, element 2i in the low nibble)
// with an e4m3 scale per 16 values along K and a float32 scale per expert; the inputs are f16
// rows holding e2m1 * e4m3 values exactly (the NVFP4 quantisation of each row without its
// float32 row scale), with that row scale apart.  Per expert e and its rows q:
//   out[q, col] = x_gs[q] * w_gs[e] * sum_k X[q, k] * e2m1(W[e*N + n, k]) * e4m3(SF[e*N + n, k/16])
// with n = row(col) (gated as in GemmParams).  N a multiple of 128, K of 64; token tiles of
// 16, 32 or 64.
struct GemmNv4Params {
  CUtensorMap tmap_w;            // packed codes [E*N rows, K/2 bytes], box {128, 64}, 128-byte swizzle
  CUtensorMap tmap_x;            // f16 inputs [P rows, K cols], box {64, BN}, 128-byte swizzle
  const uint8_t* w_sf;           // [E, N, K/16] e4m3 block scales
  const float* w_gs;             // [E] expert scales
  const float* x_gs;             // [P] row scales of the inputs
  __nv_bfloat16* out;            // [P, N] bf16 output, or
  float* out_f32;                //   fp32 output when non-null
  const int32_t* offsets;        // [E + 1]
  uint32_t* status;
  int E, N, K, P, gated;
  int stages;                    // f16 weight-tile stages
  int rstages;                   // raw stages (codes and token rows)
  // Optional down-LoRA expand in the epilogue (as GemmParams' lora_v path)
  const float* lora_v;           // [P, R] or null
  const __nv_bfloat16* lora_B;   // [S, E, N, R], or [S, 1, N, R] with lora_b_e1
  int lora_b_e1;
  const int32_t* pair_slot;      // [P], -1 = no LoRA for the pair
  LoraSlots slots;
  // The same operands by address, for the narrow-tile kernel (mma.sync, no tensor maps)
  const uint8_t* w_codes;        // [E*N, K/2] packed codes
  const __half* x16;             // [P, K] f16 inputs
};
int gemm_nvfp4_smem_bytes(int bn, int stages, int rstages, int E, int lora_R);
int gemm_nvfp4_stage_bytes(int bn);    // one f16 weight tile
int gemm_nvfp4_rstage_bytes(int bn);   // one raw stage: codes then the token rows
constexpr int kNv4RawBlocks = 4;                // 64-wide K blocks per raw stage
constexpr int kNv4RawStageBytes = 128 * 32 * kNv4RawBlocks;   // 128 weight rows x 256 e2m1 codes
cudaError_t launch_grouped_gemm_nvfp4(const GemmNv4Params& p, int bn, int grid, cudaStream_t stream, bool pdl = false);
// The NVFP4 grouped GEMM for narrow token tiles (up to 16 tokens of an expert per tile): the
// codes stream through a per-warp cp.async ring, are decoded to f16 in registers and multiplied
// on mma.sync.  K a multiple of 256; w_codes and w_sf 16-byte aligned.
cudaError_t launch_grouped_gemm_nvfp4_narrow(const GemmNv4Params& p, int grid, cudaStream_t stream, bool pdl = false);
// NVFP4 quantisation of rows (row q from src row perm[q] / k, or q without perm): per row
//   g = max(amax, 1e-10) / 2688, per 16 values s = e4m3(amax_16 / (6 g)), q = e2m1(v / (s g))
// (float32 operations, round to nearest even, saturating).  Writes the row scale g[q] and any
// of: deq [P, K] f16 = q * s (exact), codes [P, K/2] (packed), sf [P, K/16] (e4m3 codes).
cudaError_t launch_quant_nvfp4(const __nv_bfloat16* src, const int32_t* perm, int k, int P, int K, float* g,
                               __half* deq, uint8_t* codes, uint8_t* sf, cudaStream_t stream, bool pdl = false,
                               const int32_t* slot_idx = nullptr, int32_t* slot_out = nullptr);


struct FinalizeParams {
  const float* y;                // [P, H] permuted down output (down-LoRA delta included), or
  const __nv_bfloat16* y_bf16;   //   the same rounded to bf16 (when y is null)
  const float* weights;          // [T, k]
  const int32_t* inv;            // [T * k]
  int T, H, k;
  __nv_bfloat16* out;            // [T, H]
  const __nv_bfloat16* dd;       // [P, H] down-LoRA delta per permuted pair, added to y (or null)
};
cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t stream, bool pdl = false);

// ---------------------------------------------------------------- LoRA
// Tensor-core LoRA over expert tiles of 8*ntl pairs: shrink u = A . src (fp32) and, when
// B is set, expand d = bf16(scaling * B . bf16(u)) written in logical [gate | up] order.
// With B null, u is written to u_out [P, R] (down-LoRA shrink).
struct LoraParams {
  const __nv_bfloat16* src;      // hidden [T, K] (by_token) or activation [P, K]
  int by_token;
  const int32_t* perm;           // [P]
  const int32_t* slot_idx;       // [T]
  const int32_t* offsets;        // [E + 1]
  int k, P, K, E, N;             // N: expand output width (2I)
  const __nv_bfloat16* A;        // [S, E, R, K], or [S, 1, R, K] with a_e1
  const __nv_bfloat16* B;        // [S, E, N, R] or null, or [S, 1, N, R] with b_e1
  int a_e1, b_e1;                // 1: that weight holds one set per slot for every expert
  LoraSlots slots;
  float* u_out;                  // [P, R] (shrink only): scaling[s] * u for r < ranks[s]
  __nv_bfloat16* ub_out;         // [S*P, RU] (shrink only): bf16(scaling[s] * u), zero elsewhere
  int RU;                        // row stride of ub_out: R rounded up to 8
  int32_t* pair_slot_out;        // [P] (shrink only): the pair's active slot or -1
  __nv_bfloat16* d_out;          // [P, N] (expand)
  uint32_t* status;
  uint32_t where;
};
size_t lora_smem_bytes(int ntl, int R, int N, bool expand, int E);

// Tensor-core shrink of every slot at once (needs R % 8 == 0 and S*R <= 256): writes
// ub[s][q][r] = bf16(scaling[s] * A[s,e,r,:] . X[q,:]) for q's own slot s and r < ranks[s],
// zero for every other (s, r), and pair_slot[q].
struct ShrinkTcParams {
  CUtensorMap tmap_x;            // X [P rows, K cols], box {64, tb}
  CUtensorMap tmap_a;            // A [S*E*R rows, K cols], box {64, R}
  CUtensorMap tmap_a_slot[kMaxFusedSlots];   // the same rows, box {64, rows of slot s} (per_slot)
  int row_off[kMaxFusedSlots + 1];           // per_slot: first stacked B row of slot s
  int per_slot;                  // 1: only each active slot's rank rows are loaded
  int a_e1;                      // 1: A is [S, 1, R, K], one set per slot for every expert
  int tb;                        // pairs (rows of X) per tile: 16, 32, 64 or 128
  const int32_t* offsets;        // [E + 1]
  const int32_t* perm;           // [P]
  const int32_t* slot_idx;       // [T]
  int k, P, K, E, S, R;
  int stages;                    // pipeline depth (set by the launcher)
  LoraSlots slots;
  __nv_bfloat16* ub;             // [S, P, R], or [P, rs] with ub_stacked
  int packed_a;                  // 1: tmap_a is the shrink-ready A [Ea*RS rows, K], box RS rows, row_off its
                                 //    slot offsets (per_slot set); one copy per stage
  int ub_stacked;                // 1: each pair's row holds every slot's ranks, slot s at column coff[s]
  int rs;                        // stacked columns (ub_stacked), a multiple of 16
  int coff[kMaxFusedSlots + 1];
  int32_t* pair_slot;            // [P]
  uint32_t* status;
};
int lora_shrink_tc_nb(int rows);
// Expand-ready (packed) LoRA B for the fused K-stages: see pack_lora_b_kernel.
struct PackLoraBParams {
  const __nv_bfloat16* B;        // [S, Eb, N, R]
  __nv_bfloat16* Bp;             // [Eb * NT * 128, rs]
  int S, Eb, N, R, NT, gated, rs;
  int ranks[kMaxSlots];
  int coff[kMaxSlots + 1];       // coff[s+1] - coff[s] = ranks[s] rounded up to 16
};
cudaError_t launch_pack_lora_b(const PackLoraBParams& p, cudaStream_t stream);
// Shrink-ready (packed) LoRA A: see pack_lora_a_kernel.
struct PackLoraAParams {
  const __nv_bfloat16* A;        // [S, Ea, R, K]
  __nv_bfloat16* Ap;             // [Ea * RS, K]
  int S, Ea, R, K, RS;
  int ranks[kMaxSlots];
  int aoff[kMaxSlots + 1];       // aoff[s+1] - aoff[s] = ranks[s] rounded up to 8
};
cudaError_t launch_pack_lora_a(const PackLoraAParams& p, cudaStream_t stream);
cudaError_t launch_lora_shrink_tc(const ShrinkTcParams& p, int grid, cudaStream_t stream, bool pdl = false);
cudaError_t launch_lora(const LoraParams& p, int ntl, int grid, cudaStream_t stream, bool pdl = false);

// Permute fused with the gate_up LoRA shrink (fused LoRA placement): xp[q] = x[perm[q]/k],
// ub[s][q][r] = bf16(scaling[s] * A_gu[s,e,r,:] . x[perm[q]/k]) for q's own active slot s and
// r < ranks[s], zero for every other (s, r < RU), pair_slot[q] = that slot or -1.
struct PermuteShrinkParams {
  const __nv_bfloat16* x;        // [T, H] hidden rows
  const int32_t* perm;           // [P]
  const int32_t* offsets;        // [E + 1]
  const int32_t* slot_idx;       // [T]
  const __nv_bfloat16* A;        // [S, E, R, H], or [S, 1, R, H] with a_e1
  int a_e1;
  int H, E, k, P, RU;
  int nr_max;                    // stacked rank rows of all active slots, rounded up to 8 (<= 32)
  LoraSlots slots;
  __nv_bfloat16* xp;             // [P, H]
  __nv_bfloat16* ub;             // [S, P, RU]
  int32_t* pair_slot;            // [P]
  uint32_t* status;
  int* zero_out;                 // [zero_n] cleared (ready flags of the GEMMs that follow), or null
  int zero_n;
};
constexpr int kPermuteShrinkMaxRows = 32;   // stacked active rank rows the fused kernel takes
size_t permute_shrink_smem_bytes(int nr_max, int E, int H);
cudaError_t launch_permute_shrink(const PermuteShrinkParams& p, int grid, cudaStream_t stream, bool pdl = false);

// Activation (gate_up output g plus the bf16 gate_up LoRA delta d, SwiGLU, bf16 out)
// fused with the down-LoRA shrink v = scaling * a . A_dn^T, over expert tiles of up to 8
// pairs.  Writes a [P, I] and v [P, R] (fp32, pairs with an adapter); pair_slot holds each
// pair's slot as the permute gathered it and is rewritten checked (-1 for no adapter).
struct ActShrinkParams {
  const __nv_bfloat16* g;        // [P, 2I] gated-interleaved gate_up output
  const __nv_bfloat16* d;        // [P, 2I] gate_up LoRA delta, logical [gate | up]
  const int32_t* offsets;        // [E+1]
  const __nv_bfloat16* A;        // down LoRA A [S, E, R, I]
  LoraSlots slots;
  int P, I, E;
  __nv_bfloat16* a;              // [P, I]
  float* v;                      // [P, R]
  int32_t* pair_slot;            // [P] in: slot_idx of the pair's token; out: checked slot
  uint32_t* status;
};
cudaError_t launch_act_shrink(const ActShrinkParams& p, int grid, cudaStream_t stream, bool pdl = false);

}  // namespace mlk
