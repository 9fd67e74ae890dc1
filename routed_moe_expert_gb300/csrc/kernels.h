// Internal launch interface between the C-ABI layer (moe_lora.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace mlk {

constexpr int kMaxSlots = 64;
constexpr int kMaxRank = 128;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kMaxRouteCtas = 256;

// "where" tags of the device status word (bits 8 and up; the low byte is the code)
enum : uint32_t {
  kWhereRouteBarrier = 1, kWhereGemmProducer = 2, kWhereGemmMma = 3, kWhereGemmEpilogue = 4,
  kWhereLoraShrinkGu = 5, kWhereLoraExpandGu = 6, kWhereLoraShrinkDn = 7, kWhereFinalize = 8,
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
};
cudaError_t launch_route_align(const RouteParams& p, int grid, cudaStream_t stream);
int route_max_coop_ctas(int E);

// ---------------------------------------------------------------- grouped GEMM
// out[q, col] = sum_k X[q, k] * W[e*N + row(col), k] for the pairs q of expert e.
// gated = 1: the 128-row weight tile n holds gate rows [64n, 64n+64) and up rows
// [N/2 + 64n, N/2 + 64n + 64); the output row is written interleaved in 64-column
// halves (gate block then up block), i.e. column 128n + j.
struct GemmParams {
  CUtensorMap tmap_w;            // weights [E*N rows, K cols], box {64, 64}
  CUtensorMap tmap_x;            // activations [P rows, K cols], box {64, BN}
  __nv_bfloat16* out;            // [P, N]
  const int32_t* offsets;        // [E + 1]
  uint32_t* status;
  int E, N, K, gated, stages;
};
int gemm_smem_bytes(int bn, int stages, int E);
int gemm_stage_bytes(int bn);
cudaError_t launch_grouped_gemm(const GemmParams& p, int bn, int grid, cudaStream_t stream);

// ---------------------------------------------------------------- elementwise
cudaError_t launch_permute(const __nv_bfloat16* x, const int32_t* perm, int P, int k, int H,
                           __nv_bfloat16* xp, cudaStream_t stream);
cudaError_t launch_activation(const __nv_bfloat16* g, const __nv_bfloat16* d, int P, int I,
                              __nv_bfloat16* a, cudaStream_t stream);

struct LoraSlots {
  int S, E, R;
  int ranks[kMaxSlots];
  float scal[kMaxSlots];
};

struct FinalizeParams {
  const __nv_bfloat16* y;        // [P, H] permuted down output
  const float* v;                // [P, R] down-LoRA shrink (null: no LoRA)
  const __nv_bfloat16* B;        // [S, E, H, R]
  const int32_t* ids;            // [T, k]
  const float* weights;          // [T, k]
  const int32_t* inv;            // [T * k]
  const int32_t* slot_idx;       // [T]
  int T, H, k;
  LoraSlots slots;
  __nv_bfloat16* out;            // [T, H]
  uint32_t* status;
};
cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- LoRA
struct ShrinkParams {
  const __nv_bfloat16* src;      // hidden [T, K] (by_token) or activation [P, K]
  int by_token;
  const int32_t* perm;           // [P]
  const int32_t* ids;            // [T, k]
  const int32_t* slot_idx;       // [T]
  int k, P, K;
  const __nv_bfloat16* A;        // [S, E, R, K]
  LoraSlots slots;
  float* u;                      // [P, R]
  uint32_t* status;
  uint32_t where;
};
cudaError_t launch_lora_shrink(const ShrinkParams& p, cudaStream_t stream);

struct ExpandParams {
  const float* u;                // [P, R]
  const int32_t* perm;
  const int32_t* ids;
  const int32_t* slot_idx;
  int k, P, N;                   // N = 2I
  const __nv_bfloat16* B;        // [S, E, N, R]
  LoraSlots slots;
  __nv_bfloat16* d;              // [P, N], logical [gate | up] order
  uint32_t* status;
};
cudaError_t launch_lora_expand(const ExpandParams& p, cudaStream_t stream);

}  // namespace mlk
