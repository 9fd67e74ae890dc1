// Host side of the C ABI declared in include/moe_lora.h: argument checks, workspace
// layout, tensor maps, stream fork/join and the launch sequence of the layer.
//
// Launch sequence of moe_lora_forward (sglang PR #28466 "bf16 MoE-LoRA for trtllm
// backend", section 1 flows (A) single-stream and (B) two-stream), narrow token tiles:
//   main: route -> [fork] -> permute -> gate_up GEMM -> [join on the LoRA-ready event]
//         -> activation + down-LoRA shrink -> down GEMM (down-LoRA expand in its
//         epilogue, fp32 out) -> finalize
//   side: [wait fork] -> gate_up LoRA shrink + expand (one kernel) -> [record ready]
// Wide token tiles, one stream: route -> permute -> tensor-core shrink -> gate_up GEMM
// (LoRA expand stages, activation epilogue) -> tensor-core shrink -> down GEMM (LoRA
// expand stages) -> finalize.  Kernels are programmatic dependents of their predecessors;
// above 512 tokens a memset of the workspace header precedes the (cooperative) routing.
// Every buffer the side stream touches lives in the caller's workspace, which exists
// before the fork, so nothing is allocated while a graph may be capturing (the
// multi-slot replay bug of sglang PR #28091, Motivation 3, cannot arise).
#include "../../include/moe_lora.h"
#include "kernels.h"

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <string>

using namespace mlk;

namespace {

thread_local char g_last_cuda_error[256] = "";

moe_lora_status cuda_fail(cudaError_t err, const char* what) {
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", what, cudaGetErrorString(err));
  return MOE_LORA_ERR_CUDA;
}

#define ML_CUDA(call, what)                         \
  do {                                              \
    cudaError_t _e = (call);                        \
    if (_e != cudaSuccess) return cuda_fail(_e, what); \
  } while (0)

// A launch of one of this library's kernels, counted on the handle (moe_lora_launch_count).
#define ML_LAUNCH(h, call, what)                    \
  do {                                              \
    ML_CUDA(call, what);                            \
    ++(h)->launches;                                \
  } while (0)

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout (all offsets 256-byte aligned).
struct Layout {
  size_t header, ids, wts, offsets, perm, inv, hist, base, total;
  size_t xp, g, d, a, v, y, pslot, ub;
  size_t sx, sa;   // FP8 path: group scales of the gate_up and down GEMM inputs
  size_t ready;    // ready flags of the shrink tiles inside the gate_up and down GEMMs
  size_t bytes;
};
// Shrink tiles of one GEMM: one per (expert, token tile), at most P / 16 + E.
size_t ready_flags(size_t P, int E) { return P / 16 + static_cast<size_t>(E) + 2; }

Layout layout_for(int T, int H, int I, int E, int k, int R, int S) {
  Layout L;
  size_t off = 0;
  auto take = [&](size_t n) {
    const size_t o = off;
    off += align_up(n, 256);
    return o;
  };
  const size_t P = static_cast<size_t>(T) * k;
  L.header = take(256);
  L.ids = take(P * 4);
  L.wts = take(P * 4);
  const size_t Eb = static_cast<size_t>(E) + 1;   // routing buckets: the experts plus the
                                                  // dropped pairs of the routed entry
  L.offsets = take((Eb + 1) * 4);
  L.perm = take(P * 4);
  L.inv = take(P * 4);
  L.hist = take(static_cast<size_t>(kMaxRouteCtas) * Eb * 4);
  L.base = take(static_cast<size_t>(kMaxRouteCtas) * Eb * 4);
  L.total = take(Eb * 4);
  L.xp = take(P * H * 2);
  L.g = take(P * 2 * I * 2);
  L.d = take(R > 0 ? P * 2 * I * 2 : 0);
  L.a = take(P * I * 2);
  L.v = take(P * R * 4);
  L.y = take(P * H * 4);
  L.pslot = take(R > 0 ? P * 4 : 0);
  // per-slot rows [S, P, R rounded up to 8], or stacked rows [P, sum of ranks rounded up to 16]
  L.ub = take(static_cast<size_t>(S) * P * ((R + 15) / 16 * 16) * 2);
  // The FP8 path keeps its e4m3 GEMM inputs in the xp region ([P, H] bytes) and in the g
  // region ([P, I] bytes, written after the activation has read g); their group scales:
  L.sx = take(P * ((static_cast<size_t>(H) + 127) / 128) * 4);
  L.sa = take(P * ((static_cast<size_t>(I) + 127) / 128) * 4);
  L.ready = take(R > 0 ? 2 * ready_flags(P, E) * 4 : 0);
  L.bytes = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

moe_lora_status check_routing_args(int T, int E, int top_k, int method, const void* logits, const float* bias,
                                   int n_group, int topk_group) {
  if (T < 0 || E < 1 || E > kMaxExperts) return MOE_LORA_ERR_INVALID_ARG;
  if (top_k < 1 || top_k > E || top_k > kMaxTopK) return MOE_LORA_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * top_k > 0x7fffffffLL) return MOE_LORA_ERR_INVALID_ARG;
  if (method != MOE_LORA_ROUTE_RENORMALIZE && method != MOE_LORA_ROUTE_DEEPSEEK_V3) return MOE_LORA_ERR_INVALID_ARG;
  if (T > 0 && logits == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  if (method == MOE_LORA_ROUTE_DEEPSEEK_V3 && bias == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  if (bias != nullptr && !aligned4(bias)) return MOE_LORA_ERR_INVALID_ARG;
  if (n_group > 1 || topk_group > 1) return MOE_LORA_ERR_UNSUPPORTED;
  if (n_group < 0 || topk_group < 0) return MOE_LORA_ERR_INVALID_ARG;
  return MOE_LORA_OK;
}

bool lora_active(const moe_lora_args* a) {
  if ((a->flags & MOE_LORA_FLAG_LORA_OFF) || a->S == 0) return false;
  for (int s = 0; s < a->S; ++s)
    if (a->h_ranks[s] > 0 && a->h_scalings[s] != 0.0f) return true;
  return false;
}

}  // namespace

struct moe_lora_handle {
  int device = 0;
  int num_sms = 0;
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_ready = nullptr;
  EncodeTiledFn encode = nullptr;
  int coop_ctas[kMaxExperts + 1];   // cache of route_max_coop_ctas by E (0 = unknown)
  uint64_t launches = 0;             // kernels launched through this handle
};

extern "C" {

const char* moe_lora_status_string(moe_lora_status s) {
  switch (s) {
    case MOE_LORA_OK: return "ok";
    case MOE_LORA_ERR_INVALID_ARG: return "invalid argument";
    case MOE_LORA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_LORA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_LORA_ERR_CUDA: return "CUDA error";
    case MOE_LORA_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_LORA_ERR_DEVICE_CHECK: return "device-side check failed (slot index outside [-1, S) or expert id out of range)";
  }
  return "unknown status";
}

const char* moe_lora_last_cuda_error(void) { return g_last_cuda_error; }

moe_lora_status moe_lora_workspace_size(const moe_lora_shape* s, size_t* bytes) {
  if (s == nullptr || bytes == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  if (s->T < 0 || s->H < 0 || s->I < 0 || s->E < 1 || s->E > kMaxExperts || s->top_k < 1 || s->top_k > s->E ||
      s->S < 0 || s->R < 0 || s->R > kMaxRank)
    return MOE_LORA_ERR_INVALID_ARG;
  *bytes = layout_for(s->T, s->H, s->I, s->E, s->top_k, s->S > 0 ? s->R : 0, s->S > 0 ? s->S : 0).bytes;
  return MOE_LORA_OK;
}

moe_lora_status moe_lora_validate(const moe_lora_args* a) {
  if (a == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  moe_lora_status st = check_routing_args(a->T, a->E, a->top_k, a->routing_method, a->router_logits,
                                          a->correction_bias, a->n_group, a->topk_group);
  if (st != MOE_LORA_OK) return st;
  if (a->H < 64 || a->H > 16384 || a->H % 64 != 0) return MOE_LORA_ERR_INVALID_ARG;
  if (a->I < 64 || a->I > 16384 || a->I % 64 != 0) return MOE_LORA_ERR_INVALID_ARG;
  if (a->S < 0 || a->S > kMaxSlots || a->R < 0 || a->R > kMaxRank) return MOE_LORA_ERR_INVALID_ARG;
  if (static_cast<long long>(a->E) * 2 * a->I > 0x7fffffffLL || static_cast<long long>(a->E) * a->H > 0x7fffffffLL)
    return MOE_LORA_ERR_INVALID_ARG;
  if (a->T == 0) return MOE_LORA_OK;
  if (a->hidden == nullptr || a->w1 == nullptr || a->w2 == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  if (!aligned16(a->hidden) || !aligned16(a->w1) || !aligned16(a->w2)) return MOE_LORA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a->router_logits) & 1u) != 0) return MOE_LORA_ERR_INVALID_ARG;
  if (!(a->flags & MOE_LORA_FLAG_LORA_OFF) && a->S > 0) {
    if (a->h_ranks == nullptr || a->h_scalings == nullptr || a->slot_idx == nullptr) return MOE_LORA_ERR_INVALID_ARG;
    for (int s = 0; s < a->S; ++s) {
      if (a->h_ranks[s] < 0 || a->h_ranks[s] > a->R) return MOE_LORA_ERR_INVALID_ARG;
      if (a->h_scalings[s] != a->h_scalings[s]) return MOE_LORA_ERR_INVALID_ARG;   // NaN scaling
    }
    if (lora_active(a)) {
      if (a->lora_A_gu == nullptr || a->lora_B_gu == nullptr || a->lora_A_dn == nullptr || a->lora_B_dn == nullptr)
        return MOE_LORA_ERR_INVALID_ARG;
      if (!aligned16(a->lora_A_gu) || !aligned16(a->lora_A_dn) || !aligned16(a->lora_B_gu) ||
          !aligned16(a->lora_B_dn) || !aligned4(a->slot_idx))
        return MOE_LORA_ERR_INVALID_ARG;
      if (!aligned16(a->lora_B_gu_packed) || !aligned16(a->lora_B_dn_packed) || !aligned16(a->lora_A_gu_packed) ||
          !aligned16(a->lora_A_dn_packed))
        return MOE_LORA_ERR_INVALID_ARG;
    }
  }
  const void* opt[] = {a->topk_ids, a->topk_weights, a->expert_offsets, a->perm, a->inv_perm};
  for (const void* o : opt)
    if (o != nullptr && !aligned4(o)) return MOE_LORA_ERR_INVALID_ARG;
  return MOE_LORA_OK;
}

moe_lora_status moe_lora_create(moe_lora_handle** out, int device) {
  if (out == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  *out = nullptr;
  int count = 0;
  ML_CUDA(cudaGetDeviceCount(&count), "cudaGetDeviceCount");
  if (device < 0 || device >= count) return MOE_LORA_ERR_INVALID_ARG;
  int major = 0, minor = 0, sms = 0;
  ML_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device), "cudaDeviceGetAttribute");
  ML_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device), "cudaDeviceGetAttribute");
  ML_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device), "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3) return MOE_LORA_ERR_UNSUPPORTED;   // built for sm_103a only
  int prev = 0;
  ML_CUDA(cudaGetDevice(&prev), "cudaGetDevice");
  ML_CUDA(cudaSetDevice(device), "cudaSetDevice");
  moe_lora_handle* h = new moe_lora_handle();
  h->device = device;
  h->num_sms = sms;
  std::memset(h->coop_ctas, 0, sizeof(h->coop_ctas));
  cudaError_t err = cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking);
  if (err == cudaSuccess) err = cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming);
  if (err == cudaSuccess) err = cudaEventCreateWithFlags(&h->ev_ready, cudaEventDisableTiming);
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (err == cudaSuccess)
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  cudaSetDevice(prev);
  if (err != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
    moe_lora_destroy(h);
    return err != cudaSuccess ? cuda_fail(err, "moe_lora_create") : MOE_LORA_ERR_CUDA;
  }
  h->encode = reinterpret_cast<EncodeTiledFn>(fn);
  *out = h;
  return MOE_LORA_OK;
}

moe_lora_status moe_lora_destroy(moe_lora_handle* h) {
  if (h == nullptr) return MOE_LORA_OK;
  if (h->side) {
    cudaStreamSynchronize(h->side);
    cudaStreamDestroy(h->side);
  }
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_ready) cudaEventDestroy(h->ev_ready);
  delete h;
  return MOE_LORA_OK;
}

}  // extern "C"

namespace {

// Routing + align.  With `ext` the top-k comes packed from outside: E is then the number of
// buckets (the local experts plus one for the dropped pairs).
moe_lora_status enqueue_route(moe_lora_handle* h, const moe_lora_bf16* logits, const float* bias, int T, int E,
                              int k, int method, float rsf, int32_t* ids, float* wts, int32_t* offsets,
                              int32_t* perm, int32_t* inv, uint8_t* ws, const Layout& L, cudaStream_t stream,
                              const moe_lora_routed* ext = nullptr, bool pdl = false) {
  if (h->coop_ctas[E] == 0) h->coop_ctas[E] = route_max_coop_ctas(E);
  // above 512 tokens: a cooperative grid of about 64 tokens per CTA
  int grid = (T + 63) / 64;
  if (grid > h->coop_ctas[E]) grid = h->coop_ctas[E];
  if (grid > kMaxRouteCtas) grid = kMaxRouteCtas;
  if (grid < 1) grid = 1;
  RouteParams p;
  std::memset(&p, 0, sizeof(p));
  p.logits = reinterpret_cast<const __nv_bfloat16*>(logits);
  p.bias = bias;
  p.T = T;
  p.E = E;
  p.k = k;
  p.method = method;
  if (ext != nullptr) {
    p.method = 2;
    p.packed = ext->packed_topk_ids;
    p.ext_experts = ext->num_experts;
    p.local_offset = ext->local_expert_offset;
  }
  p.rsf = rsf;
  p.tokens_per_cta = (T + grid - 1) / grid;
  p.ids = ids;
  p.weights = wts;
  p.offsets = offsets;
  p.perm = perm;
  p.inv = inv;
  p.hist = reinterpret_cast<int32_t*>(ws + L.hist);
  p.base = reinterpret_cast<int32_t*>(ws + L.base);
  p.total = reinterpret_cast<int32_t*>(ws + L.total);
  p.status = reinterpret_cast<uint32_t*>(ws + L.header);
  p.barrier = p.status + 1;
  const int ctas = route_cluster_ctas(T);   // one thread-block cluster up to 512 tokens
  if (ctas > 0) {
    p.tokens_per_cta = (T + ctas - 1) / ctas;
    ML_LAUNCH(h, launch_route_cluster(p, ctas, stream, pdl), "route cluster launch");
    return MOE_LORA_OK;
  }
  ML_LAUNCH(h, launch_route_align(p, grid, stream), "route_align launch");
  return MOE_LORA_OK;
}

bool make_tmap(EncodeTiledFn enc, CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token-tile width from the mean number of pairs per expert.
int pick_bn(long long P, int E) {
  const long long m2 = 2 * ((P + E - 1) / E);
  if (m2 <= 16) return 16;
  if (m2 <= 32) return 32;
  if (m2 <= 64) return 64;
  if (m2 <= 128) return 128;
  return 256;
}

// Wide token tiles run on CTA pairs (M = 256 tcgen05 pair MMAs, each SM loading half the
// token rows) when the weight rows split into an even number of 128-row tiles.
constexpr int kPairMinBn = 128;
// From this token tile on the down GEMM stores y (its output plus the down-LoRA delta) in
// bf16 for the finalize, halving the [P, H] round trip through HBM that prefill token counts
// pay for it; narrower tiles keep it in fp32.  The pages leave y's precision open (only g,
// the LoRA delta, the activation and the layer output are bf16 tensors there); the rounding
// costs about 0.3% relative L2 against the float64 oracle, inside the layer's 0.5% bound.
constexpr int kBf16YMinBn = 128;
int pair_tiles(int bn, int N) { return (bn >= kPairMinBn && N % 256 == 0) ? 2 : 1; }

// Pipeline depth from a shared-memory budget.  At narrow token tiles the gate_up GEMM leaves
// room for the side-stream LoRA kernel that runs beside it; the down GEMM runs alone.
int pick_stages(int bn, int cg, int E, int lora_R, int act_fused, bool alone, bool y_tma) {
  // Wide tiles (prefill) keep too few stages in flight to cover the load latency at 200 KB,
  // so they take the whole 227 KB a CTA may have.
  const int budget = bn >= 64 ? kMaxGemmSmem : (bn <= 32 && !alone ? 160 : 200) * 1024;
  const int fixed = gemm_smem_bytes(bn, cg, 0, E, lora_R, act_fused, y_tma);
  int s = (budget - fixed) / (gemm_stage_bytes(bn / cg) + 16);
  if (s > 16) s = 16;
  if (s < 2) s = 2;
  return s;
}

// pdl: programmatic launch behind the previous kernel of the stream, which must not be the
// one that wrote the expert offsets (the GEMM reads them before it waits).
moe_lora_status enqueue_gemm(moe_lora_handle* h, GemmParams& gp, const void* W, const void* X, int P, int bn,
                             cudaStream_t stream, bool pdl) {
  const int cg = gp.cta_pair == 2 ? 2 : 1;
  if (!make_tmap(h->encode, &gp.tmap_w, W, static_cast<uint64_t>(gp.E) * gp.N, gp.K, 64)) return MOE_LORA_ERR_CUDA;
  if (!make_tmap(h->encode, &gp.tmap_x, X, static_cast<uint64_t>(P), gp.K, bn / cg)) return MOE_LORA_ERR_CUDA;
  // The down GEMM's epilogue stores whole 16-token chunks of y (fp32, or bf16 at wide tiles)
  // with TMA; the gate_up outputs and the CUDA-core LoRA epilogue store from the lanes.
  const bool y_f32 = gp.out_f32 != nullptr;
  if (gp.gated == 0 && P >= 16 && (y_f32 || (gp.out != nullptr && gp.lora_v == nullptr))) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(gp.N), static_cast<cuuint64_t>(P)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(gp.N) * (y_f32 ? 4 : 2)};
    cuuint32_t box[2] = {32, y_f32 ? 16u : 32u};   // fp32: 16-token chunks; bf16: 32-token chunks
    cuuint32_t estr[2] = {1, 1};
    void* base = y_f32 ? static_cast<void*>(gp.out_f32) : static_cast<void*>(gp.out);
    if (h->encode(&gp.tmap_y, y_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_LORA_ERR_CUDA;
    gp.y_tma = 1;
  }
  gp.stages = pick_stages(bn, cg, gp.E, gp.lora_v != nullptr ? gp.slots.R : 0, gp.gated == 2, gp.gated == 0,
                          gp.y_tma != 0);
  ML_LAUNCH(h, launch_grouped_gemm(gp, bn, h->num_sms, stream, pdl), "grouped_gemm launch");
  return MOE_LORA_OK;
}

// e4m3 rows [rows, cols] (one byte each) in 128-byte-swizzled boxes of 128 x box_rows.
bool make_tmap_e4m3(EncodeTiledFn enc, CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The FP8 grouped GEMM: weights W8 [E*N, K], inputs X8 [P, K], token tiles of bn (16..64).
// Pipeline depth from the same shared-memory budgets as the bf16 GEMM.
moe_lora_status enqueue_gemm_fp8(moe_lora_handle* h, GemmF8Params& gp, const uint8_t* W, const uint8_t* X, int P,
                                 int bn, cudaStream_t stream, bool pdl) {
  if (!make_tmap_e4m3(h->encode, &gp.tmap_w, W, static_cast<uint64_t>(gp.E) * gp.N, gp.K, 64))
    return MOE_LORA_ERR_CUDA;
  if (!make_tmap_e4m3(h->encode, &gp.tmap_x, X, static_cast<uint64_t>(P), gp.K, bn)) return MOE_LORA_ERR_CUDA;
  const int lora_R = gp.lora_v != nullptr ? gp.slots.R : 0;
  // narrow gate_up tiles leave room for the side-stream LoRA kernel (none beside packed stages)
  const int budget = (bn <= 32 && gp.gated != 0 && !gp.lora_packed ? 160 : 200) * 1024;
  int stages = (budget - gemm_fp8_smem_bytes(bn, 0, gp.E, lora_R, gp.lora_packed)) / (gemm_fp8_stage_bytes(bn) + 16);
  if (stages > 16) stages = 16;
  if (stages < 2) stages = 2;
  gp.stages = stages;
  gp.P = P;
  ML_LAUNCH(h, launch_grouped_gemm_fp8(gp, bn, h->num_sms, stream, pdl), "grouped_gemm_fp8 launch");
  return MOE_LORA_OK;
}

// The NVFP4 grouped GEMM: packed codes W [E*N, K/2], f16 inputs X [P, K], token tiles of bn
// (16..64).  Five f16 weight-tile stages; the rest of the budget goes to raw stages (codes and
// token rows), the kernel's bytes in flight.
moe_lora_status enqueue_gemm_nvfp4(moe_lora_handle* h, GemmNv4Params& gp, const uint8_t* W, const __half* X, int P,
                                   int bn, cudaStream_t stream, bool pdl) {
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(gp.K / 2), static_cast<cuuint64_t>(gp.E) * gp.N};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(gp.K / 2)};
    cuuint32_t box[2] = {128, 64};
    cuuint32_t estr[2] = {1, 1};
    if (h->encode(&gp.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(W), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_LORA_ERR_CUDA;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(gp.K), static_cast<cuuint64_t>(P)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(gp.K) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(bn)};
    cuuint32_t estr[2] = {1, 1};
    if (h->encode(&gp.tmap_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(X), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_LORA_ERR_CUDA;
  }
  gp.w_codes = W;
  gp.x16 = X;
  gp.P = P;
  // a few tokens per expert: the codes decoded in registers, mma.sync (its scale rows are copied
  // 16 bytes at a time)
  if (bn <= 16 && gp.K % 256 == 0 && aligned16(gp.w_sf)) {
    ML_LAUNCH(h, launch_grouped_gemm_nvfp4_narrow(gp, 2 * h->num_sms, stream, pdl), "grouped_gemm_nvfp4 launch");
    return MOE_LORA_OK;
  }
  const int lora_R = gp.lora_v != nullptr ? gp.slots.R : 0;
  // (the weight stream is a quarter of the bf16 GEMM's: the kernel is short, and the whole
  // shared memory serves its rings even beside the side-stream LoRA kernel)
  const int budget = kMaxGemmSmem;
  gp.stages = 5;
  int rs = (budget - gemm_nvfp4_smem_bytes(bn, gp.stages, 0, gp.E, lora_R)) / (gemm_nvfp4_rstage_bytes(bn) + 16);
  if (rs > 8) rs = 8;
  if (rs < 2) return MOE_LORA_ERR_UNSUPPORTED;
  gp.rstages = rs;
  gp.P = P;
  ML_LAUNCH(h, launch_grouped_gemm_nvfp4(gp, bn, h->num_sms, stream, pdl), "grouped_gemm_nvfp4 launch");
  return MOE_LORA_OK;
}

LoraSlots make_slots(const moe_lora_args* a) {
  LoraSlots L;
  std::memset(&L, 0, sizeof(L));
  L.S = a->S;
  L.E = a->E;
  L.R = a->R;
  for (int s = 0; s < a->S; ++s) {
    L.ranks[s] = a->h_ranks[s];
    L.scal[s] = a->h_scalings[s];
  }
  return L;
}

// Tensor maps of the fused LoRA stages: per active slot, the slot's B rows [E*N, ranks[s]]
// (the inner extent stops at the slot's rank, so the stacked tail is zero-filled, never
// read), and the per-slot scaled shrink rows ub [S*P, RU].
bool fuse_lora_maps(moe_lora_handle* h, GemmParams& gp, const moe_lora_args* a, const moe_lora_bf16* B, int N,
                    const __nv_bfloat16* ub, const int32_t* pair_slot, int P, int bn, bool b_e1 = false) {
  const cuuint32_t box_rows = 64;
  const int R = a->R;
  const int RU = (R + 7) & ~7;
  const int Eb = b_e1 ? 1 : a->E;   // expert sets in B (one per slot when shared)
  for (int s = 0; s < a->S; ++s) {
    if (a->h_ranks[s] <= 0 || a->h_scalings[s] == 0.0f) continue;   // never in pair_slot
    const moe_lora_bf16* base = B + static_cast<size_t>(s) * Eb * N * R;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a->h_ranks[s]), static_cast<cuuint64_t>(Eb) * N};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(R) * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    if (h->encode(&gp.tmap_lb[s], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<moe_lora_bf16*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  if (!make_tmap(h->encode, &gp.tmap_lu, ub, static_cast<uint64_t>(a->S) * P, RU, bn / (gp.cta_pair == 2 ? 2 : 1)))
    return false;
  gp.lora_fused = 1;
  gp.lora_b_e1 = b_e1 ? 1 : 0;
  gp.lora_kb = (R + 63) / 64;
  gp.slots = make_slots(a);   // the stages of slot s stop at ranks[s]
  gp.P = P;
  gp.pair_slot = pair_slot;
  return true;
}

// Stacked LoRA columns of the packed layout: slot s's ranks at coff[s], each slot's block
// rounded up to 16 columns (one MMA K-step), from the ranks alone.  Returns Rs = coff[S].
int stacked_cols(const int32_t* ranks, int S, int* coff) {
  coff[0] = 0;
  for (int s = 0; s < S; ++s) coff[s + 1] = coff[s] + (ranks[s] > 0 ? (ranks[s] + 15) / 16 * 16 : 0);
  return coff[S];
}

// Stacked rows of the shrink-ready A: slot s's ranks at row aoff[s] of an expert's block, each
// slot's block rounded up to 8 rows (a swizzle atom), from the ranks alone.  Returns RS = aoff[S].
int stacked_rows(const int32_t* ranks, int S, int* aoff) {
  aoff[0] = 0;
  for (int s = 0; s < S; ++s) aoff[s + 1] = aoff[s] + (ranks[s] > 0 ? (ranks[s] + 7) / 8 * 8 : 0);
  return aoff[S];
}

// Tensor maps of the fused LoRA stages from the expand-ready (packed) B [Eb*NT*128, Rs] and
// the stacked ub [P, Rs], and the slots whose columns meet each 64-column panel.
bool packed_lora_tmaps(moe_lora_handle* h, const moe_lora_args* a, const moe_lora_bf16* Bp, int N, bool gated,
                       bool b_e1, const __nv_bfloat16* ub, int P, int ub_box_rows, CUtensorMap* lbp, CUtensorMap* lup,
                       int* rs_out, uint32_t* panel_slots) {
  int coff[kMaxFusedSlots + 1];
  if (a->S > kMaxFusedSlots) return false;
  const int rs = stacked_cols(a->h_ranks, a->S, coff);
  const int npan = (rs + 63) / 64;
  if (rs == 0 || npan > kMaxLoraPanels) return false;
  const int NT = gated ? (N >> 7) : ((N + 127) >> 7);
  const int Eb = b_e1 ? 1 : a->E;
  if (!make_tmap(h->encode, lbp, Bp, static_cast<uint64_t>(Eb) * NT * 128, static_cast<uint64_t>(rs), 64)) return false;
  if (!make_tmap(h->encode, lup, ub, static_cast<uint64_t>(P), static_cast<uint64_t>(rs),
                 static_cast<uint32_t>(ub_box_rows)))
    return false;
  for (int j = 0; j < kMaxLoraPanels; ++j) panel_slots[j] = 0;
  for (int s = 0; s < a->S; ++s) {
    if (a->h_ranks[s] <= 0 || a->h_scalings[s] == 0.0f) continue;   // never in pair_slot
    for (int j = coff[s] / 64; j * 64 < coff[s + 1]; ++j) panel_slots[j] |= 1u << s;
  }
  *rs_out = rs;
  return true;
}

bool fuse_lora_maps_packed(moe_lora_handle* h, GemmParams& gp, const moe_lora_args* a, const moe_lora_bf16* Bp,
                           int N, const __nv_bfloat16* ub, const int32_t* pair_slot, int P, int bn,
                           bool b_e1 = false) {
  int rs = 0;
  if (!packed_lora_tmaps(h, a, Bp, N, gp.gated != 0, b_e1, ub, P, bn / (gp.cta_pair == 2 ? 2 : 1), &gp.tmap_lbp,
                         &gp.tmap_lup, &rs, gp.lora_panel_slots))
    return false;
  gp.lora_fused = 1;
  gp.lora_packed = 1;
  gp.lora_rs = rs;
  gp.lora_b_e1 = b_e1 ? 1 : 0;
  gp.slots = make_slots(a);
  gp.P = P;
  gp.pair_slot = pair_slot;
  return true;
}

// The LoRA shrink as the first tiles of a fused-LoRA GEMM with a packed B (see GemmParams):
// per active slot a tensor map of its rank rows of A [S*Ea*R rows, K], the stacked ub and
// pair_slot outputs, and the ready flags.  Needs the active ranks to be multiples of 8 (each
// slot's rows then start on a swizzle-atom boundary) and at most 128 of them (one MMA M);
// returns false when they are not, and the separate shrink kernel runs instead.
bool shrink_in_gemm_maps(moe_lora_handle* h, GemmParams& gp, const moe_lora_args* a, const moe_lora_bf16* A, int K,
                         bool a_e1, __nv_bfloat16* ub, int32_t* pair_slot, int* ready,
                         const moe_lora_bf16* Ap = nullptr) {
  if (a->S > kMaxFusedSlots) return false;
  const int Ea = a_e1 ? 1 : a->E;
  if (Ap != nullptr) {   // the shrink-ready A: every slot's rows of an expert in one block
    int aoff[kMaxFusedSlots + 1];
    const int RS = stacked_rows(a->h_ranks, a->S, aoff);
    if (RS == 0 || RS > 128) return false;
    if (!make_tmap(h->encode, &gp.tmap_sa[0], Ap, static_cast<uint64_t>(Ea) * RS, K, static_cast<uint32_t>(RS)))
      return false;
    for (int s = 0; s <= kMaxFusedSlots; ++s) gp.sa_row_off[s] = aoff[s <= a->S ? s : a->S];
    gp.sa_packed = 1;
    gp.sa_R = RS;
  } else {
    const uint64_t a_rows = static_cast<uint64_t>(a->S) * Ea * a->R;
    int off = 0;
    for (int s = 0; s < kMaxFusedSlots; ++s) {
      gp.sa_row_off[s] = off;
      const int rows = (s < a->S && a->h_ranks[s] > 0 && a->h_scalings[s] != 0.0f) ? a->h_ranks[s] : 0;
      if (rows % 8 != 0) return false;
      if (rows > 0 && !make_tmap(h->encode, &gp.tmap_sa[s], A, a_rows, K, static_cast<uint32_t>(rows))) return false;
      off += rows;
    }
    gp.sa_row_off[kMaxFusedSlots] = off;
    if (off == 0 || off > 128) return false;
    gp.sa_R = a->R;
  }
  int coff[kMaxFusedSlots + 1];
  const int rs = stacked_cols(a->h_ranks, a->S, coff);
  if (rs != gp.lora_rs || rs > 384) return false;
  for (int s = 0; s <= kMaxFusedSlots; ++s) gp.coff[s] = coff[s <= a->S ? s : a->S];
  gp.sa_e1 = a_e1 ? 1 : 0;
  gp.ub_out = ub;
  gp.pair_slot = pair_slot;   // the token slots the permute gathers
  gp.perm = nullptr;   // set by the caller
  gp.shrink_ready = ready;
  gp.shrink_in_gemm = 1;
  return true;
}

// Tensor-core shrink of every slot: X [P, K] (permuted hidden or activation) against the
// stacked LoRA A [S*E*R, K]; writes ub and pair_slot.
moe_lora_status enqueue_shrink_tc(moe_lora_handle* h, const moe_lora_args* a, const void* X, const moe_lora_bf16* A,
                                  int K, const int32_t* offsets, const int32_t* perm, const LoraSlots& slots,
                                  __nv_bfloat16* ub, int32_t* pair_slot, uint32_t* status, cudaStream_t stream,
                                  bool pdl, bool a_e1 = false, bool stacked = false,
                                  const moe_lora_bf16* Ap = nullptr) {
  const int P = a->T * a->top_k;
  ShrinkTcParams sp;
  std::memset(&sp, 0, sizeof(sp));
  if (stacked) {   // ub rows in the packed-B column layout
    if (a->S > kMaxFusedSlots) return MOE_LORA_ERR_UNSUPPORTED;
    sp.ub_stacked = 1;
    sp.rs = stacked_cols(a->h_ranks, a->S, sp.coff);
  }
  // pairs per tile from the mean pairs per expert, so small experts read only their rows
  const long long m2 = 2LL * ((P + a->E - 1) / a->E);
  sp.tb = m2 <= 16 ? 16 : m2 <= 32 ? 32 : m2 <= 64 ? 64 : 128;
  if (!make_tmap(h->encode, &sp.tmap_x, X, static_cast<uint64_t>(P), K, sp.tb)) return MOE_LORA_ERR_CUDA;
  const uint64_t a_rows = static_cast<uint64_t>(a->S) * (a_e1 ? 1 : a->E) * a->R;
  sp.a_e1 = a_e1 ? 1 : 0;
  if (!make_tmap(h->encode, &sp.tmap_a, A, a_rows, K, a->R)) return MOE_LORA_ERR_CUDA;
  // the shrink-ready A: every slot's rank rows of an expert in one block of RS rows
  int aoff[kMaxFusedSlots + 1];
  const int RS = (Ap != nullptr && a->S <= kMaxFusedSlots) ? stacked_rows(a->h_ranks, a->S, aoff) : 0;
  if (RS > 0 && RS <= 256) {
    if (!make_tmap(h->encode, &sp.tmap_a, Ap, static_cast<uint64_t>(a_e1 ? 1 : a->E) * RS, K,
                   static_cast<uint32_t>(RS)))
      return MOE_LORA_ERR_CUDA;
    sp.packed_a = 1;
    sp.per_slot = 1;
    for (int s = 0; s <= a->S; ++s) sp.row_off[s] = aoff[s];
  }
  // only the active slots' rank rows, when every such rank is a multiple of 8 (each slot's
  // rows then start on a swizzle-atom boundary of the stacked tile)
  if (!sp.packed_a) sp.per_slot = a->S <= kMaxFusedSlots ? 1 : 0;
  sp.row_off[0] = 0;
  for (int s = 0; s < a->S && sp.per_slot && !sp.packed_a; ++s) {
    const int rows = (slots.ranks[s] > 0 && slots.scal[s] != 0.0f) ? slots.ranks[s] : 0;
    if (rows % 8 != 0) sp.per_slot = 0;
    sp.row_off[s + 1] = sp.row_off[s] + rows;
    if (rows > 0 && !make_tmap(h->encode, &sp.tmap_a_slot[s], A, a_rows, K,
                               static_cast<uint32_t>(rows)))
      return MOE_LORA_ERR_CUDA;
  }
  sp.offsets = offsets;
  sp.perm = perm;
  sp.slot_idx = a->slot_idx;
  sp.k = a->top_k;
  sp.P = P;
  sp.K = K;
  sp.E = a->E;
  sp.S = a->S;
  sp.R = a->R;
  sp.slots = slots;
  sp.ub = ub;
  sp.pair_slot = pair_slot;
  sp.status = status;
  int grid = (P + sp.tb - 1) / sp.tb + a->E;
  if (grid > h->num_sms) grid = h->num_sms;
  ML_LAUNCH(h, launch_lora_shrink_tc(sp, grid, stream, pdl), "lora shrink (tensor cores) launch");
  return MOE_LORA_OK;
}

void prof(const moe_lora_args* a, int stage, int which, cudaStream_t s) {
  if (a->prof_events == nullptr) return;
  void* ev = a->prof_events[2 * stage + which];
  if (ev != nullptr) cudaEventRecord(static_cast<cudaEvent_t>(ev), s);
}


}  // namespace

namespace {

// The LoRA placement the pages draw (sglang PR #28466 section 1 flow (B)): the gate_up LoRA
// chain -- shrink and expand into the bf16 delta d -- on the side stream beside the permute
// and gate_up GEMM, joined before the activation kernel; the down shrink after it; the down
// expand in the down GEMM (extra K-stages) or its epilogue.  Used when the fully fused path
// is not (16-token tiles, ranks not a multiple of 8, more than 8 slots, or
// MOE_LORA_FLAG_UNFUSED_LORA), and without LoRA at 16-token tiles.
moe_lora_status enqueue_unfused_lora_path(moe_lora_handle* h, const moe_lora_args* a, bool lora, uint8_t* ws,
                                          const Layout& L,
                                          int32_t* perm, int32_t* offsets, int32_t* ids, __nv_bfloat16* xp,
                                          __nv_bfloat16* g, __nv_bfloat16* d, __nv_bfloat16* act, float* v, float* y,
                                          int32_t* pair_slot, __nv_bfloat16* ub, const LoraSlots& slots,
                                          uint32_t* status, cudaStream_t stream,
                                          const moe_lora_fp8_weights* f8 = nullptr,
                                          const __nv_bfloat16** dn_delta = nullptr,
                                          const moe_lora_nvfp4_weights* f4 = nullptr) {
  (void)ids;
  const int T = a->T, H = a->H, I = a->I, E = a->E, k = a->top_k;
  const int P = T * k;
  const int R = lora ? a->R : 0;
  const bool so = (a->flags & MOE_LORA_FLAG_SHARED_OUTER) != 0;   // one A_gu, one B_dn per slot
  const int RU = (R + 7) & ~7;
  const bool pdl = !(a->flags & MOE_LORA_FLAG_NO_PDL);
  moe_lora_status st = MOE_LORA_OK;
  // The down-LoRA expand runs inside the down GEMM as extra K-stages when the rank stride is
  // TMA-able and the slots are few.  The gate_up expand stays a separate kernel writing the
  // bf16 delta: the pages round the gate_up GEMM output and the delta to bf16 separately,
  // and adding the delta inside the accumulator would round their sum once instead.
  // At 16-token tiles (decode) the epilogue expand costs less than an extra K-stage.
  // FP8 and NVFP4 weights: token tiles of at most 64 and the down expand in the GEMM's epilogue
  const bool q8 = f8 != nullptr || f4 != nullptr;
  const int bn = q8 ? std::min(pick_bn(P, E), 64) : pick_bn(P, E);
  const bool fused = !q8 && lora && (R % 8 == 0) && a->S <= kMaxFusedSlots && bn >= 32 &&
                     !(a->flags & MOE_LORA_FLAG_UNFUSED_LORA);
  // FP8 GEMM inputs: the permuted hidden codes in the xp region, the activation codes in
  // the g region (written after the activation has read g), and their group scales
  uint8_t* xp8 = reinterpret_cast<uint8_t*>(xp);
  uint8_t* a8 = reinterpret_cast<uint8_t*>(g);
  float* sx = reinterpret_cast<float*>(ws + L.sx);
  float* sa = reinterpret_cast<float*>(ws + L.sa);
  // NVFP4 GEMM inputs: the exact f16 values of the quantised permuted hidden rows in the xp
  // region, of the quantised activation in the g region; their row scales in sx and sa
  __half* xq4 = reinterpret_cast<__half*>(xp);
  __half* aq4 = reinterpret_cast<__half*>(g);
  const bool fused_gu = false;
  // 32-pair LoRA tiles when experts carry many pairs and the staged rows fit in smem
  const int lora_ntl = (P >= 32 * E && lora_smem_bytes(4, R, 2 * I, true, E) <= 200 * 1024) ? 4 : 1;
  int lora_grid = (P + 8 * lora_ntl - 1) / (8 * lora_ntl) + E;
  if (lora_grid > 2 * h->num_sms) lora_grid = 2 * h->num_sms;
  const bool two = lora && (((T <= 256) && !(a->flags & MOE_LORA_FLAG_FORCE_SINGLE_STREAM)) ||
                            (a->flags & MOE_LORA_FLAG_FORCE_TWO_STREAM));
  cudaStream_t ls = two ? h->side : stream;
  // Once the side stream has been forked, every return before the join below still joins
  // it back (recording the ready event on the side stream first if that has not happened),
  // so a failed enqueue never leaves a capture on `stream` with an unjoined fork.
  struct ForkJoin {
    moe_lora_handle* h;
    cudaStream_t main;
    bool forked = false, ready = false, joined = false;
    ~ForkJoin() {
      if (!forked || joined) return;
      if (!ready) cudaEventRecord(h->ev_ready, h->side);
      cudaStreamWaitEvent(main, h->ev_ready, 0);
    }
  } fj{h, stream};
  if (lora) {   // gate_up LoRA: shrink + expand into the bf16 delta d
    if (two) {
      ML_CUDA(cudaEventRecord(h->ev_fork, stream), "cudaEventRecord");
      ML_CUDA(cudaStreamWaitEvent(h->side, h->ev_fork, 0), "cudaStreamWaitEvent");
      fj.forked = true;
    }
    prof(a, MOE_LORA_STAGE_LORA_GATE_UP, 0, ls);
    LoraParams lp;
    std::memset(&lp, 0, sizeof(lp));
    lp.src = reinterpret_cast<const __nv_bfloat16*>(a->hidden);
    lp.by_token = 1;
    lp.perm = perm;
    lp.slot_idx = a->slot_idx;
    lp.offsets = offsets;
    lp.k = k;
    lp.P = P;
    lp.K = H;
    lp.E = E;
    lp.A = reinterpret_cast<const __nv_bfloat16*>(a->lora_A_gu);
    lp.a_e1 = so ? 1 : 0;   // shared-outer: one A_gu per slot
    lp.slots = slots;
    lp.status = status;
    lp.where = kWhereLoraShrinkGu;
    if (fused_gu) {
      lp.N = 0;
      lp.ub_out = ub;
      lp.RU = RU;
      lp.pair_slot_out = pair_slot;
    } else {
      lp.N = 2 * I;
      lp.B = reinterpret_cast<const __nv_bfloat16*>(a->lora_B_gu);
      lp.d_out = d;
    }
    ML_LAUNCH(h, launch_lora(lp, lora_ntl, lora_grid, ls, pdl && !two), "lora gate_up launch");
    prof(a, MOE_LORA_STAGE_LORA_GATE_UP, 1, ls);
    if (two) {
      ML_CUDA(cudaEventRecord(h->ev_ready, h->side), "cudaEventRecord");
      fj.ready = true;
    }
  }

  prof(a, MOE_LORA_STAGE_PERMUTE, 0, stream);
  // The down LoRA beside the down GEMM (flag): shrink and expand in one kernel on the side
  // stream, into a bf16 delta per pair that the finalize adds; the activation runs alone.
  const bool dn_side = lora && two && !fused && !q8 && (a->flags & MOE_LORA_FLAG_DOWN_LORA_SIDE);
  // the pairs' adapter slots ride along with the permute for the activation + down shrink
  const bool act_shrink = lora && !fused && !fused_gu && !dn_side;
  if (f8 != nullptr) {   // permute and quantise in one pass
    ML_LAUNCH(h, launch_quant_fp8(reinterpret_cast<const __nv_bfloat16*>(a->hidden), perm, k, P, H, xp8, sx, stream,
                                  pdl, a->slot_idx, act_shrink ? pair_slot : nullptr),
              "permute + quant launch");
  } else if (f4 != nullptr) {   // permute and NVFP4-quantise in one pass
    ML_LAUNCH(h, launch_quant_nvfp4(reinterpret_cast<const __nv_bfloat16*>(a->hidden), perm, k, P, H, sx, xq4, nullptr,
                                    nullptr, stream, pdl, a->slot_idx, act_shrink ? pair_slot : nullptr),
              "permute + NVFP4 quant launch");
  } else {
    ML_LAUNCH(h, launch_permute(reinterpret_cast<const __nv_bfloat16*>(a->hidden), perm, P, k, H, xp, stream, pdl,
                                a->slot_idx, act_shrink ? pair_slot : nullptr),
              "permute launch");
  }
  prof(a, MOE_LORA_STAGE_PERMUTE, 1, stream);

  if (fused_gu && two) {
    fj.joined = true;
    ML_CUDA(cudaStreamWaitEvent(stream, h->ev_ready, 0), "cudaStreamWaitEvent");
  }
  prof(a, MOE_LORA_STAGE_GATE_UP_GEMM, 0, stream);
  GemmParams gu;
  std::memset(&gu, 0, sizeof(gu));
  gu.out = g;
  gu.offsets = offsets;
  gu.status = status;
  gu.E = E;
  gu.N = 2 * I;
  gu.K = H;
  gu.gated = 1;
  if (fused_gu && !fuse_lora_maps(h, gu, a, a->lora_B_gu, 2 * I, ub, pair_slot, P, bn)) return MOE_LORA_ERR_CUDA;
  if (f8 != nullptr) {
    GemmF8Params gq;
    std::memset(&gq, 0, sizeof(gq));
    gq.w_scale = f8->w1_scale;
    gq.x_scale = sx;
    gq.out = g;
    gq.offsets = offsets;
    gq.status = status;
    gq.E = E;
    gq.N = 2 * I;
    gq.K = H;
    gq.gated = 1;
    st = enqueue_gemm_fp8(h, gq, f8->w1, xp8, P, bn, stream, pdl);
  } else if (f4 != nullptr) {
    GemmNv4Params gq;
    std::memset(&gq, 0, sizeof(gq));
    gq.w_sf = f4->w1_sf;
    gq.w_gs = f4->w1_gs;
    gq.x_gs = sx;
    gq.out = g;
    gq.offsets = offsets;
    gq.status = status;
    gq.E = E;
    gq.N = 2 * I;
    gq.K = H;
    gq.gated = 1;
    st = enqueue_gemm_nvfp4(h, gq, f4->w1, xq4, P, bn, stream, pdl);
  } else {
    st = enqueue_gemm(h, gu, a->w1, xp, P, bn, stream, pdl && !(fused_gu && two));
  }
  if (st != MOE_LORA_OK) return st;
  prof(a, MOE_LORA_STAGE_GATE_UP_GEMM, 1, stream);

  if (!fused_gu && two) {
    fj.joined = true;
    ML_CUDA(cudaStreamWaitEvent(stream, h->ev_ready, 0), "cudaStreamWaitEvent");
  }
  // (no programmatic launch right behind a wait on the side stream)
  const bool pdl_act = pdl && !two;
  if (act_shrink) {
    // activation and down-LoRA shrink in one pass; the expand runs in the down GEMM's epilogue
    prof(a, MOE_LORA_STAGE_ACTIVATION, 0, stream);
    ActShrinkParams ap;
    std::memset(&ap, 0, sizeof(ap));
    ap.g = g;
    ap.d = d;
    ap.offsets = offsets;
    ap.A = reinterpret_cast<const __nv_bfloat16*>(a->lora_A_dn);
    ap.slots = slots;
    ap.P = P;
    ap.I = I;
    ap.E = E;
    ap.a = act;
    ap.v = v;
    ap.pair_slot = pair_slot;
    ap.status = status;
    int grid = (P + 7) / 8 + E;
    if (grid > 4 * h->num_sms) grid = 4 * h->num_sms;
    ML_LAUNCH(h, launch_act_shrink(ap, grid, stream, pdl_act), "activation + down shrink launch");
    prof(a, MOE_LORA_STAGE_ACTIVATION, 1, stream);
  } else {
    prof(a, MOE_LORA_STAGE_ACTIVATION, 0, stream);
    ML_LAUNCH(h, launch_activation(g, (lora && !fused_gu) ? d : nullptr, P, I, act, stream, pdl_act),
            "activation launch");
    prof(a, MOE_LORA_STAGE_ACTIVATION, 1, stream);
  }

  // second fork: the side stream takes the down LoRA once the activation is written
  ForkJoin fj2{h, stream};
  if (dn_side) {
    __nv_bfloat16* dd = xp;   // the permuted hidden rows are dead after the gate_up GEMM: [P, H]
    ML_CUDA(cudaEventRecord(h->ev_fork, stream), "cudaEventRecord");
    ML_CUDA(cudaStreamWaitEvent(h->side, h->ev_fork, 0), "cudaStreamWaitEvent");
    fj2.forked = true;
    prof(a, MOE_LORA_STAGE_LORA_DOWN, 0, h->side);
    LoraParams lp;
    std::memset(&lp, 0, sizeof(lp));
    lp.src = act;
    lp.by_token = 0;
    lp.perm = perm;
    lp.slot_idx = a->slot_idx;
    lp.offsets = offsets;
    lp.k = k;
    lp.P = P;
    lp.K = I;
    lp.E = E;
    lp.N = H;
    lp.A = reinterpret_cast<const __nv_bfloat16*>(a->lora_A_dn);
    lp.B = reinterpret_cast<const __nv_bfloat16*>(a->lora_B_dn);
    lp.b_e1 = so ? 1 : 0;   // shared-outer: one B_dn per slot
    lp.slots = slots;
    lp.d_out = dd;
    lp.status = status;
    lp.where = kWhereLoraShrinkDn;
    const int ntl_dn = (P >= 32 * E && lora_smem_bytes(4, R, H, true, E) <= 200 * 1024) ? 4 : 1;
    ML_LAUNCH(h, launch_lora(lp, ntl_dn, lora_grid, h->side, false), "lora down (side stream) launch");
    prof(a, MOE_LORA_STAGE_LORA_DOWN, 1, h->side);
    ML_CUDA(cudaEventRecord(h->ev_ready, h->side), "cudaEventRecord");
    fj2.ready = true;
    if (dn_delta != nullptr) *dn_delta = dd;
  }

  if (lora && fused) {   // down-LoRA shrink on the activation; its expand runs inside the down GEMM
    prof(a, MOE_LORA_STAGE_LORA_DOWN, 0, stream);
    LoraParams lp;
    std::memset(&lp, 0, sizeof(lp));
    lp.src = act;
    lp.by_token = 0;
    lp.perm = perm;
    lp.slot_idx = a->slot_idx;
    lp.offsets = offsets;
    lp.k = k;
    lp.P = P;
    lp.K = I;
    lp.E = E;
    lp.N = 0;
    lp.A = reinterpret_cast<const __nv_bfloat16*>(a->lora_A_dn);
    lp.slots = slots;
    lp.ub_out = ub;
    lp.RU = RU;
    lp.pair_slot_out = pair_slot;
    lp.status = status;
    lp.where = kWhereLoraShrinkDn;
    ML_LAUNCH(h, launch_lora(lp, lora_ntl, lora_grid, stream, pdl), "lora down shrink launch");
    prof(a, MOE_LORA_STAGE_LORA_DOWN, 1, stream);
  }

  prof(a, MOE_LORA_STAGE_DOWN_GEMM, 0, stream);
  GemmParams dn;
  std::memset(&dn, 0, sizeof(dn));
  dn.out_f32 = y;
  dn.offsets = offsets;
  dn.status = status;
  dn.E = E;
  dn.N = H;
  dn.K = I;
  dn.gated = 0;
  if (fused) {
    if (!fuse_lora_maps(h, dn, a, a->lora_B_dn, H, ub, pair_slot, P, bn, so)) return MOE_LORA_ERR_CUDA;
  } else if (lora && !dn_side) {
    dn.lora_v = v;
    dn.lora_B = reinterpret_cast<const __nv_bfloat16*>(a->lora_B_dn);
    dn.lora_b_e1 = so ? 1 : 0;   // shared-outer: one B_dn per slot
    dn.pair_slot = pair_slot;
    dn.slots = slots;
  }
  // the epilogue's staged LoRA rows grow with the tile: narrow it until two stages fit
  int bn_dn = bn;
  while (!fused && lora && !dn_side && bn_dn > 16 &&
         (f8 != nullptr   ? gemm_fp8_smem_bytes(bn_dn, 2, E, R)
          : f4 != nullptr ? gemm_nvfp4_smem_bytes(bn_dn, 5, 2, E, R)
                          : gemm_smem_bytes(bn_dn, 1, 2, E, R, 0, 1)) > kMaxGemmSmem)
    bn_dn >>= 1;
  if (f8 != nullptr) {   // the activation's group quantisation, then the FP8 down GEMM
    ML_LAUNCH(h, launch_quant_fp8(act, nullptr, 1, P, I, a8, sa, stream, pdl), "activation quant launch");
    GemmF8Params dq;
    std::memset(&dq, 0, sizeof(dq));
    dq.w_scale = f8->w2_scale;
    dq.x_scale = sa;
    dq.out_f32 = y;
    dq.offsets = offsets;
    dq.status = status;
    dq.E = E;
    dq.N = H;
    dq.K = I;
    dq.gated = 0;
    if (lora) {
      dq.lora_v = v;
      dq.lora_B = reinterpret_cast<const __nv_bfloat16*>(a->lora_B_dn);
      dq.lora_b_e1 = so ? 1 : 0;
      dq.pair_slot = pair_slot;
      dq.slots = slots;
    }
    st = enqueue_gemm_fp8(h, dq, f8->w2, a8, P, bn_dn, stream, pdl);
    if (st != MOE_LORA_OK) return st;
    prof(a, MOE_LORA_STAGE_DOWN_GEMM, 1, stream);
    return MOE_LORA_OK;
  }
  if (f4 != nullptr) {   // the activation's NVFP4 quantisation, then the NVFP4 down GEMM
    ML_LAUNCH(h, launch_quant_nvfp4(act, nullptr, 1, P, I, sa, aq4, nullptr, nullptr, stream, pdl),
              "activation NVFP4 quant launch");
    GemmNv4Params dq;
    std::memset(&dq, 0, sizeof(dq));
    dq.w_sf = f4->w2_sf;
    dq.w_gs = f4->w2_gs;
    dq.x_gs = sa;
    dq.out_f32 = y;
    dq.offsets = offsets;
    dq.status = status;
    dq.E = E;
    dq.N = H;
    dq.K = I;
    dq.gated = 0;
    if (lora) {
      dq.lora_v = v;
      dq.lora_B = reinterpret_cast<const __nv_bfloat16*>(a->lora_B_dn);
      dq.lora_b_e1 = so ? 1 : 0;
      dq.pair_slot = pair_slot;
      dq.slots = slots;
    }
    st = enqueue_gemm_nvfp4(h, dq, f4->w2, aq4, P, bn_dn, stream, pdl);
    if (st != MOE_LORA_OK) return st;
    prof(a, MOE_LORA_STAGE_DOWN_GEMM, 1, stream);
    return MOE_LORA_OK;
  }
  st = enqueue_gemm(h, dn, a->w2, act, P, bn_dn, stream, pdl);
  if (st != MOE_LORA_OK) return st;
  prof(a, MOE_LORA_STAGE_DOWN_GEMM, 1, stream);
  if (dn_side) {   // join: the finalize adds the side stream's delta
    fj2.joined = true;
    ML_CUDA(cudaStreamWaitEvent(stream, h->ev_ready, 0), "cudaStreamWaitEvent");
  }

  return MOE_LORA_OK;
}

// FP8 block-scale weights with the fused LoRA placement (needs the expand-ready B copies):
// permute + quantise the hidden rows for the FP8 gate_up GEMM and permute them in bf16 for
// the LoRA shrink; the tensor-core shrink writes the stacked ub rows; the FP8 gate_up GEMM
// runs the gate_up expand as bf16 K-stages into its own accumulator and writes g and the
// bf16 delta d separately; the activation adds them (as on the side-stream placement); the
// down shrink reads the bf16 activation, which is then quantised for the FP8 down GEMM, whose
// LoRA K-stages add the down delta to its fp32 sum.
moe_lora_status enqueue_fp8_fused_lora(moe_lora_handle* h, const moe_lora_args* a, uint8_t* ws, const Layout& L,
                                       int32_t* perm, int32_t* offsets, __nv_bfloat16* xp, __nv_bfloat16* g,
                                       __nv_bfloat16* d, __nv_bfloat16* act, float* y, int32_t* pair_slot,
                                       __nv_bfloat16* ub, const LoraSlots& slots, uint32_t* status,
                                       cudaStream_t stream, const moe_lora_fp8_weights* f8) {
  const int T = a->T, H = a->H, I = a->I, E = a->E, k = a->top_k;
  const int P = T * k;
  const bool so = (a->flags & MOE_LORA_FLAG_SHARED_OUTER) != 0;
  const bool pdl = !(a->flags & MOE_LORA_FLAG_NO_PDL);
  const int bn = std::min(pick_bn(P, E), 64);
  uint8_t* xp8 = reinterpret_cast<uint8_t*>(xp);   // e4m3 permuted hidden rows [P, H] bytes
  uint8_t* a8 = reinterpret_cast<uint8_t*>(g);     // e4m3 activation [P, I] (after g is read)
  float* sx = reinterpret_cast<float*>(ws + L.sx);
  float* sa = reinterpret_cast<float*>(ws + L.sa);
  __nv_bfloat16* xp16 = reinterpret_cast<__nv_bfloat16*>(y);   // bf16 permuted rows: y is free until the down GEMM
  moe_lora_status st = MOE_LORA_OK;

  prof(a, MOE_LORA_STAGE_PERMUTE, 0, stream);
  ML_LAUNCH(h, launch_quant_fp8(reinterpret_cast<const __nv_bfloat16*>(a->hidden), perm, k, P, H, xp8, sx, stream,
                                pdl),
            "permute + quant launch");
  ML_LAUNCH(h, launch_permute(reinterpret_cast<const __nv_bfloat16*>(a->hidden), perm, P, k, H, xp16, stream, pdl),
            "permute launch");
  prof(a, MOE_LORA_STAGE_PERMUTE, 1, stream);
  prof(a, MOE_LORA_STAGE_LORA_GATE_UP, 0, stream);
  st = enqueue_shrink_tc(h, a, xp16, a->lora_A_gu, H, offsets, perm, slots, ub, pair_slot, status, stream, pdl, so,
                         true, a->lora_A_gu_packed);
  if (st != MOE_LORA_OK) return st;
  prof(a, MOE_LORA_STAGE_LORA_GATE_UP, 1, stream);

  prof(a, MOE_LORA_STAGE_GATE_UP_GEMM, 0, stream);
  GemmF8Params gq;
  std::memset(&gq, 0, sizeof(gq));
  gq.w_scale = f8->w1_scale;
  gq.x_scale = sx;
  gq.out = g;
  gq.d_out = d;
  gq.offsets = offsets;
  gq.status = status;
  gq.E = E;
  gq.N = 2 * I;
  gq.K = H;
  gq.gated = 1;
  gq.pair_slot = pair_slot;
  gq.slots = slots;
  gq.lora_packed = 1;
  if (!packed_lora_tmaps(h, a, a->lora_B_gu_packed, 2 * I, true, false, ub, P, bn, &gq.tmap_lbp, &gq.tmap_lup,
                         &gq.lora_rs, gq.lora_panel_slots))
    return MOE_LORA_ERR_CUDA;
  st = enqueue_gemm_fp8(h, gq, f8->w1, xp8, P, bn, stream, pdl);
  if (st != MOE_LORA_OK) return st;
  prof(a, MOE_LORA_STAGE_GATE_UP_GEMM, 1, stream);

  prof(a, MOE_LORA_STAGE_ACTIVATION, 0, stream);
  ML_LAUNCH(h, launch_activation(g, d, P, I, act, stream, pdl), "activation launch");
  prof(a, MOE_LORA_STAGE_ACTIVATION, 1, stream);
  prof(a, MOE_LORA_STAGE_LORA_DOWN, 0, stream);
  st = enqueue_shrink_tc(h, a, act, a->lora_A_dn, I, offsets, perm, slots, ub, pair_slot, status, stream, pdl, false,
                         true, a->lora_A_dn_packed);
  if (st != MOE_LORA_OK) return st;
  prof(a, MOE_LORA_STAGE_LORA_DOWN, 1, stream);

  prof(a, MOE_LORA_STAGE_DOWN_GEMM, 0, stream);
  ML_LAUNCH(h, launch_quant_fp8(act, nullptr, 1, P, I, a8, sa, stream, pdl), "activation quant launch");
  GemmF8Params dq;
  std::memset(&dq, 0, sizeof(dq));
  dq.w_scale = f8->w2_scale;
  dq.x_scale = sa;
  dq.out_f32 = y;
  dq.offsets = offsets;
  dq.status = status;
  dq.E = E;
  dq.N = H;
  dq.K = I;
  dq.gated = 0;
  dq.pair_slot = pair_slot;
  dq.slots = slots;
  dq.lora_packed = 1;
  dq.lora_b_e1 = so ? 1 : 0;
  if (!packed_lora_tmaps(h, a, a->lora_B_dn_packed, H, false, so, ub, P, bn, &dq.tmap_lbp, &dq.tmap_lup, &dq.lora_rs,
                         dq.lora_panel_slots))
    return MOE_LORA_ERR_CUDA;
  st = enqueue_gemm_fp8(h, dq, f8->w2, a8, P, bn, stream, pdl);
  if (st != MOE_LORA_OK) return st;
  prof(a, MOE_LORA_STAGE_DOWN_GEMM, 1, stream);
  return MOE_LORA_OK;
}

}  // namespace

extern "C" {

moe_lora_status moe_lora_route(moe_lora_handle* h, const moe_lora_bf16* router_logits, const float* correction_bias,
                               int T, int E, int top_k, int routing_method, float routed_scaling_factor, int n_group,
                               int topk_group, int32_t* topk_ids, float* topk_weights, int32_t* expert_offsets,
                               int32_t* perm, int32_t* inv_perm, void* workspace, size_t workspace_bytes,
                               moe_lora_stream stream) {
  if (h == nullptr || workspace == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  moe_lora_status st = check_routing_args(T, E, top_k, routing_method, router_logits, correction_bias, n_group,
                                          topk_group);
  if (st != MOE_LORA_OK) return st;
  if (expert_offsets == nullptr || (T > 0 && (!topk_ids || !topk_weights || !perm || !inv_perm)))
    return MOE_LORA_ERR_INVALID_ARG;
  const Layout L = layout_for(T, 0, 0, E, top_k, 0, 0);
  if (workspace_bytes < L.bytes) return MOE_LORA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  ML_CUDA(cudaMemsetAsync(ws, 0, 256, stream), "cudaMemsetAsync");
  if (T == 0) {
    ML_CUDA(cudaMemsetAsync(expert_offsets, 0, (static_cast<size_t>(E) + 1) * 4, stream), "cudaMemsetAsync");
    return MOE_LORA_OK;
  }
  return enqueue_route(h, router_logits, correction_bias, T, E, top_k, routing_method, routed_scaling_factor,
                       topk_ids, topk_weights, expert_offsets, perm, inv_perm, ws, L, stream);
}

// Size and checks of the expand-ready LoRA B copy (see include/moe_lora.h).
static moe_lora_status packed_lora_b_dims(int S, int E_b, int N, int R, int gated, const int32_t* h_ranks,
                                          int* NT, int* rs, int* coff) {
  if (S < 1 || S > kMaxSlots || E_b < 1 || E_b > kMaxExperts || N < 1 || R < 1 || R > kMaxRank || h_ranks == nullptr)
    return MOE_LORA_ERR_INVALID_ARG;
  if (gated != 0 && gated != 1) return MOE_LORA_ERR_INVALID_ARG;
  if (gated && N % 128 != 0) return MOE_LORA_ERR_INVALID_ARG;
  for (int s = 0; s < S; ++s)
    if (h_ranks[s] < 0 || h_ranks[s] > R) return MOE_LORA_ERR_INVALID_ARG;
  *NT = gated ? N / 128 : (N + 127) / 128;
  *rs = stacked_cols(h_ranks, S, coff);
  if (*rs == 0) return MOE_LORA_ERR_INVALID_ARG;
  if (static_cast<long long>(E_b) * *NT * 128 > 0x7fffffffLL) return MOE_LORA_ERR_INVALID_ARG;
  return MOE_LORA_OK;
}

moe_lora_status moe_lora_packed_lora_b_size(int S, int E_b, int N, int R, int gated, const int32_t* h_ranks,
                                            size_t* bytes) {
  if (bytes == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  int NT = 0, rs = 0, coff[kMaxSlots + 1];
  const moe_lora_status st = packed_lora_b_dims(S, E_b, N, R, gated, h_ranks, &NT, &rs, coff);
  if (st != MOE_LORA_OK) return st;
  *bytes = static_cast<size_t>(E_b) * NT * 128 * rs * 2;
  return MOE_LORA_OK;
}

moe_lora_status moe_lora_pack_lora_b(moe_lora_handle* h, const moe_lora_bf16* B, int S, int E_b, int N, int R,
                                     int gated, const int32_t* h_ranks, moe_lora_bf16* packed,
                                     moe_lora_stream stream) {
  if (h == nullptr || B == nullptr || packed == nullptr || !aligned16(packed)) return MOE_LORA_ERR_INVALID_ARG;
  PackLoraBParams pp;
  std::memset(&pp, 0, sizeof(pp));
  moe_lora_status st = packed_lora_b_dims(S, E_b, N, R, gated, h_ranks, &pp.NT, &pp.rs, pp.coff);
  if (st != MOE_LORA_OK) return st;
  pp.B = reinterpret_cast<const __nv_bfloat16*>(B);
  pp.Bp = reinterpret_cast<__nv_bfloat16*>(packed);
  pp.S = S;
  pp.Eb = E_b;
  pp.N = N;
  pp.R = R;
  pp.gated = gated;
  for (int s = 0; s < S; ++s) pp.ranks[s] = h_ranks[s];
  ML_LAUNCH(h, launch_pack_lora_b(pp, stream), "pack LoRA B launch");
  return MOE_LORA_OK;
}

static moe_lora_status packed_lora_a_dims(int S, int E_a, int K, int R, const int32_t* h_ranks, int* RS, int* aoff) {
  if (S < 1 || S > kMaxSlots || E_a < 1 || E_a > kMaxExperts || K < 8 || K % 8 != 0 || R < 1 || R > kMaxRank ||
      h_ranks == nullptr)
    return MOE_LORA_ERR_INVALID_ARG;
  for (int s = 0; s < S; ++s)
    if (h_ranks[s] < 0 || h_ranks[s] > R) return MOE_LORA_ERR_INVALID_ARG;
  *RS = stacked_rows(h_ranks, S, aoff);
  if (*RS == 0) return MOE_LORA_ERR_INVALID_ARG;
  if (static_cast<long long>(E_a) * *RS > 0x7fffffffLL) return MOE_LORA_ERR_INVALID_ARG;
  return MOE_LORA_OK;
}

moe_lora_status moe_lora_packed_lora_a_size(int S, int E_a, int K, int R, const int32_t* h_ranks, size_t* bytes) {
  if (bytes == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  int RS = 0, aoff[kMaxSlots + 1];
  const moe_lora_status st = packed_lora_a_dims(S, E_a, K, R, h_ranks, &RS, aoff);
  if (st != MOE_LORA_OK) return st;
  *bytes = static_cast<size_t>(E_a) * RS * K * 2;
  return MOE_LORA_OK;
}

moe_lora_status moe_lora_pack_lora_a(moe_lora_handle* h, const moe_lora_bf16* A, int S, int E_a, int K, int R,
                                     const int32_t* h_ranks, moe_lora_bf16* packed, moe_lora_stream stream) {
  if (h == nullptr || A == nullptr || packed == nullptr || !aligned16(A) || !aligned16(packed))
    return MOE_LORA_ERR_INVALID_ARG;
  PackLoraAParams pp;
  std::memset(&pp, 0, sizeof(pp));
  moe_lora_status st = packed_lora_a_dims(S, E_a, K, R, h_ranks, &pp.RS, pp.aoff);
  if (st != MOE_LORA_OK) return st;
  pp.A = reinterpret_cast<const __nv_bfloat16*>(A);
  pp.Ap = reinterpret_cast<__nv_bfloat16*>(packed);
  pp.S = S;
  pp.Ea = E_a;
  pp.R = R;
  pp.K = K;
  for (int s = 0; s < S; ++s) pp.ranks[s] = h_ranks[s];
  ML_LAUNCH(h, launch_pack_lora_a(pp, stream), "pack LoRA A launch");
  return MOE_LORA_OK;
}

moe_lora_status moe_lora_permute(moe_lora_handle* h, const moe_lora_bf16* hidden, const int32_t* perm, int T, int H,
                                 int top_k, moe_lora_bf16* permuted, moe_lora_stream stream) {
  if (h == nullptr || T < 0 || H < 8 || H % 8 != 0 || top_k < 1) return MOE_LORA_ERR_INVALID_ARG;
  if (T == 0) return MOE_LORA_OK;
  if (!hidden || !perm || !permuted || !aligned16(hidden) || !aligned16(permuted)) return MOE_LORA_ERR_INVALID_ARG;
  ML_LAUNCH(h, launch_permute(reinterpret_cast<const __nv_bfloat16*>(hidden), perm, T * top_k, top_k, H,
                         reinterpret_cast<__nv_bfloat16*>(permuted), stream),
          "permute launch");
  return MOE_LORA_OK;
}

}  // extern "C"

namespace {

// The forward of moe_lora_forward and moe_lora_forward_routed (`ext` set: the routing
// comes packed and the output may stay unfinalized).  Arguments are validated.
moe_lora_status forward_impl(moe_lora_handle* h, const moe_lora_args* a, const moe_lora_routed* ext,
                             moe_lora_bf16* out, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                             const moe_lora_fp8_weights* f8 = nullptr, const moe_lora_nvfp4_weights* f4 = nullptr) {
  moe_lora_status st = MOE_LORA_OK;
  const int T = a->T, H = a->H, I = a->I, E = a->E, k = a->top_k;
  const bool lora = lora_active(a);
  // programmatic launches: each kernel after the routing starts behind its predecessor
  const bool pdl = !(a->flags & MOE_LORA_FLAG_NO_PDL);
  const Layout L = layout_for(T, H, I, E, k, a->S > 0 ? a->R : 0, a->S > 0 ? a->S : 0);
  if (workspace_bytes < L.bytes) return MOE_LORA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // Up to 512 tokens the routing cluster writes the status word itself, so it is launched
  // behind the previous forward's last kernel with no header memset in between.
  const bool route_pdl = pdl && T > 0 && route_cluster_ctas(T) > 0;
  if (!route_pdl) ML_CUDA(cudaMemsetAsync(ws, 0, 256, stream), "cudaMemsetAsync");
  if (T == 0) return MOE_LORA_OK;

  const int P = T * k;
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.header);
  const bool ext_out = ext != nullptr;                       // outputs of the routed entry
  const bool finalize = ext == nullptr || ext->do_finalize != 0;
  auto pick = [](auto* user, bool use, auto* own) { return (use && user != nullptr) ? user : own; };
  int32_t* ids = pick(a->topk_ids, !ext_out, reinterpret_cast<int32_t*>(ws + L.ids));
  float* wts = ext_out ? pick(ext->expert_weights, true, reinterpret_cast<float*>(ws + L.wts))
                       : pick(a->topk_weights, true, reinterpret_cast<float*>(ws + L.wts));
  int32_t* offsets = pick(a->expert_offsets, !ext_out, reinterpret_cast<int32_t*>(ws + L.offsets));
  int32_t* perm = pick(a->perm, !ext_out, reinterpret_cast<int32_t*>(ws + L.perm));
  int32_t* inv = ext_out ? pick(ext->expanded_idx_to_permuted_idx, true, reinterpret_cast<int32_t*>(ws + L.inv))
                         : pick(a->inv_perm, true, reinterpret_cast<int32_t*>(ws + L.inv));
  __nv_bfloat16* xp = reinterpret_cast<__nv_bfloat16*>(ws + L.xp);
  __nv_bfloat16* g = reinterpret_cast<__nv_bfloat16*>(ws + L.g);
  __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(ws + L.d);
  __nv_bfloat16* act = reinterpret_cast<__nv_bfloat16*>(ws + L.a);
  if (!finalize && ext->activation_output != nullptr) act = reinterpret_cast<__nv_bfloat16*>(ext->activation_output);
  float* v = reinterpret_cast<float*>(ws + L.v);
  float* y = finalize ? reinterpret_cast<float*>(ws + L.y) : ext->gemm2_output;
  int32_t* pair_slot = reinterpret_cast<int32_t*>(ws + L.pslot);

  prof(a, MOE_LORA_STAGE_ROUTE, 0, stream);
  st = enqueue_route(h, a->router_logits, a->correction_bias, T, ext ? E + 1 : E, k, a->routing_method,
                     a->routed_scaling_factor, ids, wts, offsets, perm, inv, ws, L, stream, ext, route_pdl);
  if (st != MOE_LORA_OK) return st;
  prof(a, MOE_LORA_STAGE_ROUTE, 1, stream);

  LoraSlots slots;
  std::memset(&slots, 0, sizeof(slots));
  if (lora) slots = make_slots(a);
  const int R = lora ? a->R : 0;
  const bool so = (a->flags & MOE_LORA_FLAG_SHARED_OUTER) != 0;   // one A_gu, one B_dn per slot
  __nv_bfloat16* ub = reinterpret_cast<__nv_bfloat16*>(ws + L.ub);
  // Fully fused LoRA: both shrinks on the tensor cores, both expands inside the GEMMs, the
  // activation in the gate_up GEMM's epilogue.  Needs a TMA-able rank stride, few slots and
  // the stacked ranks within one MMA N.
  // At 16-token tiles (decode) the separate activation kernel and the side-stream LoRA chain
  // cost less than the fused epilogue and the serial shrinks, so the fused paths start at
  // 32-token tiles.
  const int bn0 = pick_bn(P, E);
  const bool fuse_all = lora && (R % 8 == 0) && a->S <= kMaxFusedSlots && a->S * R <= 256 && bn0 >= 32 &&
                        !(a->flags & MOE_LORA_FLAG_UNFUSED_LORA);
  const bool act_in_gemm = f8 == nullptr && f4 == nullptr && (fuse_all || (!lora && bn0 >= 32));
  const bool y_bf16 = act_in_gemm && finalize && bn0 >= kBf16YMinBn;
  const __nv_bfloat16* dn_delta = nullptr;   // the down-LoRA delta computed beside the down GEMM
  if (act_in_gemm) {
    const int bn = bn0;
    prof(a, MOE_LORA_STAGE_PERMUTE, 0, stream);
    // The gate_up LoRA shrink: fused into the permute while the active slots' stacked ranks
    // are few (the fused kernel's MMAs then fit two warps per 16-pair tile); many stacked
    // ranks (several adapters) keep the tensor-core shrink kernel after a plain permute.
    int nr_active = 0;
    for (int s = 0; s < a->S && lora; ++s)
      if (slots.ranks[s] > 0 && slots.scal[s] != 0.0f) nr_active += slots.ranks[s];
    const bool permute_shrink = fuse_all && nr_active <= kPermuteShrinkMaxRows;
    // the expand-ready B copies, where given, replace the per-slot LoRA stages (the gate_up one
    // needs the tensor-core shrink, which can write the stacked ub rows)
    const bool gu_packed = fuse_all && !permute_shrink && a->lora_B_gu_packed != nullptr;
    const bool dn_packed = fuse_all && a->lora_B_dn_packed != nullptr;
    // The GEMMs' parameters first: with a packed B on single-CTA tiles the LoRA shrink runs as
    // the first tiles of the GEMM itself (no shrink kernel), when its A rows fit one MMA.
    const bool shrink_ok = !(a->flags & MOE_LORA_FLAG_SEPARATE_SHRINK) && bn <= 128;
    int* ready = reinterpret_cast<int*>(ws + L.ready);
    const size_t nflags = ready_flags(static_cast<size_t>(P), E);
    GemmParams gu;
    std::memset(&gu, 0, sizeof(gu));
    gu.out = act;   // the activation, written by the GEMM's epilogue
    gu.offsets = offsets;
    gu.status = status;
    gu.E = E;
    gu.N = 2 * I;
    gu.K = H;
    gu.gated = 2;
    gu.cta_pair = pair_tiles(bn, 2 * I);
    if (fuse_all && !(gu_packed ? fuse_lora_maps_packed(h, gu, a, a->lora_B_gu_packed, 2 * I, ub, pair_slot, P, bn)
                                : fuse_lora_maps(h, gu, a, a->lora_B_gu, 2 * I, ub, pair_slot, P, bn)))
      return MOE_LORA_ERR_CUDA;
    const bool gu_in_gemm = gu_packed && shrink_ok && gu.cta_pair == 1 &&
                            shrink_in_gemm_maps(h, gu, a, a->lora_A_gu, H, so, ub, pair_slot, ready, a->lora_A_gu_packed);
    GemmParams dn;
    std::memset(&dn, 0, sizeof(dn));
    if (y_bf16) dn.out = reinterpret_cast<__nv_bfloat16*>(y);
    else dn.out_f32 = y;
    dn.offsets = offsets;
    dn.status = status;
    dn.E = E;
    dn.N = H;
    dn.K = I;
    dn.gated = 0;
    dn.cta_pair = pair_tiles(bn0, H);
    // the down GEMM adds its LoRA stages to the main accumulator, so it keeps the full tile
    if (fuse_all && !(dn_packed ? fuse_lora_maps_packed(h, dn, a, a->lora_B_dn_packed, H, ub, pair_slot, P, bn0, so)
                                : fuse_lora_maps(h, dn, a, a->lora_B_dn, H, ub, pair_slot, P, bn0, so)))
      return MOE_LORA_ERR_CUDA;
    const bool dn_in_gemm = dn_packed && shrink_ok && dn.cta_pair == 1 &&
                            shrink_in_gemm_maps(h, dn, a, a->lora_A_dn, I, false, ub, pair_slot, ready + nflags,
                                                a->lora_A_dn_packed);
    gu.perm = dn.perm = perm;
    gu.slot_idx = dn.slot_idx = a->slot_idx;
    gu.k = dn.k = k;
    if (permute_shrink) {   // the permute and the gate_up LoRA shrink in one pass over the token rows
      PermuteShrinkParams ps;
      std::memset(&ps, 0, sizeof(ps));
      ps.x = reinterpret_cast<const __nv_bfloat16*>(a->hidden);
      ps.perm = perm;
      ps.offsets = offsets;
      ps.slot_idx = a->slot_idx;
      ps.A = reinterpret_cast<const __nv_bfloat16*>(a->lora_A_gu);
      ps.a_e1 = so ? 1 : 0;
      ps.H = H;
      ps.E = E;
      ps.k = k;
      ps.P = P;
      ps.RU = (R + 7) & ~7;
      ps.nr_max = (nr_active + 7) & ~7;
      ps.slots = slots;
      ps.xp = xp;
      ps.ub = ub;
      ps.pair_slot = pair_slot;
      ps.status = status;
      if (gu_in_gemm || dn_in_gemm) {   // it also clears the ready flags of the GEMMs' shrink tiles
        ps.zero_out = ready;
        ps.zero_n = static_cast<int>(2 * nflags);
      }
      int grid = (P + 63) / 64 + E;   // tiles of 64 pairs (at most), two CTAs per SM
      if (grid > 2 * h->num_sms) grid = 2 * h->num_sms;
      ML_LAUNCH(h, launch_permute_shrink(ps, grid, stream, pdl), "permute + LoRA shrink launch");
      prof(a, MOE_LORA_STAGE_PERMUTE, 1, stream);
    } else {
      // the permute also clears the ready flags of the GEMMs' shrink tiles and gathers the
      // pairs' token slots for their slot masks
      const bool flags_used = gu_in_gemm || dn_in_gemm;
      ML_LAUNCH(h, launch_permute(reinterpret_cast<const __nv_bfloat16*>(a->hidden), perm, P, k, H, xp, stream, pdl,
                                  flags_used ? a->slot_idx : nullptr, flags_used ? pair_slot : nullptr,
                                  flags_used ? ready : nullptr, flags_used ? static_cast<int>(2 * nflags) : 0),
                "permute launch");
      prof(a, MOE_LORA_STAGE_PERMUTE, 1, stream);
      if (fuse_all) {
        prof(a, MOE_LORA_STAGE_LORA_GATE_UP, 0, stream);
        if (!gu_in_gemm) {
          st = enqueue_shrink_tc(h, a, xp, a->lora_A_gu, H, offsets, perm, slots, ub, pair_slot, status, stream, pdl,
                                 so, gu_packed, a->lora_A_gu_packed);
          if (st != MOE_LORA_OK) return st;
        }
        prof(a, MOE_LORA_STAGE_LORA_GATE_UP, 1, stream);
      }
    }
    prof(a, MOE_LORA_STAGE_GATE_UP_GEMM, 0, stream);
    st = enqueue_gemm(h, gu, a->w1, xp, P, bn, stream, pdl);
    if (st != MOE_LORA_OK) return st;
    prof(a, MOE_LORA_STAGE_GATE_UP_GEMM, 1, stream);
    if (fuse_all) {
      prof(a, MOE_LORA_STAGE_LORA_DOWN, 0, stream);
      if (!dn_in_gemm) {
        st = enqueue_shrink_tc(h, a, act, a->lora_A_dn, I, offsets, perm, slots, ub, pair_slot, status, stream, pdl,
                               false, dn_packed, a->lora_A_dn_packed);
        if (st != MOE_LORA_OK) return st;
      }
      prof(a, MOE_LORA_STAGE_LORA_DOWN, 1, stream);
    }
    prof(a, MOE_LORA_STAGE_DOWN_GEMM, 0, stream);
    st = enqueue_gemm(h, dn, a->w2, act, P, bn0, stream, pdl);
    if (st != MOE_LORA_OK) return st;
    prof(a, MOE_LORA_STAGE_DOWN_GEMM, 1, stream);
  } else if (f8 != nullptr && fuse_all && a->lora_B_gu_packed != nullptr && a->lora_B_dn_packed != nullptr) {
    st = enqueue_fp8_fused_lora(h, a, ws, L, perm, offsets, xp, g, d, act, y, pair_slot, ub, slots, status, stream,
                                f8);
    if (st != MOE_LORA_OK) return st;
  } else {
    st = enqueue_unfused_lora_path(h, a, lora, ws, L, perm, offsets, ids, xp, g, d, act, v, y, pair_slot, ub,
                                   slots, status, stream, f8, &dn_delta, f4);
    if (st != MOE_LORA_OK) return st;
  }

  if (!finalize) return MOE_LORA_OK;   // the routed entry's unfinalized outputs are written
  prof(a, MOE_LORA_STAGE_FINALIZE, 0, stream);
  FinalizeParams fp;
  std::memset(&fp, 0, sizeof(fp));
  if (y_bf16) fp.y_bf16 = reinterpret_cast<const __nv_bfloat16*>(y);
  else fp.y = y;
  fp.weights = wts;
  fp.inv = inv;
  fp.T = T;
  fp.H = H;
  fp.k = k;
  fp.out = reinterpret_cast<__nv_bfloat16*>(out);
  fp.dd = dn_delta;
  // (no programmatic launch right behind the join on the side stream)
  ML_LAUNCH(h, launch_finalize(fp, stream, pdl && dn_delta == nullptr), "finalize launch");
  prof(a, MOE_LORA_STAGE_FINALIZE, 1, stream);
  return MOE_LORA_OK;
}

}  // namespace

extern "C" {

moe_lora_status moe_lora_forward(moe_lora_handle* h, const moe_lora_args* a, moe_lora_bf16* out, void* workspace,
                                 size_t workspace_bytes, moe_lora_stream stream) {
  moe_lora_status st = moe_lora_validate(a);
  if (st != MOE_LORA_OK) return st;
  if (h == nullptr || workspace == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  if (a->T > 0 && (out == nullptr || !aligned16(out))) return MOE_LORA_ERR_INVALID_ARG;
  return forward_impl(h, a, nullptr, out, workspace, workspace_bytes, stream);
}

moe_lora_status moe_lora_forward_routed(moe_lora_handle* h, const moe_lora_args* a, const moe_lora_routed* r,
                                        moe_lora_bf16* out, void* workspace, size_t workspace_bytes,
                                        moe_lora_stream stream) {
  if (a == nullptr || r == nullptr || h == nullptr || workspace == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  // the routing arguments of `a` are not used: check the rest with a stand-in routing
  moe_lora_args b = *a;
  b.router_logits = nullptr;
  b.correction_bias = nullptr;
  b.routing_method = MOE_LORA_ROUTE_RENORMALIZE;
  b.n_group = b.topk_group = 1;
  b.topk_ids = nullptr;
  b.topk_weights = nullptr;
  b.expert_offsets = nullptr;
  b.perm = nullptr;
  b.inv_perm = nullptr;
  if (b.T > 0) b.router_logits = reinterpret_cast<const moe_lora_bf16*>(r->packed_topk_ids);   // any non-null
  moe_lora_status st = moe_lora_validate(&b);
  if (st != MOE_LORA_OK) return st;
  if (b.E + 1 > kMaxExperts) return MOE_LORA_ERR_INVALID_ARG;
  if (r->num_experts < 1 || r->num_experts > 65536 || r->local_expert_offset < 0 ||
      static_cast<long long>(r->local_expert_offset) + b.E > r->num_experts || b.top_k > r->num_experts)
    return MOE_LORA_ERR_INVALID_ARG;
  if (r->do_finalize != 0 && r->do_finalize != 1) return MOE_LORA_ERR_INVALID_ARG;
  if (b.T > 0) {
    if (r->packed_topk_ids == nullptr || !aligned4(r->packed_topk_ids)) return MOE_LORA_ERR_INVALID_ARG;
    if (r->do_finalize) {
      if (out == nullptr || !aligned16(out)) return MOE_LORA_ERR_INVALID_ARG;
    } else {
      if (r->gemm2_output == nullptr || !aligned16(r->gemm2_output)) return MOE_LORA_ERR_INVALID_ARG;
      if (r->expanded_idx_to_permuted_idx == nullptr) return MOE_LORA_ERR_INVALID_ARG;
      if (r->activation_output != nullptr && !aligned16(r->activation_output)) return MOE_LORA_ERR_INVALID_ARG;
    }
    if (r->expert_weights != nullptr && !aligned4(r->expert_weights)) return MOE_LORA_ERR_INVALID_ARG;
    if (r->expanded_idx_to_permuted_idx != nullptr && !aligned4(r->expanded_idx_to_permuted_idx))
      return MOE_LORA_ERR_INVALID_ARG;
  }
  return forward_impl(h, &b, r, out, workspace, workspace_bytes, stream);
}

moe_lora_status moe_lora_forward_fp8(moe_lora_handle* h, const moe_lora_args* a, const moe_lora_fp8_weights* w,
                                     moe_lora_bf16* out, void* workspace, size_t workspace_bytes,
                                     moe_lora_stream stream) {
  if (a == nullptr || w == nullptr || h == nullptr || workspace == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  // a->w1 / a->w2 are not read: check the rest with the FP8 codes in their place
  moe_lora_args b = *a;
  b.w1 = reinterpret_cast<const moe_lora_bf16*>(w->w1);
  b.w2 = reinterpret_cast<const moe_lora_bf16*>(w->w2);
  // the fused LoRA placement needs both expand-ready B copies; otherwise the side-stream one
  if (a->lora_B_gu_packed == nullptr || a->lora_B_dn_packed == nullptr) b.flags |= MOE_LORA_FLAG_UNFUSED_LORA;
  moe_lora_status st = moe_lora_validate(&b);
  if (st != MOE_LORA_OK) return st;
  if (b.H % 128 != 0 || b.I % 128 != 0) return MOE_LORA_ERR_INVALID_ARG;
  if (b.T > 0) {
    if (out == nullptr || !aligned16(out)) return MOE_LORA_ERR_INVALID_ARG;
    if (w->w1_scale == nullptr || w->w2_scale == nullptr || !aligned4(w->w1_scale) || !aligned4(w->w2_scale))
      return MOE_LORA_ERR_INVALID_ARG;
  }
  return forward_impl(h, &b, nullptr, out, workspace, workspace_bytes, stream, w);
}

moe_lora_status moe_lora_quant_fp8(moe_lora_handle* h, const moe_lora_bf16* src, const int32_t* perm, int rows,
                                   int K, int top_k, uint8_t* codes, float* scales, moe_lora_stream stream) {
  if (h == nullptr || rows < 0 || K < 128 || K % 128 != 0 || K > 16384) return MOE_LORA_ERR_INVALID_ARG;
  if (perm != nullptr && top_k < 1) return MOE_LORA_ERR_INVALID_ARG;
  if (rows == 0) return MOE_LORA_OK;
  if (src == nullptr || codes == nullptr || scales == nullptr || !aligned16(src) || !aligned16(codes) ||
      !aligned4(scales) || (perm != nullptr && !aligned4(perm)))
    return MOE_LORA_ERR_INVALID_ARG;
  ML_LAUNCH(h, launch_quant_fp8(reinterpret_cast<const __nv_bfloat16*>(src), perm, perm != nullptr ? top_k : 1, rows, K,
                                codes, scales, stream),
            "quant launch");
  return MOE_LORA_OK;
}

moe_lora_status moe_lora_grouped_gemm_fp8(moe_lora_handle* h, const uint8_t* w, const float* w_scale,
                                          const uint8_t* x, const float* x_scale, const int32_t* expert_offsets,
                                          int E, int N, int K, int P, float* out, moe_lora_stream stream) {
  if (h == nullptr || E < 1 || E > kMaxExperts || N < 128 || N % 128 != 0 || K < 128 || K % 128 != 0 || P < 0 ||
      N > 65536 || K > 65536)
    return MOE_LORA_ERR_INVALID_ARG;
  if (static_cast<long long>(E) * N > 0x7fffffffLL) return MOE_LORA_ERR_INVALID_ARG;
  if (P == 0) return MOE_LORA_OK;
  if (!w || !w_scale || !x || !x_scale || !expert_offsets || !out || !aligned16(w) || !aligned16(x) ||
      !aligned16(out) || !aligned4(w_scale) || !aligned4(x_scale) || !aligned4(expert_offsets))
    return MOE_LORA_ERR_INVALID_ARG;
  GemmF8Params gq;
  std::memset(&gq, 0, sizeof(gq));
  gq.w_scale = w_scale;
  gq.x_scale = x_scale;
  gq.out_f32 = out;
  gq.offsets = expert_offsets;
  gq.E = E;
  gq.N = N;
  gq.K = K;
  gq.gated = 0;
  return enqueue_gemm_fp8(h, gq, w, x, P, std::min(pick_bn(P, E), 64), stream, false);
}

moe_lora_status moe_lora_forward_nvfp4(moe_lora_handle* h, const moe_lora_args* a, const moe_lora_nvfp4_weights* w,
                                       moe_lora_bf16* out, void* workspace, size_t workspace_bytes,
                                       moe_lora_stream stream) {
  if (a == nullptr || w == nullptr || h == nullptr || workspace == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  // a->w1 / a->w2 are not read: check the rest with the packed codes in their place
  moe_lora_args b = *a;
  b.w1 = reinterpret_cast<const moe_lora_bf16*>(w->w1);
  b.w2 = reinterpret_cast<const moe_lora_bf16*>(w->w2);
  b.flags |= MOE_LORA_FLAG_UNFUSED_LORA;
  moe_lora_status st = moe_lora_validate(&b);
  if (st != MOE_LORA_OK) return st;
  if (b.H % 128 != 0 || b.I % 64 != 0) return MOE_LORA_ERR_INVALID_ARG;
  if (b.T > 0) {
    if (out == nullptr || !aligned16(out)) return MOE_LORA_ERR_INVALID_ARG;
    if (w->w1_sf == nullptr || w->w2_sf == nullptr || w->w1_gs == nullptr || w->w2_gs == nullptr ||
        !aligned4(w->w1_sf) || !aligned4(w->w2_sf) || !aligned4(w->w1_gs) || !aligned4(w->w2_gs))
      return MOE_LORA_ERR_INVALID_ARG;
  }
  return forward_impl(h, &b, nullptr, out, workspace, workspace_bytes, stream, nullptr, w);
}

moe_lora_status moe_lora_quant_nvfp4(moe_lora_handle* h, const moe_lora_bf16* src, const int32_t* perm, int rows,
                                     int K, int top_k, float* g, uint8_t* codes, uint8_t* block_scales,
                                     uint16_t* deq_f16, moe_lora_stream stream) {
  if (h == nullptr || rows < 0 || K < 16 || K % 16 != 0 || K > 65536) return MOE_LORA_ERR_INVALID_ARG;
  if (codes != nullptr && K % 32 != 0) return MOE_LORA_ERR_INVALID_ARG;
  if (perm != nullptr && top_k < 1) return MOE_LORA_ERR_INVALID_ARG;
  if (rows == 0) return MOE_LORA_OK;
  if (src == nullptr || g == nullptr || !aligned16(src) || !aligned4(g) || (perm != nullptr && !aligned4(perm)) ||
      (codes != nullptr && !aligned16(codes)) || (deq_f16 != nullptr && !aligned16(deq_f16)))
    return MOE_LORA_ERR_INVALID_ARG;
  ML_LAUNCH(h, launch_quant_nvfp4(reinterpret_cast<const __nv_bfloat16*>(src), perm, perm != nullptr ? top_k : 1, rows,
                                  K, g, reinterpret_cast<__half*>(deq_f16), codes, block_scales, stream),
            "NVFP4 quant launch");
  return MOE_LORA_OK;
}

moe_lora_status moe_lora_grouped_gemm_nvfp4(moe_lora_handle* h, const uint8_t* w, const uint8_t* w_sf,
                                            const float* w_gs, const uint16_t* x, const float* x_gs,
                                            const int32_t* expert_offsets, int E, int N, int K, int P, float* out,
                                            moe_lora_stream stream) {
  if (h == nullptr || E < 1 || E > kMaxExperts || N < 128 || N % 128 != 0 || K < 64 || K % 64 != 0 || P < 0 ||
      N > 65536 || K > 65536)
    return MOE_LORA_ERR_INVALID_ARG;
  if (static_cast<long long>(E) * N > 0x7fffffffLL) return MOE_LORA_ERR_INVALID_ARG;
  if (P == 0) return MOE_LORA_OK;
  if (!w || !w_sf || !w_gs || !x || !x_gs || !expert_offsets || !out || !aligned16(w) || !aligned16(x) ||
      !aligned16(out) || !aligned4(w_sf) || !aligned4(w_gs) || !aligned4(x_gs) || !aligned4(expert_offsets))
    return MOE_LORA_ERR_INVALID_ARG;
  GemmNv4Params gq;
  std::memset(&gq, 0, sizeof(gq));
  gq.w_sf = w_sf;
  gq.w_gs = w_gs;
  gq.x_gs = x_gs;
  gq.out_f32 = out;
  gq.offsets = expert_offsets;
  gq.E = E;
  gq.N = N;
  gq.K = K;
  gq.gated = 0;
  return enqueue_gemm_nvfp4(h, gq, w, reinterpret_cast<const __half*>(x), P, std::min(pick_bn(P, E), 64), stream,
                            false);
}

moe_lora_status moe_lora_launch_count(const moe_lora_handle* h, uint64_t* count) {
  if (h == nullptr || count == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  *count = h->launches;
  return MOE_LORA_OK;
}

moe_lora_status moe_lora_check_status(const void* workspace, moe_lora_stream stream, uint32_t* detail) {
  if (workspace == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  ML_CUDA(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
  uint32_t word = 0;
  ML_CUDA(cudaMemcpy(&word, workspace, 4, cudaMemcpyDeviceToHost), "cudaMemcpy");
  if (detail) *detail = word;
  const uint32_t code = word & 0xffu;
  if (code == 0) return MOE_LORA_OK;
  if (code == MOE_LORA_ERR_TIMEOUT) return MOE_LORA_ERR_TIMEOUT;
  return MOE_LORA_ERR_DEVICE_CHECK;
}

}  // extern "C"
