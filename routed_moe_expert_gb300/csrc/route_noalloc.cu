// moe_lora_route_noalloc: routing + expert alignment for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc or hand over a workspace: code that runs inside a
// host framework whose device allocator is off limits to plug-ins, allocation-free
// real-time paths that must never touch the allocator after start-up, or a process
// whose only device memory is the input and output tensors it was given.  For them this
// entry point runs the same routing kernel as moe_lora_route, but keeps the kernel's
// scratch (per-CTA expert counts and prefixes, the grid-barrier counter and the status
// word) in a fixed array that lives in the library's own device image.
//
// The array is kNoAllocScratchBytes (512 KiB) per GPU; every GPU that loads the library
// holds it until the process exits.  The routing grid is reduced until its scratch fits
// (each routing CTA needs 8*E bytes); a shape that does not fit even one CTA is rejected.
// All calls share the array and it keeps the previous call's contents: the status word
// and barrier counter are cleared on `stream` at the start of every call, and calls whose
// work overlaps on the GPU (different streams, or different threads) race on it.
// The array's address is looked up once per device and kept for the life of the process,
// so the entry point must not be called on a device after cudaDeviceReset (or any other
// reset of its primary context) in the same process: the kept address would belong to the
// context that was torn down.
#include "../../include/moe_lora.h"
#include "kernels.h"

#include <cstring>
#include <mutex>

using namespace mlk;

namespace {

constexpr size_t kNoAllocScratchBytes = 512u * 1024u;
constexpr size_t kHeaderBytes = 256;   // status word at 0, grid-barrier counter at 4

// Device scratch of the no-allocation routing entry point.  In host code this name is a
// host-side stand-in, not a device address: host code passes the address obtained from
// cudaGetSymbolAddress instead.
static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char* g_scratch_ptr[kMaxDevices] = {};
// Cooperative routing CTAs that fit on the device, per expert count (0 = not yet asked),
// so a call after the first does no occupancy query.
int g_coop_ctas[kMaxDevices][kMaxExperts + 1] = {};

// Once per device, with that device current: resolve the array's device address; and
// once per (device, E): the cooperative grid limit of the routing kernel.
moe_lora_status setup_device(int dev, int E, unsigned char** ptr, int* coop) {
  if (dev < 0 || dev >= kMaxDevices) return MOE_LORA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return MOE_LORA_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  if (g_coop_ctas[dev][E] == 0) g_coop_ctas[dev][E] = route_max_coop_ctas(E);
  *ptr = g_scratch_ptr[dev];
  *coop = g_coop_ctas[dev][E];
  return MOE_LORA_OK;
}

}  // namespace

extern "C" moe_lora_status moe_lora_route_noalloc(const moe_lora_bf16* router_logits, const float* correction_bias,
                                                  int T, int E, int top_k, int routing_method,
                                                  float routed_scaling_factor, int n_group, int topk_group,
                                                  int32_t* topk_ids, float* topk_weights, int32_t* expert_offsets,
                                                  int32_t* perm, int32_t* inv_perm, moe_lora_stream stream) {
  if (T < 0 || E < 1 || E > kMaxExperts || top_k < 1 || top_k > E || top_k > kMaxTopK)
    return MOE_LORA_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * top_k > 0x7fffffffLL) return MOE_LORA_ERR_INVALID_ARG;
  if (routing_method != MOE_LORA_ROUTE_RENORMALIZE && routing_method != MOE_LORA_ROUTE_DEEPSEEK_V3)
    return MOE_LORA_ERR_INVALID_ARG;
  if (routing_method == MOE_LORA_ROUTE_DEEPSEEK_V3 && correction_bias == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  if (n_group > 1 || topk_group > 1) return MOE_LORA_ERR_UNSUPPORTED;
  if (n_group < 0 || topk_group < 0) return MOE_LORA_ERR_INVALID_ARG;
  if (expert_offsets == nullptr) return MOE_LORA_ERR_INVALID_ARG;
  if (T > 0 && (router_logits == nullptr || !topk_ids || !topk_weights || !perm || !inv_perm))
    return MOE_LORA_ERR_INVALID_ARG;

  // scratch needed by one routing CTA: hist and base rows of E counters; plus totals
  const size_t per_cta = 2u * static_cast<size_t>(E) * 4u;
  const size_t fixed = kHeaderBytes + static_cast<size_t>(E) * 4u;
  if (fixed + per_cta > kNoAllocScratchBytes) return MOE_LORA_ERR_UNSUPPORTED;   // cannot fit one CTA

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_LORA_ERR_CUDA;
  unsigned char* scratch = nullptr;
  int coop = 0;
  moe_lora_status st = setup_device(dev, E, &scratch, &coop);
  if (st != MOE_LORA_OK) return st;

  if (cudaMemsetAsync(scratch, 0, kHeaderBytes, stream) != cudaSuccess) return MOE_LORA_ERR_CUDA;
  if (T == 0) {
    if (cudaMemsetAsync(expert_offsets, 0, (static_cast<size_t>(E) + 1) * 4, stream) != cudaSuccess)
      return MOE_LORA_ERR_CUDA;
    return MOE_LORA_OK;
  }

  int grid = (T + 63) / 64;
  if (grid > coop) grid = coop;
  if (grid > kMaxRouteCtas) grid = kMaxRouteCtas;
  const int fit = static_cast<int>((kNoAllocScratchBytes - fixed) / per_cta);
  if (grid > fit) grid = fit;
  if (grid < 1) grid = 1;

  RouteParams p;
  std::memset(&p, 0, sizeof(p));
  p.logits = reinterpret_cast<const __nv_bfloat16*>(router_logits);
  p.bias = correction_bias;
  p.T = T;
  p.E = E;
  p.k = top_k;
  p.method = routing_method;
  p.rsf = routed_scaling_factor;
  p.tokens_per_cta = (T + grid - 1) / grid;
  p.ids = topk_ids;
  p.weights = topk_weights;
  p.offsets = expert_offsets;
  p.perm = perm;
  p.inv = inv_perm;
  p.status = reinterpret_cast<uint32_t*>(scratch);
  p.barrier = p.status + 1;
  p.total = reinterpret_cast<int32_t*>(scratch + kHeaderBytes);
  p.hist = p.total + E;
  p.base = p.hist + static_cast<size_t>(grid) * E;
  const int ctas = route_cluster_ctas(T);   // one cluster up to 512 tokens: no scratch beyond the header
  if (ctas > 0) {
    p.tokens_per_cta = (T + ctas - 1) / ctas;
    if (launch_route_cluster(p, ctas, stream) != cudaSuccess) return MOE_LORA_ERR_CUDA;
    return MOE_LORA_OK;
  }
  if (launch_route_align(p, grid, stream) != cudaSuccess) return MOE_LORA_ERR_CUDA;
  return MOE_LORA_OK;
}
