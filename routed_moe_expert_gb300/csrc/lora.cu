// Per-expert LoRA shrink (A) and expand (B) with per-token adapter slots of mixed rank.
//
// shrink: u[q, r] = sum_k A[s, e, r, k] * src[row(q), k]    for r < ranks[s]   (fp32)
// expand: d[q, n] = bf16( scaling[s] * sum_{r<ranks[s]} B[s, e, n, r] * u[q, r] )
// for the pair q (permuted order) with expert e and token slot s; pairs whose token
// has no adapter (slot -1, rank 0 or scaling 0) get d = 0 and no shrink.
//
// The gate_up chain (shrink on the hidden row, expand into the bf16 delta added before
// SwiGLU) is sglang PR #28466's merged_experts_fused_moe_lora_add(gate_up), section 1
// flow (B): "gate_up shrink + expand -> gate_up_lora_delta", run on the side stream;
// the down chain's shrink runs on the activation and its expand is fused into the
// finalize.  The split of K across the 32 lanes of a warp, reduced in a fixed order,
// is the split-K shrink of sglang PR #27329 "Experimental fast LoRA path"
// (Optimizations: "Split-K LoRA shrink with the fp32->bf16 cast fused into the LoRA-B
// expand"): the fp32 shrink result is read by the expand, which rounds once, on output.
// Only ranks r < ranks[s] are read, so the unused tail of a stacked adapter never
// enters the result.
#include "common.cuh"
#include "kernels.h"

namespace mlk {

// Slot of a pair's token, or -1 when it gets no LoRA.  Records a device-check status
// for an index outside [-1, S).
MLDEV int lora_slot(const LoraSlots& L, const int32_t* slot_idx, int t, uint32_t* status, uint32_t where) {
  const int s = slot_idx[t];
  if (s < -1 || s >= L.S) {
    record_status(status, kDevBadSlot, where);
    return -1;
  }
  if (s < 0 || L.ranks[s] <= 0 || L.scal[s] == 0.0f) return -1;
  return s;
}

// One warp per permuted pair q; lanes split K in 8-element vectors.
__global__ void __launch_bounds__(256) lora_shrink_kernel(const ShrinkParams p) {
  const int q = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (q >= p.P) return;
  const int pp = p.perm[q];
  const int t = pp / p.k;
  const int s = lora_slot(p.slots, p.slot_idx, t, lane == 0 ? p.status : nullptr, p.where);
  if (s < 0) return;
  const int e = p.ids[pp];
  const int rank = p.slots.ranks[s];
  const int K8 = p.K >> 3;
  const int row = p.by_token ? t : q;
  const uint4* xr = reinterpret_cast<const uint4*>(p.src + static_cast<size_t>(row) * p.K);
  const uint4* Ab = reinterpret_cast<const uint4*>(
      p.A + (static_cast<size_t>(s) * p.slots.E + e) * static_cast<size_t>(p.slots.R) * p.K);
  for (int r0 = 0; r0 < rank; r0 += 4) {
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int v = lane; v < K8; v += 32) {
      float xf[8];
      unpack8(__ldg(xr + v), xf);
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        if (r0 + rr < rank) {
          float af[8];
          unpack8(__ldg(Ab + static_cast<size_t>(r0 + rr) * K8 + v), af);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[rr] += af[i] * xf[i];
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      float v = acc[rr];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0 && r0 + rr < rank) p.u[static_cast<size_t>(q) * p.slots.R + r0 + rr] = v;
    }
  }
}

cudaError_t launch_lora_shrink(const ShrinkParams& p, cudaStream_t stream) {
  if (p.P == 0) return cudaSuccess;
  lora_shrink_kernel<<<(p.P + 7) / 8, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

// One CTA per permuted pair q; each thread produces 8 consecutive n.
__global__ void __launch_bounds__(256) lora_expand_kernel(const ExpandParams p) {
  __shared__ float u_s[kMaxRank];
  __shared__ int slot_s;
  const int q = blockIdx.x, tid = threadIdx.x;
  const int pp = p.perm[q];
  if (tid == 0) slot_s = lora_slot(p.slots, p.slot_idx, pp / p.k, p.status, kWhereLoraExpandGu);
  __syncthreads();
  const int s = slot_s;
  const int N8 = p.N >> 3;
  uint4* drow = reinterpret_cast<uint4*>(p.d + static_cast<size_t>(q) * p.N);
  if (s < 0) {
    for (int n8 = tid; n8 < N8; n8 += blockDim.x) drow[n8] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const int rank = p.slots.ranks[s];
  for (int r = tid; r < rank; r += blockDim.x) u_s[r] = p.u[static_cast<size_t>(q) * p.slots.R + r];
  __syncthreads();
  const float sc = p.slots.scal[s];
  const int e = p.ids[pp];
  const __nv_bfloat16* Bb = p.B + (static_cast<size_t>(s) * p.slots.E + e) * static_cast<size_t>(p.N) * p.slots.R;
  for (int n8 = tid; n8 < N8; n8 += blockDim.x) {
    float out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const __nv_bfloat16* Brow = Bb + static_cast<size_t>(n8 * 8 + i) * p.slots.R;
      float acc = 0.0f;
      for (int r = 0; r < rank; ++r) acc += bf2f(Brow[r]) * u_s[r];
      out[i] = sc * acc;
    }
    drow[n8] = pack8(out);
  }
}

cudaError_t launch_lora_expand(const ExpandParams& p, cudaStream_t stream) {
  if (p.P == 0) return cudaSuccess;
  lora_expand_kernel<<<p.P, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mlk
