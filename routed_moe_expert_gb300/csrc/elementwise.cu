// Memory-bound stages of the routed MoE-LoRA layer: token permute, SwiGLU activation
// with the gate_up LoRA delta, and the weighted top-k finalize.
#include <cuda_fp8.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace mlk {

// ---------------------------------------------------------------------------------
// permute: xp[q, :] = x[perm[q] / k, :]   (sglang PR #28466, Files changed, launcher
// row: "moe::dev::permute (bf16 gather)").  One warp per permuted row, 16-byte vectors.
// With slot_out set it also gathers each pair's adapter slot, slot_out[q] = slot_idx[t]
// (checked later by the kernel that uses it).  zero_out[0, zero_n) is cleared (the ready
// flags of the GEMMs that follow).
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) permute_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ perm,
                                                      int P, int k, int H8, uint4* __restrict__ xp,
                                                      const int32_t* __restrict__ slot_idx, int32_t* slot_out,
                                                      int* zero_out, int zero_n) {
  pdl_wait();
  pdl_trigger();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < zero_n; i += gridDim.x * blockDim.x) zero_out[i] = 0;
  const int q = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (q >= P) return;
  const int t = perm[q] / k;
  if (slot_out != nullptr && (threadIdx.x & 31) == 0) slot_out[q] = slot_idx[t];
  const uint4* src = x + static_cast<size_t>(t) * H8;
  uint4* dst = xp + static_cast<size_t>(q) * H8;
  // the permuted rows are read next (LoRA shrink, gate_up GEMM): keep them in L2 if they fit
  const uint64_t pol = l2_policy_evict_last();
  for (int v = threadIdx.x & 31; v < H8; v += 32) st_global_v4_hint(dst + v, __ldg(src + v), pol);
}

cudaError_t launch_permute(const __nv_bfloat16* x, const int32_t* perm, int P, int k, int H,
                           __nv_bfloat16* xp, cudaStream_t stream, bool pdl, const int32_t* slot_idx,
                           int32_t* slot_out, int* zero_out, int zero_n) {
  if (P == 0) return cudaSuccess;
  return launch_k(permute_kernel, dim3((P + 7) / 8), dim3(256), 0, stream, pdl, reinterpret_cast<const uint4*>(x),
                  perm, P, k, H / 8, reinterpret_cast<uint4*>(xp), slot_idx, slot_out, zero_out, zero_n);
}

// ---------------------------------------------------------------------------------
// activation: a[q, i] = bf16( silu(g_gate + d_gate) * (g_up + d_up) )
// (sglang PR #28466, launcher row: "moe::dev::activation (de-interleaves on read, adds
// gate_up_lora_delta pre-SwiGLU, captures activation_lora_input, bf16 out)").
// g is the gated-interleaved GEMM output: row q, block b of 128 columns = 64 gate
// features [64b, 64b+64) then the matching 64 up features.  d (or null) is the LoRA
// delta in the logical [gate | up] order.  The output a is also the down-LoRA input.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) activation_kernel(const __nv_bfloat16* __restrict__ g,
                                                         const __nv_bfloat16* __restrict__ d, int P, int I,
                                                         __nv_bfloat16* __restrict__ a) {
  pdl_wait();
  pdl_trigger();
  const int I8 = I >> 3;
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<size_t>(P) * I8) return;
  const int q = static_cast<int>(idx / I8);
  const int i0 = static_cast<int>(idx % I8) * 8;
  const int blk = i0 >> 6, j = i0 & 63;
  const size_t row = static_cast<size_t>(q) * 2 * I;
  float gf[8], uf[8];
  unpack8(*reinterpret_cast<const uint4*>(g + row + blk * 128 + j), gf);
  unpack8(*reinterpret_cast<const uint4*>(g + row + blk * 128 + 64 + j), uf);
  if (d != nullptr) {
    float dg[8], du[8];
    unpack8(*reinterpret_cast<const uint4*>(d + row + i0), dg);
    unpack8(*reinterpret_cast<const uint4*>(d + row + I + i0), du);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      gf[i] += dg[i];
      uf[i] += du[i];
    }
  }
  float out[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) out[i] = gf[i] / (1.0f + expf(-gf[i])) * uf[i];
  *reinterpret_cast<uint4*>(a + static_cast<size_t>(q) * I + i0) = pack8(out);
}

cudaError_t launch_activation(const __nv_bfloat16* g, const __nv_bfloat16* d, int P, int I,
                              __nv_bfloat16* a, cudaStream_t stream, bool pdl) {
  const size_t n = static_cast<size_t>(P) * (I / 8);
  if (n == 0) return cudaSuccess;
  return launch_k(activation_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, stream, pdl, g, d,
                  P, I, a);
}

// ---------------------------------------------------------------------------------
// finalize: out[t, h] = bf16( sum_{j<k} w[t,j] * y[inv[t*k + j], h] ), fixed j order, fp32.
// y (fp32, or bf16 at wide token tiles) already holds the down GEMM output plus the
// (unweighted) down-LoRA delta, added in the down GEMM's epilogue, so this is the vLLM API
// page's _finalize_with_w2_lora
// ("fused_moe/experts/trtllm_lora_moe": routing-weighted sum over top_k of the base rows
// plus the routing-weighted down-LoRA delta).  A CTA covers 512 h (fp32 y) or 1024 h (bf16 y)
// of one token.
// ---------------------------------------------------------------------------------
constexpr int kFinThreads = 128;   // one 16-byte vector of y each: 512 h (fp32) or 1024 h (bf16) per CTA

MLDEV void unpack_y(const uint4& v, float (&f)[4]) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}
MLDEV void unpack_y(const uint4& v, float (&f)[8]) { unpack8(v, f); }

// Each thread sums one 16-byte vector of the token's k rows of y (4 fp32 or 8 bf16 values):
// the k loads (and those of the side-stream delta) go out together, 8 pairs at a time, and
// are added in the fixed order j = 0, 1, ..., k - 1.
template <typename YT, bool DD>
__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const FinalizeParams p, const YT* __restrict__ y) {
  constexpr int V = 16 / sizeof(YT);
  __shared__ int q_s[kMaxTopK];
  __shared__ float w_s[kMaxTopK];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x, k = p.k, tid = threadIdx.x;
  if (tid < k) {
    const size_t pp = static_cast<size_t>(t) * k + tid;
    q_s[tid] = p.inv[pp];
    w_s[tid] = p.weights[pp];
  }
  __syncthreads();
  const int hv = blockIdx.y * kFinThreads + tid;   // vector index within the row
  if (hv >= p.H / V) return;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.0f;
  const uint4* yv = reinterpret_cast<const uint4*>(y);
  // the down-LoRA delta computed beside the down GEMM (bf16 [P, H]): V values = 2V bytes
  using DT = typename std::conditional<V == 8, uint4, uint2>::type;
  const DT* dv = DD ? reinterpret_cast<const DT*>(p.dd) : nullptr;
  const size_t HV = static_cast<size_t>(p.H / V);
  for (int j0 = 0; j0 < k; j0 += 8) {
    uint4 raw[8];
    DT rawd[DD ? 8 : 1];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int j = j0 + jj;
      // a pair of an expert outside the local range (routed entry) has q < 0: skipped
      const int q = j < k ? q_s[j] : -1;
      raw[jj] = q >= 0 ? __ldg(yv + static_cast<size_t>(q) * HV + hv) : make_uint4(0u, 0u, 0u, 0u);
      if constexpr (DD) rawd[jj] = q >= 0 ? __ldg(dv + static_cast<size_t>(q) * HV + hv) : DT{};
    }
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int j = j0 + jj;
      if (j >= k || q_s[j] < 0) continue;
      float v[V];
      unpack_y(raw[jj], v);
      if constexpr (DD) {
        const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&rawd[jj]);
#pragma unroll
        for (int i = 0; i < V / 2; ++i) {
          const float2 d = __bfloat1622float2(d2[i]);
          v[2 * i] += d.x;
          v[2 * i + 1] += d.y;
        }
      }
      const float w = w_s[j];
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += w * v[i];
    }
  }
  if constexpr (V == 8) {
    reinterpret_cast<uint4*>(p.out + static_cast<size_t>(t) * p.H)[hv] = pack8(acc);
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0], acc[1]);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2], acc[3]);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&lo);
    o.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(p.out + static_cast<size_t>(t) * p.H)[hv] = o;
  }
}

cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t stream, bool pdl) {
  if (p.T == 0) return cudaSuccess;
  const bool f32 = p.y != nullptr;
  const int HV = p.H / (f32 ? 4 : 8);
  const dim3 grid(p.T, (HV + kFinThreads - 1) / kFinThreads);
  const bool dd = p.dd != nullptr;
  if (f32)
    return dd ? launch_k(finalize_kernel<float, true>, grid, dim3(kFinThreads), 0, stream, pdl, p, p.y)
              : launch_k(finalize_kernel<float, false>, grid, dim3(kFinThreads), 0, stream, pdl, p, p.y);
  return dd ? launch_k(finalize_kernel<__nv_bfloat16, true>, grid, dim3(kFinThreads), 0, stream, pdl, p, p.y_bf16)
            : launch_k(finalize_kernel<__nv_bfloat16, false>, grid, dim3(kFinThreads), 0, stream, pdl, p, p.y_bf16);
}

// ---------------------------------------------------------------------------------
// FP8 group quantisation, with an optional gather: the per_token_group_quant_fp8 step
// and the post-activation quant of the pages' FP8 flow (sglang PR #28466, section 1 flow
// (A) diagram).  Row q of the output comes from source row t = perm[q] / k (or t = q
// without perm).  Per group g of 128 consecutive values v of that row:
//   s = max(amax, 1e-10) / 448,   codes[q, 128g + i] = e4m3(v_i / s),   scale[g * P + q] = s,
// with the scale and the quotients IEEE float32 divisions rounded to nearest and the
// conversion rounded to nearest even and saturated at +-448.  One warp per row, 4 values
// per lane and group.  With slot_out set it also gathers each pair's adapter slot.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_fp8_kernel(const __nv_bfloat16* __restrict__ src,
                                                        const int32_t* __restrict__ perm, int k, int P, int K,
                                                        uint8_t* __restrict__ codes, float* __restrict__ scale,
                                                        const int32_t* __restrict__ slot_idx, int32_t* slot_out) {
  pdl_wait();
  pdl_trigger();
  const int q = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (q >= P) return;
  const int t = perm != nullptr ? perm[q] / k : q;
  if (slot_out != nullptr && lane == 0) slot_out[q] = slot_idx[t];
  const uint2* s = reinterpret_cast<const uint2*>(src + static_cast<size_t>(t) * K);
  uint32_t* d = reinterpret_cast<uint32_t*>(codes + static_cast<size_t>(q) * K);
  const int G = K >> 7;
#pragma unroll 4
  for (int g = 0; g < G; ++g) {
    const uint2 v = __ldg(s + g * 32 + lane);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
    const float f[4] = {lo.x, lo.y, hi.x, hi.y};
    float amax = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sc = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      packed |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fdiv_rn(f[i], sc), __NV_SATFINITE, __NV_E4M3))
                << (8 * i);
    d[g * 32 + lane] = packed;
    if (lane == 0) scale[static_cast<size_t>(g) * P + q] = sc;
  }
}

cudaError_t launch_quant_fp8(const __nv_bfloat16* src, const int32_t* perm, int k, int P, int K, uint8_t* codes,
                             float* scale, cudaStream_t stream, bool pdl, const int32_t* slot_idx, int32_t* slot_out) {
  if (P == 0) return cudaSuccess;
  if (K % 128 != 0) return cudaErrorInvalidValue;
  return launch_k(quant_fp8_kernel, dim3((P + 7) / 8), dim3(256), 0, stream, pdl, src, perm, k, P, K, codes, scale,
                  slot_idx, slot_out);
}

}  // namespace mlk
