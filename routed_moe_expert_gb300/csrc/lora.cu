// Per-expert LoRA shrink (A) and expand (B) on the tensor cores, with per-token adapter
// slots of mixed rank.
//
//   shrink: u[q, r] = sum_k A[s, e, r, k] * src[row(q), k]                   (fp32)
//   expand: d[q, n] = bf16( scaling[s] * sum_{r<ranks[s]} B[s, e, n, r] * bf16(u[q, r]) )
//
// for the pair q (permuted order) of expert e whose token has slot s.  Pairs whose
// token has no adapter (slot -1, rank 0 or scaling 0) get d = 0 and no u.
//
// The gate_up chain (shrink on the hidden row, expand into the bf16 delta that the
// activation adds before SwiGLU) is sglang PR #28466's merged_experts_fused_moe_lora_add
// (gate_up), section 1 flow (B), run on the side stream; the down chain uses the shrink
// only (on the activation), and its expand is applied in the down GEMM's epilogue.
// The shrink splits K across the 8 warps of a CTA and reduces the partial sums in a
// fixed warp order, and the expand casts the fp32 shrink result to bf16 as it loads it:
// the split-K shrink with the fp32->bf16 cast fused into the expand of sglang PR #27329
// "Experimental fast LoRA path" (Optimizations).
//
// A CTA tile is one expert and up to 8*NTL consecutive permuted pairs of it, so every
// (slot, expert) adapter block is read once per tile.  Pairs of different slots share a
// tile: each slot present is processed in turn with the other pairs' columns zeroed.
// Only ranks r < ranks[s] are read, so the unused tail of a stacked adapter never
// enters the result.  Tensor-core work is mma.sync m16n8k16 (bf16 in, fp32 accumulate):
// these are small GEMMs (M = rank, N = 8 pairs) that sit beside the tcgen05 expert GEMMs.
#include "common.cuh"
#include "kernels.h"

namespace mlk {

constexpr int kLoraThreads = 256;
constexpr int kLoraWarps = 8;

MLDEV void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

MLDEV uint32_t ld_b32(const __nv_bfloat16* p) { return __ldg(reinterpret_cast<const unsigned int*>(p)); }

MLDEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

size_t lora_smem_bytes(int ntl, int R, int N, bool expand, int E) {
  const int PT = 8 * ntl;
  const int RP = ((R + 15) / 16) * 16;
  size_t b = 0;
  b += static_cast<size_t>(kLoraWarps) * RP * PT * 4;     // per-warp partials
  b += static_cast<size_t>(PT) * RP * 4;                  // u (fp32)
  b += static_cast<size_t>(PT) * (RP + 8) * 2;            // u as bf16 (padded rows)
  if (expand) b += static_cast<size_t>(PT) * N * 2;       // staged d rows
  b += static_cast<size_t>(PT) * 12 + 16;                 // pair info + slot mask
  b += 4 * (static_cast<size_t>(E) + 1);                  // schedule
  return b;
}

// NTL: n-tiles of 8 pairs per CTA tile; MTX: rank m-tiles of 16 the kernel is built for
// (ranks <= 16*MTX).  The shrink loads UK k-steps of fragments before issuing their MMAs.
template <int NTL, int MTX>
__global__ void __launch_bounds__(kLoraThreads) lora_mma_kernel(const LoraParams p) {
  constexpr int PT = 8 * NTL;
  constexpr int UK = MTX <= 2 ? 4 : (MTX <= 4 ? 2 : 1);
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_wait();
  pdl_trigger();
  const int R = p.slots.R;
  const int RP = ((R + 15) / 16) * 16;
  const bool expand = p.B != nullptr;
  float* red = reinterpret_cast<float*>(smem);                                  // [8][RP][PT]
  float* u_s = red + kLoraWarps * RP * PT;                                      // [PT][RP]
  __nv_bfloat16* ub = reinterpret_cast<__nv_bfloat16*>(u_s + PT * RP);         // [PT][RP+8]
  __nv_bfloat16* dst = ub + PT * (RP + 8);                                      // [PT][N]
  int* prow = reinterpret_cast<int*>(dst + (expand ? PT * p.N : 0));            // [PT]
  int* pslot = prow + PT;                                                       // [PT]
  int* pq = pslot + PT;                                                         // [PT]
  unsigned* smask = reinterpret_cast<unsigned*>(pq + PT);                       // [2]: slots 0-31, 32-63
  int* tile_start = reinterpret_cast<int*>(smask + 4);                          // [E+1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int E = p.E;

  if (warp == 0) {   // tile schedule over experts: ceil(M_e / PT) tiles each
    int carry = 0;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      const int cnt = (e < E) ? (p.offsets[e + 1] - p.offsets[e] + PT - 1) / PT : 0;
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      if (e < E) tile_start[e] = carry + incl - cnt;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tile_start[E] = carry;
  }
  __syncthreads();
  const int total = tile_start[E];
  const int K16 = p.K >> 4;

  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int q0 = p.offsets[e] + (tile - tile_start[e]) * PT;
    const int np = min(PT, p.offsets[e + 1] - q0);

    if (tid == 0) smask[0] = smask[1] = 0u;
    __syncthreads();
    if (tid < PT) {
      int s = -1, row = 0, q = q0 + tid;
      if (tid < np) {
        const int pp = p.perm[q];
        const int t = pp / p.k;
        row = p.by_token ? t : q;
        s = p.slot_idx[t];
        if (s < -1 || s >= p.slots.S) {
          record_status(p.status, kDevBadSlot, p.where);
          s = -1;
        } else if (s >= 0 && (p.slots.ranks[s] <= 0 || p.slots.scal[s] == 0.0f)) {
          s = -1;
        }
        if (s >= 0) atomicOr(&smask[s >> 5], 1u << (s & 31));
      }
      prow[tid] = row;
      pslot[tid] = s;
      pq[tid] = q;
      if (p.pair_slot_out != nullptr && tid < np) p.pair_slot_out[q] = s;
    }
    if (expand) {
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      for (int i = tid; i < PT * p.N / 8; i += kLoraThreads) d4[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    if (p.ub_out != nullptr) {   // every slot's row of these pairs starts at zero
      const int nz = p.slots.S * np * p.RU;
      for (int i = tid; i < nz; i += kLoraThreads) {
        const int sl = i / (np * p.RU);
        const int rem = i - sl * np * p.RU;
        const int n = rem / p.RU, r = rem - n * p.RU;
        p.ub_out[(static_cast<size_t>(sl) * p.P + pq[n]) * p.RU + r] = __float2bfloat16_rn(0.0f);
      }
      __syncthreads();
    }
    const unsigned mask0 = smask[0], mask1 = smask[1];

    for (int s = 0; s < p.slots.S; ++s) {
      if (!(((s < 32 ? mask0 : mask1) >> (s & 31)) & 1u)) continue;
      const int rank = p.slots.ranks[s];
      const int MT = (rank + 15) >> 4;
      const __nv_bfloat16* A = p.A + (static_cast<size_t>(s) * E + e) * static_cast<size_t>(R) * p.K;

      // ---------------- shrink: warps split the K steps; partials to smem
      float acc[MTX][NTL][4];
#pragma unroll
      for (int mt = 0; mt < MTX; ++mt)
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.0f;
      const __nv_bfloat16* xrow[NTL];
      bool xon[NTL];
#pragma unroll
      for (int nt = 0; nt < NTL; ++nt) {
        const int n = nt * 8 + g;
        xon[nt] = (n < np) && (pslot[n] == s);
        xrow[nt] = p.src + static_cast<size_t>(prow[n]) * p.K;
      }
      for (int ks0 = warp; ks0 < K16; ks0 += kLoraWarps * UK) {
        uint32_t bf[UK][NTL][2];
        uint32_t af[UK][MTX][4];
#pragma unroll
        for (int u = 0; u < UK; ++u) {   // all loads of UK k-steps first
          const int ks = ks0 + u * kLoraWarps;
          const bool kon = ks < K16;
          const int k0 = ks * 16 + 2 * c;
#pragma unroll
          for (int nt = 0; nt < NTL; ++nt) {
            bf[u][nt][0] = (kon && xon[nt]) ? ld_b32(xrow[nt] + k0) : 0u;
            bf[u][nt][1] = (kon && xon[nt]) ? ld_b32(xrow[nt] + k0 + 8) : 0u;
          }
#pragma unroll
          for (int mt = 0; mt < MTX; ++mt) {
            const int r0 = mt * 16 + g, r1 = r0 + 8;
            const bool on0 = kon && r0 < rank, on1 = kon && r1 < rank;
            af[u][mt][0] = on0 ? ld_b32(A + static_cast<size_t>(r0) * p.K + k0) : 0u;
            af[u][mt][1] = on1 ? ld_b32(A + static_cast<size_t>(r1) * p.K + k0) : 0u;
            af[u][mt][2] = on0 ? ld_b32(A + static_cast<size_t>(r0) * p.K + k0 + 8) : 0u;
            af[u][mt][3] = on1 ? ld_b32(A + static_cast<size_t>(r1) * p.K + k0 + 8) : 0u;
          }
        }
#pragma unroll
        for (int u = 0; u < UK; ++u)
#pragma unroll
          for (int mt = 0; mt < MTX; ++mt)
            if (mt < MT)
#pragma unroll
              for (int nt = 0; nt < NTL; ++nt) mma_bf16_16816(acc[mt][nt], af[u][mt], bf[u][nt]);
      }
      // partial [r][n] of this warp
      float* rw = red + warp * RP * PT;
#pragma unroll
      for (int mt = 0; mt < MTX; ++mt) {
        if (mt < MT) {
#pragma unroll
          for (int nt = 0; nt < NTL; ++nt) {
            const int r0 = mt * 16 + g, n0 = nt * 8 + 2 * c;
            rw[r0 * PT + n0] = acc[mt][nt][0];
            rw[r0 * PT + n0 + 1] = acc[mt][nt][1];
            rw[(r0 + 8) * PT + n0] = acc[mt][nt][2];
            rw[(r0 + 8) * PT + n0 + 1] = acc[mt][nt][3];
          }
        }
      }
      __syncthreads();
      // fixed-order reduction over the 8 warps
      for (int i = tid; i < MT * 16 * PT; i += kLoraThreads) {
        const int r = i / PT, n = i - r * PT;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kLoraWarps; ++w) v += red[w * RP * PT + i];
        const bool mine = (n < np) && (pslot[n] == s) && (r < rank);
        u_s[n * RP + r] = mine ? v : 0.0f;
        if (!expand && mine) {
          const float sv = p.slots.scal[s] * v;
          if (p.u_out != nullptr) p.u_out[static_cast<size_t>(pq[n]) * R + r] = sv;
          if (p.ub_out != nullptr)
            p.ub_out[(static_cast<size_t>(s) * p.P + pq[n]) * p.RU + r] = __float2bfloat16_rn(sv);
        }
      }
      __syncthreads();
      if (!expand) continue;

      // ---------------- expand: B operand = bf16(u), features split across warps
      for (int i = tid; i < PT * MT * 16; i += kLoraThreads) {
        const int n = i / (MT * 16), r = i - n * (MT * 16);
        ub[n * (RP + 8) + r] = __float2bfloat16_rn(u_s[n * RP + r]);
      }
      __syncthreads();
      const float sc = p.slots.scal[s];
      const __nv_bfloat16* Bm = p.B + (static_cast<size_t>(s) * E + e) * static_cast<size_t>(p.N) * R;
      const int NM = p.N >> 4;
      constexpr int UE = 4;   // feature m-tiles whose B-row loads are issued together
      for (int fm0 = warp; fm0 < NM; fm0 += kLoraWarps * UE) {
        float acc2[UE][NTL][4];
#pragma unroll
        for (int ue = 0; ue < UE; ++ue)
#pragma unroll
          for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc2[ue][nt][i] = 0.0f;
        for (int kt = 0; kt < MT; ++kt) {
          const int r0 = kt * 16 + 2 * c, r1 = r0 + 8;
          // B rows have stride R (any rank); pairs past the rank load as zero
          auto pair = [&](const __nv_bfloat16* row, int r) -> uint32_t {
            if (r + 1 < rank && (R & 1) == 0) return ld_b32(row + r);   // 4-byte aligned pair
            const float lo = r < rank ? __bfloat162float(row[r]) : 0.0f;
            const float hi = r + 1 < rank ? __bfloat162float(row[r + 1]) : 0.0f;
            return pack_bf16x2(lo, hi);
          };
          uint32_t af[UE][4];
#pragma unroll
          for (int ue = 0; ue < UE; ++ue) {
            const int fm = fm0 + ue * kLoraWarps;
            const int f0 = (fm < NM ? fm : 0) * 16 + g;
            const __nv_bfloat16* b0 = Bm + static_cast<size_t>(f0) * R;
            const __nv_bfloat16* b1 = Bm + static_cast<size_t>(f0 + 8) * R;
            af[ue][0] = pair(b0, r0);
            af[ue][1] = pair(b1, r0);
            af[ue][2] = pair(b0, r1);
            af[ue][3] = pair(b1, r1);
          }
          uint32_t bfr[NTL][2];
#pragma unroll
          for (int nt = 0; nt < NTL; ++nt) {
            const __nv_bfloat16* urow = ub + (nt * 8 + g) * (RP + 8);
            bfr[nt][0] = *reinterpret_cast<const uint32_t*>(urow + kt * 16 + 2 * c);
            bfr[nt][1] = *reinterpret_cast<const uint32_t*>(urow + kt * 16 + 2 * c + 8);
          }
#pragma unroll
          for (int ue = 0; ue < UE; ++ue)
#pragma unroll
            for (int nt = 0; nt < NTL; ++nt) mma_bf16_16816(acc2[ue][nt], af[ue], bfr[nt]);
        }
#pragma unroll
        for (int ue = 0; ue < UE; ++ue) {
          const int fm = fm0 + ue * kLoraWarps;
          if (fm >= NM) continue;
          const int f0 = fm * 16 + g, f1 = f0 + 8;
#pragma unroll
          for (int nt = 0; nt < NTL; ++nt) {
            const int n0 = nt * 8 + 2 * c, n1 = n0 + 1;
            if (n0 < np && pslot[n0] == s) {
              dst[n0 * p.N + f0] = __float2bfloat16_rn(sc * acc2[ue][nt][0]);
              dst[n0 * p.N + f1] = __float2bfloat16_rn(sc * acc2[ue][nt][2]);
            }
            if (n1 < np && pslot[n1] == s) {
              dst[n1 * p.N + f0] = __float2bfloat16_rn(sc * acc2[ue][nt][1]);
              dst[n1 * p.N + f1] = __float2bfloat16_rn(sc * acc2[ue][nt][3]);
            }
          }
        }
      }
      __syncthreads();
    }

    if (expand) {   // staged rows (zeros for pairs without an adapter) -> d
      const int N8 = p.N >> 3;
      const uint4* s4 = reinterpret_cast<const uint4*>(dst);
      for (int i = tid; i < np * N8; i += kLoraThreads) {
        const int n = i / N8, j = i - n * N8;
        reinterpret_cast<uint4*>(p.d_out + static_cast<size_t>(pq[n]) * p.N)[j] = s4[i];
      }
    }
    __syncthreads();
  }
}

template <int NTL, int MTX>
static cudaError_t launch_t(const LoraParams& p, int grid, size_t smem, cudaStream_t stream, bool pdl) {
  cudaError_t err = cudaFuncSetAttribute(lora_mma_kernel<NTL, MTX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_k(lora_mma_kernel<NTL, MTX>, dim3(grid), dim3(kLoraThreads), smem, stream, pdl, p);
}

template <int NTL>
static cudaError_t launch_ntl(const LoraParams& p, int grid, size_t smem, cudaStream_t stream, bool pdl) {
  const int R = p.slots.R;
  if (R <= 16) return launch_t<NTL, 1>(p, grid, smem, stream, pdl);
  if (R <= 32) return launch_t<NTL, 2>(p, grid, smem, stream, pdl);
  if (R <= 64) return launch_t<NTL, 4>(p, grid, smem, stream, pdl);
  return launch_t<NTL, 8>(p, grid, smem, stream, pdl);
}

cudaError_t launch_lora(const LoraParams& p, int ntl, int grid, cudaStream_t stream, bool pdl) {
  if (p.P == 0) return cudaSuccess;
  const size_t smem = lora_smem_bytes(ntl, p.slots.R, p.N, p.B != nullptr, p.E);
  return ntl == 1 ? launch_ntl<1>(p, grid, smem, stream, pdl) : launch_ntl<4>(p, grid, smem, stream, pdl);
}

}  // namespace mlk
