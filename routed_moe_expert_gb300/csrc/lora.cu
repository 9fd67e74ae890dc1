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
  b += 8 * (static_cast<size_t>(E) + 1);                  // schedule and staged offsets
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
  int* seg = tile_start + (p.E + 1);                                            // [E+1] offsets

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int E = p.E;

  if (warp == 0) build_tile_schedule(p.offsets, E, PT, 1, seg, tile_start);   // ceil(M_e / PT) tiles each
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
    const int q0 = seg[e] + (tile - tile_start[e]) * PT;
    const int np = min(PT, seg[e + 1] - q0);

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
      const __nv_bfloat16* A =
          p.A + (static_cast<size_t>(s) * (p.a_e1 ? 1 : E) + (p.a_e1 ? 0 : e)) * static_cast<size_t>(R) * p.K;

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
      const __nv_bfloat16* Bm =
          p.B + (static_cast<size_t>(s) * (p.b_e1 ? 1 : E) + (p.b_e1 ? 0 : e)) * static_cast<size_t>(p.N) * R;
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

// ---------------------------------------------------------------------------------
// Activation with the down-LoRA shrink in the same pass (narrow expert tiles): for a tile
// of up to 8 pairs of one expert,
//   a[q, i] = bf16( silu(g_gate + d_gate) * (g_up + d_up) )      (as activation_kernel)
//   v[q, r] = scaling[s] * sum_i a[q, i] * A_dn[s, e, r, i]       (fp32, r < ranks[s])
// with the bf16 activation rows kept in shared memory for the shrink.  The shrink runs on
// the tensor cores (mma.sync m16n8k16: M = rank rows of the slot's A block, N = the 8
// pairs, K = I split over the 8 warps), one slot present in the tile at a time; the warps'
// partial sums are added in warp order.  Rank rows past the slot's rank are never loaded
// and their results never stored.  The down GEMM's epilogue applies the expand from v.
// Pairs without an adapter get pair_slot -1 and no v.
// ---------------------------------------------------------------------------------
constexpr int kActTile = 8;

template <int MTX>
__global__ void __launch_bounds__(kLoraThreads) act_shrink_kernel(const ActShrinkParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_wait();
  pdl_trigger();
  const int E = p.E, I = p.I, I8 = p.I >> 3, R = p.slots.R;
  const int AS = I + 8;   // activation row stride in shared memory (bank-conflict padding)
  __nv_bfloat16* a_s = reinterpret_cast<__nv_bfloat16*>(smem);                 // [8][AS]
  float* red = reinterpret_cast<float*>(a_s + kActTile * AS);                   // [8 warps][16*MTX][8]
  int* pslot = reinterpret_cast<int*>(red + kLoraWarps * 16 * MTX * kActTile); // [8]
  unsigned* smask = reinterpret_cast<unsigned*>(pslot + kActTile);              // [2]
  int* tile_start = reinterpret_cast<int*>(smask + 2);                          // [E+1]
  int* seg = tile_start + (E + 1);                                              // [E+1] offsets
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;

  if (warp == 0) build_tile_schedule(p.offsets, E, kActTile, 1, seg, tile_start);   // ceil(M_e / 8) tiles each
  __syncthreads();
  const int total = tile_start[E];

  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int q0 = seg[e] + (tile - tile_start[e]) * kActTile;
    const int np = min(kActTile, seg[e + 1] - q0);
    if (tid == 0) smask[0] = smask[1] = 0u;
    __syncthreads();
    if (tid < np) {
      const int q = q0 + tid;
      int s = p.pair_slot[q];
      if (s < -1 || s >= p.slots.S) {
        record_status(p.status, kDevBadSlot, kWhereLoraShrinkDn);
        s = -1;
      } else if (s >= 0 && (p.slots.ranks[s] <= 0 || p.slots.scal[s] == 0.0f)) {
        s = -1;
      }
      pslot[tid] = s;
      p.pair_slot[q] = s;
      if (s >= 0) atomicOr(&smask[s >> 5], 1u << (s & 31));
    }
    // activation rows of the tile -> global and shared memory
    for (int i = tid; i < np * I8; i += kLoraThreads) {
      const int n = i / I8, i0 = (i - n * I8) * 8;
      const int blk = i0 >> 6, j = i0 & 63;
      const size_t row = static_cast<size_t>(q0 + n) * 2 * I;
      float gf[8], uf[8], dg[8], du[8];
      unpack8(*reinterpret_cast<const uint4*>(p.g + row + blk * 128 + j), gf);
      unpack8(*reinterpret_cast<const uint4*>(p.g + row + blk * 128 + 64 + j), uf);
      unpack8(*reinterpret_cast<const uint4*>(p.d + row + i0), dg);
      unpack8(*reinterpret_cast<const uint4*>(p.d + row + I + i0), du);
      float out[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const float zg = gf[m] + dg[m], zu = uf[m] + du[m];
        out[m] = __fdividef(zg, 1.0f + __expf(-zg)) * zu;
      }
      const uint4 v = pack8(out);
      *reinterpret_cast<uint4*>(p.a + static_cast<size_t>(q0 + n) * I + i0) = v;
      *reinterpret_cast<uint4*>(a_s + n * AS + i0) = v;
    }
    __syncthreads();
    const unsigned m0 = smask[0], m1 = smask[1];
    for (int s = 0; s < p.slots.S; ++s) {
      if (!(((s < 32 ? m0 : m1) >> (s & 31)) & 1u)) continue;
      const int rank = p.slots.ranks[s];
      const int MT = (rank + 15) >> 4;
      const __nv_bfloat16* A = p.A + (static_cast<size_t>(s) * E + e) * static_cast<size_t>(R) * I;
      float acc[MTX][4];
#pragma unroll
      for (int mt = 0; mt < MTX; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][i] = 0.0f;
      // the A fragments of KU k-steps are loaded before their MMAs, so their latencies overlap
      constexpr int KU = MTX >= 8 ? 1 : 8 / MTX;
      const int nks = I >> 4;
      for (int ks0 = warp; ks0 < nks; ks0 += kLoraWarps * KU) {
        uint32_t af[KU][MTX][4], bf[KU][2];
#pragma unroll
        for (int u = 0; u < KU; ++u) {
          const int ks = ks0 + u * kLoraWarps;
          const bool kin = ks < nks;
          const int k0 = (kin ? ks : 0) * 16 + 2 * c;
          bf[u][0] = kin ? *reinterpret_cast<const uint32_t*>(a_s + g * AS + k0) : 0u;
          bf[u][1] = kin ? *reinterpret_cast<const uint32_t*>(a_s + g * AS + k0 + 8) : 0u;
#pragma unroll
          for (int mt = 0; mt < MTX; ++mt) {
            const int r0 = mt * 16 + g, r1 = r0 + 8;
            const bool ok0 = kin && mt < MT && r0 < rank, ok1 = kin && mt < MT && r1 < rank;
            const __nv_bfloat16* A0 = A + static_cast<size_t>(r0) * I + k0;
            const __nv_bfloat16* A1 = A + static_cast<size_t>(r1) * I + k0;
            af[u][mt][0] = ok0 ? ld_b32(A0) : 0u;
            af[u][mt][1] = ok1 ? ld_b32(A1) : 0u;
            af[u][mt][2] = ok0 ? ld_b32(A0 + 8) : 0u;
            af[u][mt][3] = ok1 ? ld_b32(A1 + 8) : 0u;
          }
        }
#pragma unroll
        for (int u = 0; u < KU; ++u)
#pragma unroll
          for (int mt = 0; mt < MTX; ++mt)
            if (ks0 + u * kLoraWarps < nks && mt < MT) mma_bf16_16816(acc[mt], af[u][mt], bf[u]);
      }
      // partials [row][pair] of this warp, then the fixed-order sum over warps
      float* rw = red + warp * 16 * MTX * kActTile;
#pragma unroll
      for (int mt = 0; mt < MTX; ++mt) {
        if (mt < MT) {
          rw[(mt * 16 + g) * kActTile + 2 * c] = acc[mt][0];
          rw[(mt * 16 + g) * kActTile + 2 * c + 1] = acc[mt][1];
          rw[(mt * 16 + g + 8) * kActTile + 2 * c] = acc[mt][2];
          rw[(mt * 16 + g + 8) * kActTile + 2 * c + 1] = acc[mt][3];
        }
      }
      __syncthreads();
      for (int i = tid; i < np * rank; i += kLoraThreads) {
        const int n = i / rank, r = i - n * rank;
        if (pslot[n] != s) continue;
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kLoraWarps; ++w) sum += red[(w * 16 * MTX + r) * kActTile + n];
        p.v[static_cast<size_t>(q0 + n) * R + r] = p.slots.scal[s] * sum;
      }
      __syncthreads();
    }
  }
}

template <int MTX>
static size_t act_shrink_smem(int I, int E) {
  return static_cast<size_t>(kActTile) * (I + 8) * 2 + static_cast<size_t>(kLoraWarps) * 16 * MTX * kActTile * 4 +
         4 * (kActTile + 2 + 2 * (static_cast<size_t>(E) + 1));
}

template <int MTX>
static cudaError_t launch_act_mtx(const ActShrinkParams& p, int grid, cudaStream_t stream, bool pdl) {
  const size_t smem = act_shrink_smem<MTX>(p.I, p.E);
  cudaError_t err = cudaFuncSetAttribute(act_shrink_kernel<MTX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_k(act_shrink_kernel<MTX>, dim3(grid), dim3(kLoraThreads), smem, stream, pdl, p);
}

cudaError_t launch_act_shrink(const ActShrinkParams& p, int grid, cudaStream_t stream, bool pdl) {
  if (p.P == 0) return cudaSuccess;
  const int R = p.slots.R;
  if (R <= 16) return launch_act_mtx<1>(p, grid, stream, pdl);
  if (R <= 32) return launch_act_mtx<2>(p, grid, stream, pdl);
  if (R <= 64) return launch_act_mtx<4>(p, grid, stream, pdl);
  return launch_act_mtx<8>(p, grid, stream, pdl);
}

}  // namespace mlk
