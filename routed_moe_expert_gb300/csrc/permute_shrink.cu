// Token permute fused with the gate_up LoRA shrink, for the fused (wide-tile) LoRA placement.
//
//   xp[q, :]     = x[perm[q] / k, :]                                    (the permute)
//   ub[s, q, r]  = bf16( scaling[s] * sum_h A_gu[s, e, r, h] * x[t, h] )  for s = slot(t), r < ranks[s]
//   ub[s', q, r] = 0                                                    for every other (s', r < RU)
//   pair_slot[q] = slot(t), or -1 when the token has no active adapter
//
// for the pairs q of expert e (t = perm[q] / k).  The permute is the pages' moe::dev::permute
// (sglang PR #28466, Files changed, launcher row) and the shrink the A half of the gate_up
// LoRA (section 1, merged_experts_fused_moe_lora_add); its expand runs inside the gate_up
// GEMM.  Both read the same token rows, so one pass does both: the hidden rows are gathered
// once into shared memory (they stay in L2: every token is read by k pairs), written out as
// the permuted rows and multiplied there by the adapter rows.  The separate shrink kernel had
// to read the permuted rows back from HBM (k times the hidden states' bytes).
//
// A CTA tile is up to 64 consecutive permuted pairs of one expert; the rank rows of every
// slot present among them are stacked as the N side of mma.sync m16n8k16 (M = the pairs, K = H
// in 64-wide chunks).  Chunks of the token rows and adapter rows move by cp.async through a
// ring of 4 or 8 stages (16-byte pieces, 128-byte rows with the 16-byte chunk index XORed with
// the row index, so ldmatrix reads them without bank conflicts).
#include "common.cuh"
#include "kernels.h"

namespace mlk {

constexpr int kPsThreads = 256;
constexpr int kPsTile = 64;     // pairs per tile
constexpr int kPsMaxStages = 8;
constexpr int kPsMaxRows = 256; // stacked rank rows per tile (S * R <= 256 on the fused path)

MLDEV void cp_async16(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
               : "memory");
}
MLDEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
MLDEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

MLDEV void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
MLDEV void ldsm_x2(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
MLDEV void mma_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// byte offset of 16-byte piece c of row r in a tile of 128-byte rows
MLDEV uint32_t sw_off(int r, int c) { return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4)); }

// The ring is as deep as fits 200 KB (at most 8 stages, at least 4): the adapter rows of a tile
// stream from HBM chunk by chunk, so the bytes in flight set its speed.
int permute_shrink_stages(int nr_max) {
  const int stage = (kPsTile + ((nr_max + 7) & ~7)) * 128;
  return 8 * stage <= 200 * 1024 ? 8 : 4;
}

size_t permute_shrink_smem_bytes(int nr_max, int E) {
  const int nr = (nr_max + 7) & ~7;
  return 128 + static_cast<size_t>(permute_shrink_stages(nr_max)) * (kPsTile + nr) * 128 + kPsTile * 8 + nr * 8 +
         4 * (4 + kMaxFusedSlots) + 8 * (static_cast<size_t>(E) + 1);
}

// NT8: n8 tiles of stacked rank rows each warp covers (two warps per 16-pair m-tile);
// NS: depth of the cp.async ring.
template <int NT8, int NS>
__global__ void __launch_bounds__(kPsThreads) permute_shrink_kernel(const PermuteShrinkParams p) {
  constexpr int kPsStages = NS;
  extern __shared__ __align__(128) uint8_t ps_smem[];
  uint8_t* smem = ps_smem + ((128u - (smem_u32(ps_smem) & 127u)) & 127u);
  const int NRMAX = p.nr_max;                               // stacked rows the stages hold (multiple of 8)
  const int STAGE = (kPsTile + NRMAX) * 128;
  int* prow = reinterpret_cast<int*>(smem + kPsStages * STAGE);   // [64] source token row
  int* pslot = prow + kPsTile;                                    // [64] active slot or -1
  long long* arow = reinterpret_cast<long long*>(pslot + kPsTile);   // [NRMAX] A row element offsets
  int* sinfo = reinterpret_cast<int*>(arow + NRMAX);               // [4]: slot mask, rows
  int* soff = sinfo + 4;                                           // [8] first stacked row per slot
  int* tile_start = soff + kMaxFusedSlots;                         // [E+1]
  int* seg = tile_start + (p.E + 1);                               // [E+1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E, H = p.H, KCH = p.H >> 6;
  const int R = p.slots.R;
  const int Ea = p.a_e1 ? 1 : E;

  // The hidden rows are read k times (once per pair of the token): keep them in L2.  The
  // permuted rows are written once here and read next by the gate_up GEMM from HBM anyway:
  // stream them, so they do not push the hidden rows out of L2.
  const uint64_t pol_keep = l2_policy_evict_last();
  const uint64_t pol_stream = l2_policy_evict_first();
  uint64_t pol_normal;   // the adapter rows: reused across an expert's tiles, or read once
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol_normal));
  pdl_wait();    // the routing (perm, offsets) comes from the previous kernel
  pdl_trigger();
  if (warp == 0) build_tile_schedule(p.offsets, E, kPsTile, 1, seg, tile_start);
  __syncthreads();
  const int total = tile_start[E];

  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int q0 = seg[e] + (tile - tile_start[e]) * kPsTile;
    const int np = min(kPsTile, seg[e + 1] - q0);
    if (tid == 0) sinfo[0] = 0;
    __syncthreads();
    if (tid < kPsTile) {
      int s = -1, t = 0;
      if (tid < np) {
        t = p.perm[q0 + tid] / p.k;
        s = p.slot_idx[t];
        if (s < -1 || s >= p.slots.S) {
          record_status(p.status, kDevBadSlot, kWhereLoraShrinkGu);
          s = -1;
        } else if (s >= 0 && (p.slots.ranks[s] <= 0 || p.slots.scal[s] == 0.0f)) {
          s = -1;
        }
        if (s >= 0) atomicOr(reinterpret_cast<unsigned*>(&sinfo[0]), 1u << s);
        p.pair_slot[q0 + tid] = s;
      }
      prow[tid] = t;
      pslot[tid] = s;
    }
    __syncthreads();
    const unsigned smask = static_cast<unsigned>(sinfo[0]);
    // stacked rank rows of the slots present (slot order): A row offsets, first row per slot
    if (tid == 0) {
      int j = 0;
      for (int s = 0; s < p.slots.S && s < kMaxFusedSlots; ++s) {
        soff[s] = j;
        if (!((smask >> s) & 1u)) continue;
        const long long base = (static_cast<long long>(s) * Ea + (p.a_e1 ? 0 : e)) * R;
        for (int r = 0; r < p.slots.ranks[s]; ++r, ++j) arow[j] = (base + r) * H;
      }
      sinfo[1] = j;
    }
    __syncthreads();
    const int nr = sinfo[1];                 // stacked rows of this tile (0: no adapter at all)
    const int nr8 = (nr + 7) & ~7;

    // ---------------- K loop: gather token rows (and adapter rows) chunk by chunk
    auto issue = [&](int kc) {
      uint8_t* st = smem + (kc % kPsStages) * STAGE;
      const uint32_t sx = smem_u32(st);
      const uint32_t sa = sx + kPsTile * 128;
      for (int i = tid; i < np * 8; i += kPsThreads) {
        const int r = i >> 3, c = i & 7;
        cp_async16(sx + sw_off(r, c), p.x + static_cast<size_t>(prow[r]) * H + kc * 64 + c * 8, pol_keep);
      }
      for (int i = tid; i < nr * 8; i += kPsThreads) {
        const int r = i >> 3, c = i & 7;
        cp_async16(sa + sw_off(r, c), p.A + arow[r] + kc * 64 + c * 8, pol_normal);
      }
    };
    // warp w: m-tile (w & 3) of 16 pairs, n8 tiles [(w >> 2) * NT8, +NT8) of the stacked rows
    const int mt = warp & 3, nb = (warp >> 2) * NT8;
    float acc[NT8][4];
#pragma unroll
    for (int j = 0; j < NT8; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[j][i] = 0.0f;
#pragma unroll
    for (int s = 0; s < kPsStages - 1; ++s) {
      if (s < KCH) issue(s);
      cp_async_commit();
    }
    for (int kc = 0; kc < KCH; ++kc) {
      cp_async_wait<kPsStages - 2>();
      __syncthreads();   // chunk kc is in; every thread is done with chunk kc - 1's stage
      uint8_t* st = smem + (kc % kPsStages) * STAGE;
      // the permuted rows: this chunk of each pair's row, from shared memory
      for (int i = tid; i < np * 8; i += kPsThreads) {
        const int r = i >> 3, c = i & 7;
        const uint4 v = *reinterpret_cast<const uint4*>(st + sw_off(r, c));
        st_global_v4_hint(p.xp + static_cast<size_t>(q0 + r) * H + kc * 64 + c * 8, v, pol_stream);
      }
      if (nr > 0 && mt * 16 < np) {
        const uint32_t sx = smem_u32(st), sa = sx + kPsTile * 128;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t af[4];
          const int ar = mt * 16 + (lane & 15);
          ldsm_x4(sx + sw_off(ar, kk * 2 + (lane >> 4)), af);
#pragma unroll
          for (int j = 0; j < NT8; ++j) {
            const int n0 = (nb + j) * 8;
            if (n0 < nr8) {   // warp-uniform
              uint32_t bfr[2];
              const int br = n0 + (lane & 7);
              ldsm_x2(sa + sw_off(br, kk * 2 + ((lane >> 3) & 1)), bfr);
              mma_16816(acc[j], af, bfr);
            }
          }
        }
      }
      if (kc + kPsStages - 1 < KCH) issue(kc + kPsStages - 1);
      cp_async_commit();
    }
    cp_async_wait<0>();
    __syncthreads();   // every stage is free: reuse the first as u [64][nr8] fp32

    // ---------------- ub rows: the pair's own slot gets bf16(scaling * u), every other zero
    float* u_s = reinterpret_cast<float*>(smem);
    const int g = lane >> 2, c4 = lane & 3;
    if (nr > 0 && mt * 16 < np) {
#pragma unroll
      for (int j = 0; j < NT8; ++j) {
        const int n0 = (nb + j) * 8 + 2 * c4;
        if ((nb + j) * 8 < nr8) {
          const int r0 = mt * 16 + g;
          u_s[r0 * nr8 + n0] = acc[j][0];
          u_s[r0 * nr8 + n0 + 1] = acc[j][1];
          u_s[(r0 + 8) * nr8 + n0] = acc[j][2];
          u_s[(r0 + 8) * nr8 + n0 + 1] = acc[j][3];
        }
      }
    }
    __syncthreads();
    const int RU8 = p.RU >> 3;   // 16-byte pieces per ub row
    const int nzw = p.slots.S * np * RU8;
    for (int i = tid; i < nzw; i += kPsThreads) {
      const int s = i / (np * RU8);
      const int rem = i - s * np * RU8;
      const int n = rem / RU8, r0 = (rem - n * RU8) * 8;
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = 0.0f;
      if (pslot[n] == s) {
        const float sc = p.slots.scal[s];
        const int rank = p.slots.ranks[s];
        const float* ur = u_s + n * nr8 + soff[s];   // s is an active slot below kMaxFusedSlots
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (r0 + u < rank) v[u] = sc * ur[r0 + u];
      }
      *reinterpret_cast<uint4*>(p.ub + (static_cast<size_t>(s) * p.P + q0 + n) * p.RU + r0) = pack8(v);
    }
    __syncthreads();   // u_s and the pair info are rewritten by the next tile
  }
}

cudaError_t launch_permute_shrink(const PermuteShrinkParams& p, int grid, cudaStream_t stream, bool pdl) {
  if (p.P == 0) return cudaSuccess;
  if (p.H % 64 != 0 || p.RU % 8 != 0 || p.nr_max % 8 != 0 || p.nr_max > kPsMaxRows || p.slots.S > kMaxFusedSlots)
    return cudaErrorInvalidValue;
  const int smem = static_cast<int>(permute_shrink_smem_bytes(p.nr_max, p.E));
  const int n8 = p.nr_max / 8;   // two warps share an m-tile: each covers half the n8 tiles
  const bool deep = permute_shrink_stages(p.nr_max) == 8;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    return launch_k(kern, dim3(grid), dim3(kPsThreads), static_cast<size_t>(smem), stream, pdl, p);
  };
  if (n8 <= 2) return deep ? go(permute_shrink_kernel<1, 8>) : go(permute_shrink_kernel<1, 4>);
  if (n8 <= 4) return deep ? go(permute_shrink_kernel<2, 8>) : go(permute_shrink_kernel<2, 4>);
  if (n8 <= 8) return deep ? go(permute_shrink_kernel<4, 8>) : go(permute_shrink_kernel<4, 4>);
  if (n8 <= 16) return deep ? go(permute_shrink_kernel<8, 8>) : go(permute_shrink_kernel<8, 4>);
  return deep ? go(permute_shrink_kernel<16, 8>) : go(permute_shrink_kernel<16, 4>);
}

}  // namespace mlk
