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
// GEMM.  Both read the same token rows, so one pass does both: each hidden row is read once
// per pair (from L2: every token is read by k pairs), written out as the permuted row and
// kept in shared memory long enough to be multiplied by the adapter rows.
//
// A CTA tile is up to 64 consecutive permuted pairs of one expert, taken in chunks of CW
// columns.  Warp w moves the tile's rows 8w..8w+7: each lane loads the same 16-byte pieces
// of those rows in every chunk into registers (the next chunk's loads are in flight while
// the tensor cores work on the current one), then stores them to xp and to shared memory,
// in rows of CW*2 bytes with the 16-byte piece index XORed with the row index so ldmatrix
// reads them without bank conflicts.  A piece costs one load, one global store and one
// shared store; its addresses move by a constant from chunk to chunk.  The adapter rows of
// every slot present in the tile are stacked as the N side of mma.sync m16n8k16 (M = the
// pairs); the eight warps split each chunk as four 16-pair m-tiles by two halves of its
// k-steps, and the two halves' sums are added in a fixed order at the end of the tile.
#include "common.cuh"
#include "kernels.h"

namespace mlk {

constexpr int kPsThreads = 256;
constexpr int kPsTile = 64;   // pairs per tile

MLDEV uint4 ld_global_nc_v4_hint(const void* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}
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

// Stacked adapter rows a tile holds: 8, 16 or 32 (the kernel's n8 tiles times 8).
static int ps_rows8(int nr_max) { return nr_max <= 8 ? 8 : nr_max <= 16 ? 16 : 32; }
// Chunk width: the widest of 512, 256, 128, 64 columns that divides H; 512-wide chunks (16
// pieces in flight per lane) only up to 16 stacked rows, where the registers still hold them.
static int ps_chunk(int H, int rows8) {
  return (H % 512 == 0 && rows8 <= 16) ? 512 : H % 256 == 0 ? 256 : H % 128 == 0 ? 128 : 64;
}

size_t permute_shrink_smem_bytes(int nr_max, int E, int H) {
  const int rows8 = ps_rows8(nr_max);
  return 128 + static_cast<size_t>(kPsTile + rows8) * ps_chunk(H, rows8) * 2 + kPsTile * 16 * 4 + 2 * kPsTile * 4 +
         rows8 * 8 + 4 * (4 + kMaxFusedSlots) + 8 * (static_cast<size_t>(E) + 1);
}

// CW: chunk width (columns); NT8: n8 tiles of stacked adapter rows.
template <int CW, int NT8>
__global__ void __launch_bounds__(kPsThreads, 2) permute_shrink_kernel(const PermuteShrinkParams p) {
  constexpr int kRowBytes = CW * 2;                  // one row of a chunk in shared memory
  constexpr int kPieces = CW / 8;                    // 16-byte pieces per row of a chunk
  constexpr int kPerRow = kPieces >= 32 ? kPieces / 32 : 1;   // pieces of one row per lane
  constexpr int kLanesPerRow = kPieces / kPerRow;    // lanes sharing one row
  constexpr int kRowsPerStep = 32 / kLanesPerRow;    // rows the warp covers in one step
  constexpr int kSteps = 8 / kRowsPerStep;           // steps over the warp's 8 rows
  constexpr int kXPer = kSteps * kPerRow;            // token-row pieces per lane and chunk
  constexpr int kRows8 = NT8 * 8;                    // stacked adapter rows in shared memory
  constexpr int kAPer = (kRows8 * kPieces + kPsThreads - 1) / kPsThreads;   // adapter pieces per thread
  constexpr int kHalfSteps = CW / 32;                // k-steps of 16 per half chunk
  extern __shared__ __align__(128) uint8_t ps_smem[];
  uint8_t* smem = ps_smem + ((128u - (smem_u32(ps_smem) & 127u)) & 127u);
  float* part = reinterpret_cast<float*>(smem + (kPsTile + kRows8) * kRowBytes);   // [64][16] k-half 1 sums
  int* prow = reinterpret_cast<int*>(part + kPsTile * 16);         // [64] source token row
  int* pslot = prow + kPsTile;                                     // [64] active slot or -1
  long long* arow = reinterpret_cast<long long*>(pslot + kPsTile);   // [kRows8] A row element offsets, -1 = padding
  int* sinfo = reinterpret_cast<int*>(arow + kRows8);              // [4]: slot mask, rows
  int* soff = sinfo + 4;                                           // [8] first stacked row per slot
  int* tile_start = soff + kMaxFusedSlots;                         // [E+1]
  int* seg = tile_start + (p.E + 1);                               // [E+1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E, H = p.H, KCH = p.H / CW;
  const int R = p.slots.R;
  const int Ea = p.a_e1 ? 1 : E;
  const int lr = lane / kLanesPerRow, lc = lane % kLanesPerRow;   // row within a step, first piece

  // The hidden rows are read k times (once per pair of the token): keep them in L2.  The
  // permuted rows are written once here and read next by the gate_up GEMM from HBM anyway:
  // stream them, so they do not push the hidden rows out of L2.
  const uint64_t pol_keep = l2_policy_evict_last();
  const uint64_t pol_stream = l2_policy_evict_first();
  pdl_wait();    // the routing (perm, offsets) comes from the previous kernel
  pdl_trigger();
  if (warp == 0) build_tile_schedule(p.offsets, E, kPsTile, 1, seg, tile_start);
  __syncthreads();
  const int total = tile_start[E];
  const int mt = warp & 3, kh = warp >> 2;   // the warp's m-tile and k-half of every chunk
  const uint32_t xs_u = smem_u32(smem), as_u = xs_u + kPsTile * kRowBytes;

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
      prow[tid] = t;   // rows past np read token 0's row: loaded, never stored
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
        for (int r = 0; r < p.slots.ranks[s] && j < kRows8; ++r, ++j) arow[j] = (base + r) * H;
      }
      for (int r = j; r < kRows8; ++r) arow[r] = -1;   // padding rows: zeros in shared memory
      sinfo[1] = j;
    }
    __syncthreads();
    const int nr = sinfo[1];                 // stacked rows of this tile (0: no adapter at all)
    const int nr8 = (nr + 7) & ~7;

    // this lane's token rows (one per step) and their 16-byte pieces lc + kLanesPerRow * u
    int trow[kSteps];
#pragma unroll
    for (int st = 0; st < kSteps; ++st) trow[st] = prow[8 * warp + st * kRowsPerStep + lr];
    __nv_bfloat16* drow = p.xp + static_cast<size_t>(q0 + 8 * warp + lr) * H + lc * 8;

    float acc[NT8][4];
#pragma unroll
    for (int j = 0; j < NT8; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[j][i] = 0.0f;

    uint4 xv[kXPer], av[kAPer];
    // this thread's adapter-row pieces: stacked row pi / kPieces, piece pi % kPieces (rows
    // past the stack are not loaded, padding rows load as zeros)
    auto load_chunk = [&](int kc) {
#pragma unroll
      for (int st = 0; st < kSteps; ++st)
#pragma unroll
        for (int u = 0; u < kPerRow; ++u)
          xv[st * kPerRow + u] = ld_global_nc_v4_hint(
              p.x + static_cast<size_t>(trow[st]) * H + (lc * 8 + kc * CW + u * kLanesPerRow * 8), pol_keep);
#pragma unroll
      for (int i = 0; i < kAPer; ++i) {
        const int pi = tid + kPsThreads * i;
        const int r = pi / kPieces;
        av[i] = make_uint4(0u, 0u, 0u, 0u);
        if (r < kRows8) {
          const long long off = arow[r];
          if (off >= 0) av[i] = ld_global_nc_v4_hint(p.A + off + (pi % kPieces) * 8 + kc * CW, pol_keep);
        }
      }
    };
    load_chunk(0);
    for (int kc = 0; kc < KCH; ++kc) {
      // the chunk's rows: out to the permuted copy and into shared memory
#pragma unroll
      for (int st = 0; st < kSteps; ++st) {
        const int r = 8 * warp + st * kRowsPerStep + lr;
#pragma unroll
        for (int u = 0; u < kPerRow; ++u) {
          const int c = lc + u * kLanesPerRow;
          const uint4 v = xv[st * kPerRow + u];
          if (r < np)
            st_global_v4_hint(drow + static_cast<size_t>(st * kRowsPerStep) * H + kc * CW + u * kLanesPerRow * 8, v,
                              pol_stream);
          *reinterpret_cast<uint4*>(smem + r * kRowBytes + ((c ^ (r & 7)) << 4)) = v;
        }
      }
#pragma unroll
      for (int i = 0; i < kAPer; ++i) {
        const int pi = tid + kPsThreads * i;
        const int r = pi / kPieces, c = pi % kPieces;
        if (r < kRows8) *reinterpret_cast<uint4*>(smem + (kPsTile + r) * kRowBytes + ((c ^ (r & 7)) << 4)) = av[i];
      }
      __syncthreads();   // chunk kc is in shared memory
      if (kc + 1 < KCH) load_chunk(kc + 1);   // in flight during the MMAs
      __syncwarp();   // the loads above branch per thread; ldmatrix and mma.sync are .aligned
      if (nr > 0 && mt * 16 < np) {
        const int ar = mt * 16 + (lane & 15);
#pragma unroll
        for (int k2 = 0; k2 < kHalfSteps; ++k2) {
          const int kk = kh * kHalfSteps + k2;
          uint32_t af[4];
          ldsm_x4(xs_u + ar * kRowBytes + (((kk * 2 + (lane >> 4)) ^ (ar & 7)) << 4), af);
#pragma unroll
          for (int j = 0; j < NT8; ++j) {
            if (j * 8 < nr8) {   // warp-uniform
              uint32_t bfr[2];
              const int br = j * 8 + (lane & 7);
              ldsm_x2(as_u + br * kRowBytes + (((kk * 2 + ((lane >> 3) & 1)) ^ (br & 7)) << 4), bfr);
              mma_16816(acc[j], af, bfr);
            }
          }
        }
      }
      __syncthreads();   // every warp is done with chunk kc's shared memory
    }

    // ---------------- k-half 1 parks its sums, k-half 0 adds them (a fixed order), 16 columns at a time
    float* u_s = reinterpret_cast<float*>(smem);   // [64][nr8] fp32 (the chunk buffer is free)
    const int g = lane >> 2, c4 = lane & 3;
    const bool mm = nr > 0 && mt * 16 < np;
#pragma unroll
    for (int j0 = 0; j0 < NT8; j0 += 2) {
      if (mm && kh == 1) {
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          if (j0 + jj < NT8) {
            const int r0 = mt * 16 + g, n0 = jj * 8 + 2 * c4;
            part[r0 * 16 + n0] = acc[j0 + jj][0];
            part[r0 * 16 + n0 + 1] = acc[j0 + jj][1];
            part[(r0 + 8) * 16 + n0] = acc[j0 + jj][2];
            part[(r0 + 8) * 16 + n0 + 1] = acc[j0 + jj][3];
          }
        }
      }
      __syncthreads();
      if (mm && kh == 0) {
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          if (j0 + jj < NT8 && (j0 + jj) * 8 < nr8) {
            const int r0 = mt * 16 + g, n0 = jj * 8 + 2 * c4, col = (j0 + jj) * 8 + 2 * c4;
            u_s[r0 * nr8 + col] = acc[j0 + jj][0] + part[r0 * 16 + n0];
            u_s[r0 * nr8 + col + 1] = acc[j0 + jj][1] + part[r0 * 16 + n0 + 1];
            u_s[(r0 + 8) * nr8 + col] = acc[j0 + jj][2] + part[(r0 + 8) * 16 + n0];
            u_s[(r0 + 8) * nr8 + col + 1] = acc[j0 + jj][3] + part[(r0 + 8) * 16 + n0 + 1];
          }
        }
      }
      __syncthreads();
    }

    // ---------------- ub rows: the pair's own slot gets bf16(scaling * u), every other zero
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
  if (p.H % 64 != 0 || p.RU % 8 != 0 || p.nr_max % 8 != 0 || p.nr_max <= 0 || p.nr_max > kPermuteShrinkMaxRows ||
      p.slots.S > kMaxFusedSlots)
    return cudaErrorInvalidValue;
  const int smem = static_cast<int>(permute_shrink_smem_bytes(p.nr_max, p.E, p.H));
  const int rows8 = ps_rows8(p.nr_max);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    return launch_k(kern, dim3(grid), dim3(kPsThreads), static_cast<size_t>(smem), stream, pdl, p);
  };
  auto by_rows = [&](auto cw) -> cudaError_t {
    constexpr int C = decltype(cw)::value;
    if (rows8 == 8) return go(permute_shrink_kernel<C, 1>);
    if (rows8 == 16) return go(permute_shrink_kernel<C, 2>);
    return go(permute_shrink_kernel<C, 4>);
  };
  switch (ps_chunk(p.H, rows8)) {
    case 512:   // (rows8 <= 16 here)
      return rows8 == 8 ? go(permute_shrink_kernel<512, 1>) : go(permute_shrink_kernel<512, 2>);
    case 256: return by_rows(std::integral_constant<int, 256>());
    case 128: return by_rows(std::integral_constant<int, 128>());
    default: return by_rows(std::integral_constant<int, 64>());
  }
}

}  // namespace mlk
