// LoRA shrink on the 5th-generation tensor cores, all slots at once.
//
//   u[q, s, r] = sum_k X[q, k] * A[s, e, r, k]        (pair q of expert e, fp32 in TMEM)
//   ub[s, q, r] = bf16( scaling[s] * u[q, s, r] )  for s = the slot of q's token and r < ranks[s]
//   ub[s', q, r] = 0                               for every other slot s' (and r >= ranks[s])
//   pair_slot[q] = s, or -1 when q's token has no active adapter
// or, with ub_stacked, the same values in one row per pair: ub[q, coff[s] + r], the columns
// [coff[s], coff[s+1]) holding slot s's ranks padded with zeros to a multiple of 16 (the
// column layout of the expand-ready LoRA B, so one K-stage of the GEMM covers every slot).
//
// This is the shrink (A) half of the per-expert LoRA of sglang PR #28466 (section 1,
// merged_experts_fused_moe_lora_add) for the gate_up chain (X = permuted hidden) and the
// down chain (X = activation).  Its output feeds the expand (B) half, which runs inside the
// grouped GEMMs as extra K-stages.  The tile is up to TB pairs of one expert (TB rows of X by
// TMA, TB in {16..128} from the mean pairs per expert; the MMA runs at M = 128 and the rows
// past TB are never read back) by N = every slot's rank rows of A for that expert, stacked
// (N <= 256), so one pass over K serves all slots present.  When every active rank is a
// multiple of 8, each slot's block is loaded with its own tensor map whose box is exactly
// its rank rows, packed one after another (each at a 1024-byte swizzle-atom boundary), so
// the padding rows of a stacked adapter are never fetched; otherwise all R rows of every
// slot are loaded and the tails only produce accumulator columns that are never read.
// Warp roles as in the grouped GEMM: TMA producer, MMA issuer + TMEM owner, 4 epilogue
// warps; bounded waits throughout.
#include "common.cuh"
#include "kernels.h"

namespace mlk {

constexpr int kShrinkThreads = 192;
constexpr int kShrinkMaxStages = 12;


static int shrink_stages(int nb) {   // as many 16 KB + N*128 B stages as fit in ~200 KB
  const int s = (200 * 1024) / (16384 + nb * 128);
  return s < kShrinkMaxStages ? s : kShrinkMaxStages;
}

int lora_shrink_tc_smem(int nb, int E) {
  const int st = shrink_stages(nb);
  return 1024 + st * (16384 + nb * 128) + (2 * st + 5) * 8 + 16 + 8 * (E + 1) + 16;
}

template <int NB>
__global__ void __launch_bounds__(kShrinkThreads, 1) lora_shrink_tc_kernel(const __grid_constant__ ShrinkTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  constexpr uint32_t A_BYTES = 16384;
  constexpr uint32_t STAGE = A_BYTES + NB * 128;
  constexpr uint32_t TMEM_COLS = (2 * NB <= 32) ? 32 : (2 * NB <= 64 ? 64 : (2 * NB <= 128 ? 128 : (2 * NB <= 256 ? 256 : 512)));
  const int S = p.stages;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* tile_start = reinterpret_cast<int*>(tmem_slot + 4);
  int* seg = tile_start + (p.E + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int KB = p.K >> 6;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 128);
    mbar_init(&tempty[1], 128);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmap_x);
    if (p.per_slot && !p.packed_a) {
      for (int s = 0; s < p.S; ++s)
        if (p.row_off[s + 1] > p.row_off[s]) tma_prefetch_desc(&p.tmap_a_slot[s]);
    } else {
      tma_prefetch_desc(&p.tmap_a);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) build_tile_schedule(p.offsets, E, p.tb, 1, seg, tile_start);   // tiles of TB pairs per expert
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();   // the rows to shrink come from the previous kernel (expert offsets from earlier)
  pdl_trigger();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tile_start[E];
  const int nrows = p.per_slot ? p.row_off[p.S] : p.S * p.R;   // stacked B rows actually loaded
  auto decode = [&](int tile, int& e, int& qt) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    e = lo;
    qt = tile - tile_start[e];
  };

  if (warp == 0) {
    if (lane == 0) {   // ---------------------------------------------- TMA producer
      const uint64_t pol_x = l2_policy_evict_first();
      const uint64_t pol_a = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int e, qt;
        decode(tile, e, qt);
        const int xr = seg[e] + qt * p.tb;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, kWhereLoraShrinkTc)) {
            ok = false;
            break;
          }
          uint8_t* a = smem + stage * STAGE;
          // bytes actually copied: TB rows of X and nrows rows of A (rows TB..127 of the A
          // tile and nrows..NB-1 of the B tile keep stale data; they only feed accumulator
          // lanes and columns that are never read)
          mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(p.tb + nrows) * 128u);
          tma_load_2d(a, &p.tmap_x, &full[stage], kb * 64, xr, pol_x);
          if (p.packed_a) {   // every slot's rank rows for expert e, contiguous in the shrink-ready A
            tma_load_2d(a + A_BYTES, &p.tmap_a, &full[stage], kb * 64, (p.a_e1 ? 0 : e) * nrows, pol_a);
          } else if (p.per_slot) {   // each active slot's rank rows of A for expert e, packed
            for (int s = 0; s < p.S; ++s)
              if (p.row_off[s + 1] > p.row_off[s])
                tma_load_2d(a + A_BYTES + p.row_off[s] * 128, &p.tmap_a_slot[s], &full[stage], kb * 64,
                            (s * (p.a_e1 ? 1 : E) + (p.a_e1 ? 0 : e)) * p.R, pol_a);
          } else {            // each slot's R rows of A for expert e, stacked
            for (int s = 0; s < p.S; ++s)
              tma_load_2d(a + A_BYTES + s * p.R * 128, &p.tmap_a, &full[stage], kb * 64, (s * (p.a_e1 ? 1 : E) + (p.a_e1 ? 0 : e)) * p.R, pol_a);
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok)
        for (int s = 0; s < S; ++s)
          if ((issued_mask >> s) & 1u) mbar_wait_drain(&full[s], (issued_parity >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {   // ---------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(128, NB);
      int stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        if (!mbar_wait(&tempty[acc], aphase ^ 1u, abort_flag, p.status, kWhereLoraShrinkTc)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * NB);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status, kWhereLoraShrinkTc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * STAGE);
          const uint64_t ad = sw128_kmajor_desc(a_addr);
          const uint64_t bd = sw128_kmajor_desc(a_addr + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) umma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          aphase ^= 1u;
        }
      }
    }
  } else {   // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // pair row of the tile == TMEM lane
    int acc = 0;
    uint32_t aphase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int e, qt;
      decode(tile, e, qt);
      const int q = seg[e] + qt * p.tb + row;
      const bool valid = row < p.tb && q < seg[e + 1];
      int sl = -1;
      if (valid) {
        sl = p.slot_idx[p.perm[q] / p.k];
        if (sl < -1 || sl >= p.slots.S) {
          record_status(p.status, kDevBadSlot, kWhereLoraShrinkTc);
          sl = -1;
        } else if (sl >= 0 && (p.slots.ranks[sl] <= 0 || p.slots.scal[sl] == 0.0f)) {
          sl = -1;
        }
      }
      if (!mbar_wait(&tfull[acc], aphase, abort_flag, p.status, kWhereLoraShrinkTc)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * NB);
      // Every column (s2, r) of the accumulator goes to ub[s2][q][r]: the scaled value when
      // s2 is this pair's slot and r < its rank, zero otherwise.  Ranks (per_slot) and R are
      // multiples of 8, so each 8 columns lie in one slot row and leave as one 16-byte store;
      // with per_slot the rows past a slot's loaded rows are written as zeros afterwards.
      const float sc = sl >= 0 ? p.slots.scal[sl] : 0.0f;
      const int rank = sl >= 0 ? p.slots.ranks[sl] : 0;
      const int ncol = nrows;
#pragma unroll 1
      for (int c = 0; c < ncol; c += 16) {   // tcgen05.ld is warp-wide: same columns in every lane
        uint32_t v[16];
        __syncwarp();   // after the per-lane wait and stores: tcgen05.ld is .aligned
        tmem_ld_x16(taddr + c, v);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int h8 = 0; h8 < 2; ++h8) {
            const int col0 = c + 8 * h8;
            if (col0 >= ncol) break;
            int s2, r0;
            if (p.per_slot) {
              s2 = 0;
              while (p.row_off[s2 + 1] <= col0) ++s2;
              r0 = col0 - p.row_off[s2];
            } else {
              s2 = col0 / p.R;
              r0 = col0 - s2 * p.R;
            }
            float f[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              f[i] = (s2 == sl && r0 + i < rank) ? sc * __uint_as_float(v[8 * h8 + i]) : 0.0f;
            if (p.ub_stacked) {   // slot s2's columns of the pair's stacked row
              if (r0 < p.coff[s2 + 1] - p.coff[s2])
                *reinterpret_cast<uint4*>(p.ub + static_cast<size_t>(q) * p.rs + p.coff[s2] + r0) = pack8(f);
            } else {
              *reinterpret_cast<uint4*>(p.ub + (static_cast<size_t>(s2) * p.P + q) * p.R + r0) = pack8(f);
            }
          }
        }
      }
      if (valid && p.ub_stacked) {   // the columns no accumulator column covered: zero
        for (int s2 = 0; s2 < p.S; ++s2) {
          const int ru = p.coff[s2 + 1] - p.coff[s2];
          const int z0 = p.per_slot ? p.row_off[s2 + 1] - p.row_off[s2] : min(p.R, ru);
          for (int r0 = z0; r0 < ru; r0 += 8)
            *reinterpret_cast<uint4*>(p.ub + static_cast<size_t>(q) * p.rs + p.coff[s2] + r0) =
                make_uint4(0u, 0u, 0u, 0u);
        }
      } else if (valid && p.per_slot) {
        for (int s2 = 0; s2 < p.S; ++s2)
          for (int r0 = p.row_off[s2 + 1] - p.row_off[s2]; r0 < p.R; r0 += 8)
            *reinterpret_cast<uint4*>(p.ub + (static_cast<size_t>(s2) * p.P + q) * p.R + r0) =
                make_uint4(0u, 0u, 0u, 0u);
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1u;
      }
      if (valid) p.pair_slot[q] = sl;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (*abort_flag) {
      if (lane == 0) {
        umma_commit(drain);
        mbar_wait_drain(drain, 0);
      }
      __syncwarp();
    }
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int NB>
static cudaError_t launch_nb(const ShrinkTcParams& p_in, int grid, cudaStream_t stream, bool pdl) {
  ShrinkTcParams p = p_in;
  p.stages = shrink_stages(NB);
  const int smem = lora_shrink_tc_smem(NB, p.E);
  cudaError_t err =
      cudaFuncSetAttribute(lora_shrink_tc_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  return launch_k(lora_shrink_tc_kernel<NB>, dim3(grid), dim3(kShrinkThreads), smem, stream, pdl, p);
}

int lora_shrink_tc_nb(int rows) {
  const int n = rows;
  return n <= 16 ? 16 : n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : n <= 256 ? 256 : 0;
}

cudaError_t launch_lora_shrink_tc(const ShrinkTcParams& p, int grid, cudaStream_t stream, bool pdl) {
  if (p.P == 0) return cudaSuccess;
  switch (lora_shrink_tc_nb(p.per_slot ? p.row_off[p.S] : p.S * p.R)) {
    case 16: return launch_nb<16>(p, grid, stream, pdl);
    case 32: return launch_nb<32>(p, grid, stream, pdl);
    case 64: return launch_nb<64>(p, grid, stream, pdl);
    case 128: return launch_nb<128>(p, grid, stream, pdl);
    case 256: return launch_nb<256>(p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
  }
}

// Expand-ready copy of a stacked LoRA B [S, Eb, N, R] for the fused LoRA K-stages of the
// grouped GEMM: row (eb * NT + nt) * 128 + r holds the weight row that is row r of 128-row
// tile nt (for the gated gate_up layout: gate row 64 nt + r for r < 64, else up row
// N/2 + 64 nt + r - 64; otherwise row 128 nt + r, zero past N), and its columns stack the
// slots: slot s's ranks[s] values in [coff[s], coff[s] + ranks[s]), zero up to coff[s+1]
// (ranks rounded up to 16).  One thread per 8 output columns (one 16-byte store).
__global__ void pack_lora_b_kernel(const __grid_constant__ PackLoraBParams p) {
  const int cv = p.rs >> 3;
  const long long total = static_cast<long long>(p.Eb) * p.NT * 128 * cv;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long prow = i / cv;
    const int c0 = static_cast<int>(i - prow * cv) * 8;
    const int r = static_cast<int>(prow & 127);
    const long long tn = prow >> 7;
    const int nt = static_cast<int>(tn % p.NT);
    const int eb = static_cast<int>(tn / p.NT);
    const int n = p.gated ? (r < 64 ? 64 * nt + r : (p.N >> 1) + 64 * nt + (r - 64)) : 128 * nt + r;
    int s = 0;
    while (p.coff[s + 1] <= c0) ++s;   // c0 < coff[S], so s < S
    const int rr0 = c0 - p.coff[s];
    const __nv_bfloat16* src = p.B + ((static_cast<size_t>(s) * p.Eb + eb) * p.N + n) * p.R;
    float f[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      f[j] = 0.0f;
      if (n < p.N && rr0 + j < p.ranks[s]) f[j] = bf2f(src[rr0 + j]);   // the rank tail is never read
    }
    *reinterpret_cast<uint4*>(p.Bp + prow * p.rs + c0) = pack8(f);
  }
}

cudaError_t launch_pack_lora_b(const PackLoraBParams& p, cudaStream_t stream) {
  const long long total = static_cast<long long>(p.Eb) * p.NT * 128 * (p.rs >> 3);
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  pack_lora_b_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

// Shrink-ready copy of a stacked LoRA A [S, Ea, R, K] for the tensor-core shrinks: row
// e * RS + aoff[s] + r is A[s, e, r, :] for r < ranks[s] and zero up to aoff[s+1] (ranks
// rounded up to 8), so every slot's rank rows of an expert are one contiguous block of RS
// rows.  One thread per 8 values (one 16-byte store); the rank tails of A are never read.
__global__ void pack_lora_a_kernel(const __grid_constant__ PackLoraAParams p) {
  const int cv = p.K >> 3;
  const long long total = static_cast<long long>(p.Ea) * p.RS * cv;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long prow = i / cv;
    const int c0 = static_cast<int>(i - prow * cv) * 8;
    const int e = static_cast<int>(prow / p.RS);
    const int j = static_cast<int>(prow - static_cast<long long>(e) * p.RS);
    int s = 0;
    while (p.aoff[s + 1] <= j) ++s;   // j < aoff[S], so s < S
    const int r = j - p.aoff[s];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < p.ranks[s])
      v = *reinterpret_cast<const uint4*>(p.A + ((static_cast<size_t>(s) * p.Ea + e) * p.R + r) * p.K + c0);
    *reinterpret_cast<uint4*>(p.Ap + prow * p.K + c0) = v;
  }
}

cudaError_t launch_pack_lora_a(const PackLoraAParams& p, cudaStream_t stream) {
  const long long total = static_cast<long long>(p.Ea) * p.RS * (p.K >> 3);
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  pack_lora_a_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mlk
