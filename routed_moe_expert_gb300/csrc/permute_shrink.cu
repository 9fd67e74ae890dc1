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
// kept in shared memory long enough for the tensor cores to multiply it by the adapter rows.
//
// A CTA tile is up to 64 consecutive permuted pairs of one expert, taken in chunks of CW
// columns.  Warp w moves the tile's rows 8w..8w+7: each lane loads the same 16-byte pieces
// of those rows in every chunk into registers (two chunks in flight: the next chunk's loads
// while the current one is stored), then stores them to xp and into one of two shared-memory
// chunk buffers, laid out as 64-column panels with the 128-byte swizzle (the K-major operand
// layout of tcgen05.mma).  The adapter rows of every slot present in the tile are stacked
// into the same buffer as NB (16 or 32) more rows per panel.  One thread then issues the
// chunk's tcgen05.mma (M = 128: the tile's 64 pairs and 64 rows that are never read back,
// N = NB, K = CW) into a TMEM accumulator and commits it to the buffer's mbarrier; the
// copying warps go on with the next chunk and only wait for that mbarrier before they refill
// the same buffer two chunks later.  At the end of the tile two warps read the 64 pair rows
// of the accumulator.
#include "common.cuh"
#include "kernels.h"

namespace mlk {

constexpr int kPsThreads = 256;
constexpr int kPsTile = 64;         // pairs per tile
constexpr int kPsPanel = 64 * 128;  // one 64-column panel of the tile's token rows (bytes)
constexpr uint32_t kPsTmemCols = 32;

MLDEV uint4 ld_global_nc_v4_hint(const void* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

// Stacked adapter rows of the MMA's N: 16 or 32.
static int ps_nb(int nr_max) { return nr_max <= 16 ? 16 : 32; }
// Chunk width: 256 columns when H allows, else 128 or 64.
static int ps_chunk(int H) { return H % 256 == 0 ? 256 : H % 128 == 0 ? 128 : 64; }
// One chunk buffer: CW/64 token-row panels, then CW/64 adapter-row panels of NB rows.
static int ps_buf_bytes(int cw, int nb) { return (cw / 64) * (kPsPanel + nb * 128); }

size_t permute_shrink_smem_bytes(int nr_max, int E, int H) {
  const int nb = ps_nb(nr_max);
  // 1024 for the alignment of the buffers, two buffers, 8 KB read past the last token-row
  // panel by the M = 128 MMAs (rows 64..127, never read back), then the tile's bookkeeping
  return 1024 + 2 * static_cast<size_t>(ps_buf_bytes(ps_chunk(H), nb)) + kPsPanel + 2 * 8 + 16 +
         kPsTile * nb * 4 + 2 * kPsTile * 4 + nb * 8 + 4 * (4 + kMaxFusedSlots) + 8 * (static_cast<size_t>(E) + 1);
}

// CW: chunk width (columns); NB: stacked adapter rows (the MMA's N).
template <int CW, int NB>
__global__ void __launch_bounds__(kPsThreads, 2) permute_shrink_kernel(const PermuteShrinkParams p) {
  constexpr int kPieces = CW / 8;                    // 16-byte pieces per row of a chunk
  constexpr int kPerRow = kPieces >= 32 ? kPieces / 32 : 1;   // pieces of one row per lane
  constexpr int kLanesPerRow = kPieces / kPerRow;    // lanes sharing one row
  constexpr int kRowsPerStep = 32 / kLanesPerRow;    // rows the warp covers in one step
  constexpr int kSteps = 8 / kRowsPerStep;           // steps over the warp's 8 rows
  constexpr int kXPer = kSteps * kPerRow;            // token-row pieces per lane and chunk
  constexpr int kAPer = (NB * kPieces + kPsThreads - 1) / kPsThreads;   // adapter pieces per thread
  constexpr int kPanels = CW / 64;
  constexpr int kABase = kPanels * kPsPanel;         // adapter panels after the token-row panels
  constexpr int kBuf = kPanels * (kPsPanel + NB * 128);
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, NB);
  extern __shared__ __align__(1024) uint8_t ps_smem[];
  uint8_t* smem = ps_smem + ((1024u - (smem_u32(ps_smem) & 1023u)) & 1023u);
  uint64_t* mma_done = reinterpret_cast<uint64_t*>(smem + 2 * kBuf + kPsPanel);   // [2] per buffer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* u_s = reinterpret_cast<float*>(tmem_slot + 4);            // [64][NB] the tile's shrink, fp32
  int* prow = reinterpret_cast<int*>(u_s + kPsTile * NB);          // [64] source token row
  int* pslot = prow + kPsTile;                                     // [64] active slot or -1
  long long* arow = reinterpret_cast<long long*>(pslot + kPsTile);   // [NB] A row element offsets, -1 = padding
  int* sinfo = reinterpret_cast<int*>(arow + NB);                  // [4]: slot mask, rows
  int* soff = sinfo + 4;                                           // [8] first stacked row per slot
  int* tile_start = soff + kMaxFusedSlots;                         // [E+1]
  int* seg = tile_start + (p.E + 1);                               // [E+1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E, H = p.H, KCH = p.H / CW;
  const int R = p.slots.R;
  const int Ea = p.a_e1 ? 1 : E;
  const int lr = lane / kLanesPerRow, lc = lane % kLanesPerRow;   // row within a step, first piece

  if (tid == 0) {
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kPsTmemCols);
    tmem_relinquish();
  }
  // The hidden rows are read k times (once per pair of the token): keep them in L2.  The
  // permuted rows are written once here and read next by the gate_up GEMM from HBM anyway:
  // stream them, so they do not push the hidden rows out of L2.
  const uint64_t pol_keep = l2_policy_evict_last();
  const uint64_t pol_stream = l2_policy_evict_first();
  pdl_wait();    // the routing (perm, offsets) comes from the previous kernel
  pdl_trigger();
  // the ready flags of the shrink tiles of the GEMMs that follow start at zero
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.zero_n; i += gridDim.x * blockDim.x) p.zero_out[i] = 0;
  if (warp == 1) build_tile_schedule(p.offsets, E, kPsTile, 1, seg, tile_start);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = tile_start[E];
  const uint32_t smem0 = smem_u32(smem);
  uint32_t cc = 0;   // chunks issued by this CTA so far: buffer cc & 1, its use cc >> 1

  for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
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
        for (int r = 0; r < p.slots.ranks[s] && j < NB; ++r, ++j) arow[j] = (base + r) * H;
      }
      for (int r = j; r < NB; ++r) arow[r] = -1;   // padding rows: zeros in shared memory
      sinfo[1] = j;
    }
    __syncthreads();
    const int nr = sinfo[1];                 // stacked rows of this tile (0: no adapter at all)

    // this lane's token rows (one per step) and their 16-byte pieces lc + kLanesPerRow * u
    int trow[kSteps];
#pragma unroll
    for (int st = 0; st < kSteps; ++st) trow[st] = prow[8 * warp + st * kRowsPerStep + lr];
    __nv_bfloat16* drow = p.xp + static_cast<size_t>(q0 + 8 * warp + lr) * H + lc * 8;

    // Two register sets: chunk kc + 1 is in flight while chunk kc is stored, and a set is
    // refilled (chunk kc + 2) as soon as its chunk is in shared memory.
    uint4 xa[kXPer], aa[kAPer], xb[kXPer], ab[kAPer];
    // this thread's adapter-row pieces: stacked row pi / kPieces, piece pi % kPieces (padding
    // rows load as zeros)
    auto load_chunk = [&](uint4 (&xv)[kXPer], uint4 (&av)[kAPer], int kc) {
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
        if (r < NB && nr > 0) {
          const long long off = arow[r];
          if (off >= 0) av[i] = ld_global_nc_v4_hint(p.A + off + (pi % kPieces) * 8 + kc * CW, pol_keep);
        }
      }
    };
    // byte offset of piece c (0 <= c < kPieces) of row r in a region of 64-column panels
    auto panel_off = [](int r, int c, int panel_bytes) -> uint32_t {
      return static_cast<uint32_t>((c >> 3) * panel_bytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    };
    bool ok = true;
    auto step = [&](uint4 (&xv)[kXPer], uint4 (&av)[kAPer], int kc) {
      const uint32_t buf = cc & 1u;
      uint8_t* bp = smem + buf * kBuf;
      // the buffer's previous chunk (two chunks ago) has been multiplied
      if (cc >= 2 && !mbar_wait(&mma_done[buf], ((cc >> 1) - 1) & 1u, abort_flag, p.status, kWhereLoraShrinkGu))
        ok = false;
      // the chunk's rows: out to the permuted copy and into the buffer
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
          *reinterpret_cast<uint4*>(bp + panel_off(r, c, kPsPanel)) = v;
        }
      }
#pragma unroll
      for (int i = 0; i < kAPer; ++i) {
        const int pi = tid + kPsThreads * i;
        const int r = pi / kPieces, c = pi % kPieces;
        if (r < NB) *reinterpret_cast<uint4*>(bp + kABase + panel_off(r, c, NB * 128)) = av[i];
      }
      fence_proxy_async_smem();   // the generic-proxy stores above are read by tcgen05.mma
      __syncthreads();            // chunk kc is in the buffer
      if (kc + 2 < KCH) load_chunk(xv, av, kc + 2);   // this set's next chunk
      if (tid == 0) {
        if (nr > 0) {
          tc_fence_after();
          const uint32_t xb0 = smem0 + buf * kBuf, ab0 = xb0 + kABase;
#pragma unroll
          for (int kk = 0; kk < CW / 16; ++kk) {
            const uint64_t ad = sw128_kmajor_desc(xb0 + (kk >> 2) * kPsPanel) + 2 * (kk & 3);
            const uint64_t bd = sw128_kmajor_desc(ab0 + (kk >> 2) * NB * 128) + 2 * (kk & 3);
            umma_bf16(tmem, ad, bd, kIdesc, (kc | kk) != 0 ? 1u : 0u);
          }
        }
        umma_commit(&mma_done[buf]);   // (with no MMA issued since the last commit it completes at once)
      }
      ++cc;
    };
    load_chunk(xa, aa, 0);
    if (KCH > 1) load_chunk(xb, ab, 1);
    for (int kc = 0; kc < KCH; kc += 2) {
      step(xa, aa, kc);
      if (kc + 1 < KCH) step(xb, ab, kc + 1);
    }

    // ---------------- the tile's shrink: wait for its last chunk's MMAs, read the 64 pair rows
    if (!mbar_wait(&mma_done[(cc - 1) & 1u], ((cc - 1) >> 1) & 1u, abort_flag, p.status, kWhereLoraShrinkGu))
      ok = false;
    tc_fence_after();
    __syncwarp();   // the waits above end per thread; tcgen05.ld is .aligned
    if (warp < 2 && nr > 0) {   // TMEM lanes 0..63 = the tile's pairs
      uint32_t v[16];
#pragma unroll
      for (int c0 = 0; c0 < NB; c0 += 16) {
        tmem_ld_x16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) u_s[(warp * 32 + lane) * NB + c0 + i] = __uint_as_float(v[i]);
      }
    }
    tc_fence_before();
    __syncthreads();   // u_s is complete; the accumulator may be overwritten by the next tile

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
        const float* ur = u_s + n * NB + soff[s];   // s is an active slot below kMaxFusedSlots
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (r0 + u < rank) v[u] = sc * ur[r0 + u];
      }
      *reinterpret_cast<uint4*>(p.ub + (static_cast<size_t>(s) * p.P + q0 + n) * p.RU + r0) = pack8(v);
    }
    __syncthreads();   // u_s and the pair info are rewritten by the next tile
    if (!ok) break;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(*tmem_slot, kPsTmemCols);
  }
}

cudaError_t launch_permute_shrink(const PermuteShrinkParams& p, int grid, cudaStream_t stream, bool pdl) {
  if (p.P == 0) return cudaSuccess;
  if (p.H % 64 != 0 || p.RU % 8 != 0 || p.nr_max % 8 != 0 || p.nr_max <= 0 || p.nr_max > kPermuteShrinkMaxRows ||
      p.slots.S > kMaxFusedSlots)
    return cudaErrorInvalidValue;
  const int smem = static_cast<int>(permute_shrink_smem_bytes(p.nr_max, p.E, p.H));
  const int nb = ps_nb(p.nr_max);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    return launch_k(kern, dim3(grid), dim3(kPsThreads), static_cast<size_t>(smem), stream, pdl, p);
  };
  switch (ps_chunk(p.H)) {
    case 256: return nb == 16 ? go(permute_shrink_kernel<256, 16>) : go(permute_shrink_kernel<256, 32>);
    case 128: return nb == 16 ? go(permute_shrink_kernel<128, 16>) : go(permute_shrink_kernel<128, 32>);
    default: return nb == 16 ? go(permute_shrink_kernel<64, 16>) : go(permute_shrink_kernel<64, 32>);
  }
}

}  // namespace mlk
