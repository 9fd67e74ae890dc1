// Grouped (per-expert) GEMM on the 5th-generation tensor cores: TMA -> shared memory
// -> tcgen05.mma -> TMEM -> registers -> global.
//
// For every expert e and its routed pairs q in [offsets[e], offsets[e+1]):
//     out[q, col] = sum_k X[q, k] * W[e*N + row(col), k]
// which is the gate_up GEMM (W = w1, X = permuted hidden, N = 2I, K = H) and the down
// GEMM (W = w2, X = activation, N = H, K = I) of the routed MoE layer (sglang PR #28466
// "bf16 MoE-LoRA for trtllm backend", Files changed, launcher row: "gate_up as raw
// Gemm2::Runner ... K=hidden, N=2*inter, gated-interleaved out", "down Gemm2::Runner
// (K=inter, N=hidden)").
//
// Orientation: the weights are the MMA "A" operand (M = 128 weight rows per tile) and
// the expert's tokens are "B" (N = BN token columns), so a decode expert with a handful
// of tokens still streams full 128-row weight tiles (BN as small as 16).  The TMEM
// accumulator is [128 lanes = weight rows] x [BN columns = tokens].
//
// Persistent CTAs (one per SM) walk a static round-robin list of tiles (e, n-tile,
// token-tile), token-tile fastest so CTAs that run together share a weight tile in L2.
// Warp roles: warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer, warps 2-5 =
// epilogue (each owns one 32-lane quarter of TMEM).  Two TMEM accumulators let the
// epilogue of one tile overlap the MMAs of the next.
//
// gated = 1 (gate_up): the 128 A rows of n-tile n are the 64 gate rows [64n, 64n+64)
// and the 64 up rows [N/2 + 64n, ...), so each tile holds matching gate/up features; the
// output row is stored "gated-interleaved": column 128n + j is gate feature 64n + j for
// j < 64 and up feature 64n + j - 64 for j >= 64.
//
// gated = 2 (gate_up with the activation fused): the tile rows are laid out as for gated =
// 1, fused LoRA stages go to a second accumulator, and the epilogue rounds g and the LoRA
// delta to bf16 separately (the pages' two bf16 tensors) and adds them; the four epilogue
// warps park these values in shared memory as [feature][token] and then each thread forms
// a = bf16(silu(gate) * up) -- the activation of sglang PR #28466's launcher row -- for 8
// consecutive features of one token and writes them to the [P, N/2] output in one 16-byte
// store.
//
// Every mbarrier wait is bounded (2 s); a timeout records MOE_LORA_ERR_TIMEOUT, raises a
// CTA-wide abort flag, drains the copies already issued and frees TMEM before returning.
#include "common.cuh"
#include "kernels.h"

namespace mlk {

constexpr int kGemmThreads = 192;
constexpr int kAByte = 128 * 128;        // 128 rows x 64 bf16 (one 128-byte swizzle row each)
constexpr int kMaxStages = 16;
constexpr int kTileRing = 32;   // > kMaxStages: the producer runs at most kMaxStages tiles ahead
constexpr int kXchgStride = 17;                       // floats per feature row (padded against bank conflicts)
constexpr int kXchgFloats = 2 * 128 * kXchgStride;    // two buffers of 128 rows (64 gate, 64 up) x 16 tokens
constexpr int kYbufFloats = 4 * 16 * 32;              // per epilogue warp: 16 tokens x 32 features (x2 for fp32)
constexpr uint64_t kPeerDrainNs = 100000;             // 100 us for an aborted odd CTA's copies to land

int gemm_stage_bytes(int rows) { return kAByte + rows * 128; }

int gemm_smem_bytes(int bn, int cg, int stages, int E, int lora_R, int act_fused, int y_tma) {
  // Carve-up, in order (see the kernel): 1 KB alignment slack; stage buffers; full/empty
  // barriers (2*stages), tfull/tempty (4), drain (1), dfull/dfree (2); tmem slot + abort flag
  // (16 B); tile_start and seg (E+1 ints each); the tile slot ring; 4 ints of padding; and, for
  // the CUDA-core LoRA epilogue, BN token slots then BN x RP8 floats aligned to 16 bytes; then,
  // for the plain epilogues, the four warps' 16 x 32 float store buffers (two each when whole
  // chunks leave by TMA, one staged while the previous one is stored).
  const int ring = 4 * (kTileRing + 4);
  const int lora = lora_R > 0 ? bn * 4 + 16 + bn * ((lora_R + 7) / 8 * 8) * 4 : 0;
  const int xchg = act_fused ? kXchgFloats * 4 : 0;   // gate -> up hand-off (fused activation)
  const int ybuf = act_fused ? 0 : (lora_R > 0 ? 0 : bn * 4 + 16) + 128 + (y_tma ? 2 : 1) * kYbufFloats * 4;
  return 1024 + stages * gemm_stage_bytes(bn / cg) + (2 * stages + 7) * 8 + 16 + 8 * (E + 1) + ring +
         (lora > xchg ? lora : xchg) + ybuf;
}

MLDEV void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }   // the 4 epilogue warps

// Fused LoRA expand stages sit after this many of a tile's KB main K-stages (at least one main
// stage goes first, so the main accumulator is initialised by a main MMA).  Placed before the
// end of the main loop, their MMAs (and, at 256-token tiles, the wait for the idle accumulator)
// overlap the tile's remaining main stages instead of following them.
__host__ __device__ constexpr int lora_stage_pos(int KB) { return KB >= 4 ? (3 * KB) / 4 : 1; }
// 64-wide K blocks of slot `rank`'s LoRA stage that hold data (the rest is zero fill), and the
// 16-deep MMA steps of block kb that do.
MLDEV int lora_blocks(int rank, int lora_kb) { return min(lora_kb, (rank + 63) >> 6); }
MLDEV int lora_ksteps(int rank, int kb) { return min(4, (rank - 64 * kb + 15) >> 4); }

// LoRA expand of one 16-token chunk on the CUDA cores, for output feature `feat` (this
// thread's weight row): val[j] += sum_{r < ranks[s]} lora_B[s, e, feat, r] * v_s[c + j][r]
// for each token j of the chunk with slot s = lslot[c + j] >= 0.  Tokens are taken slot by
// slot (the slots are the same in every lane of the warp); v_s rows are staged per tile,
// RP8 = R rounded up to 8 floats each, zero past the slot's rank.
MLDEV void lora_expand_chunk(const GemmParams& p, const int* lslot, const float* v_s, int c, int nvalid, int e,
                             int feat, float (&val)[16]) {
  const int R = p.slots.R;
  const int RP8 = (R + 7) & ~7;
  uint32_t done = 0;
#pragma unroll 1
  for (int j0 = 0; j0 < 16 && c + j0 < nvalid; ++j0) {
    if ((done >> j0) & 1u) continue;
    const int sl = lslot[c + j0];
    uint32_t m = 0;
    for (int j = j0; j < 16 && c + j < nvalid; ++j)
      if (lslot[c + j] == sl) m |= 1u << j;
    done |= m;
    if (sl < 0) continue;
    const int rank = p.slots.ranks[sl];
    const size_t be = p.lora_b_e1 ? static_cast<size_t>(sl) : static_cast<size_t>(sl) * p.E + e;
    const __nv_bfloat16* Brow = p.lora_B + (be * p.N + feat) * static_cast<size_t>(R);
#pragma unroll 1
    for (int r0 = 0; r0 < rank; r0 += 8) {
      float b[8];   // zero past the rank: the stacked tail is never read
      if ((R & 7) == 0 && r0 + 8 <= rank) {
        unpack8(__ldg(reinterpret_cast<const uint4*>(Brow + r0)), b);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = (r0 + i < rank) ? bf2f(Brow[r0 + i]) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if ((m >> j) & 1u) {
          const float4* vj = reinterpret_cast<const float4*>(v_s + (c + j) * RP8 + r0);
          const float4 v0 = vj[0], v1 = vj[1];
          val[j] += b[0] * v0.x + b[1] * v0.y + b[2] * v0.z + b[3] * v0.w + b[4] * v1.x + b[5] * v1.y +
                    b[6] * v1.z + b[7] * v1.w;
        }
      }
    }
  }
}

// Fused LoRA K-stages come either per slot (slot s's rows of B, its own rank as the K extent,
// and its ub rows), or, with a packed B, per 64-column panel of every slot's ranks stacked
// side by side (B rows of the tile from the expand-ready copy, the pairs' stacked ub rows):
// a pair's ub row is zero outside its own slot's columns, so each panel's products of other
// slots add exact zeros, and far fewer (full 128-byte) rows are fetched per tile.
//
// MODE: 0 plain epilogue, 1 CUDA-core LoRA expand in the epilogue, 2 fused LoRA K-stages,
// 3 activation epilogue, 4 activation epilogue with fused LoRA K-stages into a delta
// accumulator (so g and the delta are rounded to bf16 separately).  Each mode is its own
// instantiation, so a launch carries only its own code.
//
// TMEM (512 columns): two accumulators of BN columns, and in MODE 4 up to BN = 128 two delta
// accumulators after them.  At wider tiles MODE 4 has no room for a delta buffer, so tile i's
// LoRA stages go into the idle accumulator (the one tile i+1 will use) once tile i-1's
// activation has left it; they sit in the middle of tile i's main loop, and as soon as they
// are done (`dfull`) the epilogue copies the delta, rounded to bf16, into registers and hands
// the idle buffer back (`dfree`) while tile i's last main stages still run.
//
// CG = 2: clusters of two CTAs (one TPC) share each tile as an M = 256 tcgen05 pair MMA.
// A tile is then two consecutive 128-row weight tiles (the even CTA's, then the odd CTA's)
// x BN tokens; each CTA loads its 128 weight rows and BN/2 of the token rows, so each SM
// takes in a third less per MMA than with 128 x BN tiles.  The even CTA's producer expects
// both CTAs' bytes on its full barriers, its MMA warp issues for the pair and multicasts
// the commits, and both CTAs' epilogue warps release the even CTA's accumulator barriers.
template <int BN, int MODE, int CG>
__global__ void __launch_bounds__(kGemmThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmParams p) {
  static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair per tile");
  constexpr int BNH = BN / CG;   // token rows this CTA loads per stage
  static_assert(BNH % 8 == 0, "stage buffers stay 1024-byte aligned");
  constexpr bool kFused = MODE == 2 || MODE == 4;
  constexpr bool kAct = MODE >= 3;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

  constexpr uint32_t A_BYTES = kAByte;
  constexpr uint32_t STAGE = A_BYTES + BNH * 128;
  constexpr bool delta_acc = MODE == 4;
  constexpr int kAccBufs = 2;
  static_assert(2 * BN <= 512, "two accumulators fit TMEM");
  constexpr bool kDeltaIdle = delta_acc && 4 * BN > 512;   // the delta goes into the idle accumulator
  constexpr int kDeltaBufs = (delta_acc && !kDeltaIdle) ? 2 : 0;
  constexpr uint32_t kColsUsed = static_cast<uint32_t>((kAccBufs + kDeltaBufs) * BN);
  static_assert(kColsUsed <= 512u, "accumulators exceed TMEM");
  constexpr uint32_t TMEM_COLS = kColsUsed <= 32u ? 32u : kColsUsed <= 64u ? 64u : kColsUsed <= 128u ? 128u
                                 : kColsUsed <= 256u ? 256u : 512u;   // a power of two
  const int S = p.stages;
  // accumulator releases: every epilogue thread of a single CTA, or one per epilogue warp
  // of the pair (the odd CTA's warps arrive remotely)
  constexpr uint32_t kRelease = CG == 2 ? 8u : 128u;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;       // [2]
  uint64_t* tempty = tfull + 2;      // [2]
  uint64_t* drain = tempty + 2;      // [1], used only after an abort
  uint64_t* dfull = drain + 1;       // [1], MODE 4 with kDeltaIdle: the tile's delta is complete
  uint64_t* dfree = dfull + 1;       // [1], ... and merged: the idle accumulator is free again
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dfree + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* tile_start = reinterpret_cast<int*>(tmem_slot + 4);   // [E + 1]
  int* seg = tile_start + (p.E + 1);                         // offsets copy [E + 1]
  volatile uint32_t* tile_slot_ring =                        // [kTileRing] producer -> MMA warp:
      reinterpret_cast<volatile uint32_t*>(seg + (p.E + 1));  //   LoRA slot mask of the i-th tile
  int* lslot = seg + (p.E + 1) + kTileRing + 4;              // [BN] (LoRA epilogue)
  float* v_s = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(lslot + BN) + 15) & ~static_cast<uintptr_t>(15));
  // v_s: [BN][RP8] (16-byte aligned), RP8 = R rounded up to 8

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = CG == 2 ? cluster_ctarank() : 0u;   // 0: the pair's MMA issuer
  const bool leader = crank == 0;
  const int cta0 = static_cast<int>(blockIdx.x) / CG, ncta = static_cast<int>(gridDim.x) / CG;
  const int E = p.E;
  const int NT = p.gated ? (p.N >> 7) : ((p.N + 127) >> 7);   // 128-row weight tiles per expert
  const int KB = p.K >> 6;                                    // 64-wide K blocks

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], kRelease);
    mbar_init(&tempty[1], kRelease);
    mbar_init(drain, 1);
    mbar_init(dfull, 1);
    mbar_init(dfree, kRelease);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmap_w);
    tma_prefetch_desc(&p.tmap_x);
    if (kFused && p.lora_packed) {
      tma_prefetch_desc(&p.tmap_lbp);
      tma_prefetch_desc(&p.tmap_lup);
    }
  }
  if (warp == 1) {
    if constexpr (CG == 2) {
      tmem_alloc_pair(tmem_slot, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  // ceil(M_e/BN) * NT/CG tiles per expert
  if (warp == 2) build_tile_schedule(p.offsets, E, BN, NT / CG, seg, tile_start);
  tc_fence_before();
  if constexpr (CG == 2) {   // the peer's barriers are initialised before any remote use
    cluster_arrive();
    cluster_wait();
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // With shrink_in_gemm the LoRA shrink tiles (one per expert token tile) come first.
  constexpr bool kShrinkable = kFused && CG == 1 && !kDeltaIdle;
  const int nshrink = (kShrinkable && p.shrink_in_gemm) ? tile_start[E] / (NT / CG) : 0;
  const int total = nshrink + tile_start[E];

  auto decode_shrink = [&](int t, int& e, int& qt) {   // shrink tile t: expert e, token tile qt
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] / (NT / CG) <= t) lo = mid; else hi = mid - 1;
    }
    e = lo;
    qt = t - tile_start[e] / (NT / CG);
  };
  // the active LoRA slot of pair q, from the token's slot that the permute gathered into
  // pair_slot (one load, no chain through perm; -1: none, disabled or out of range)
  auto pair_lora_slot = [&](int q) -> int {
    const int sl = p.pair_slot[q];
    if (sl < 0 || sl >= p.slots.S) return -1;
    return (p.slots.ranks[sl] > 0 && p.slots.scal[sl] != 0.0f) ? sl : -1;
  };

  auto decode = [&](int tile, int& e, int& nt, int& qt) {
    int lo = 0, hi = E - 1;   // last expert with tile_start <= tile (empty experts skipped)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int local = tile - tile_start[e];
    const int nq = (seg[e + 1] - seg[e] + BN - 1) / BN;
    const int ntp = local / nq;
    qt = local - ntp * nq;
    nt = ntp * CG + static_cast<int>(crank);   // this CTA's 128-row weight tile
  };

  // an epilogue thread's release of an accumulator barrier (kRelease arrivals complete it)
  auto release = [&](uint64_t* bar) {
    if constexpr (CG == 2) {   // one arrival per warp, on the pair's (even CTA's) barrier
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_addr(bar, 0));
    } else {
      mbar_arrive(bar);
    }
  };

  // (epilogue warps) shrink tile t in accumulator `acc`: each thread holds one stacked A row
  // (its TMEM lane) for the tile's tokens and writes that row's ub column of every token's
  // stacked row, scaled and rounded to bf16 where the token's slot is the row's slot, zero
  // elsewhere; the columns no row covers (rank padding, disabled slots) are zeroed by the
  // threads in turn; then the tile's ready flag is released.  A slot index outside [-1, S)
  // is reported here.
  auto shrink_epilogue = [&](int t, int acc, uint32_t aphase) -> bool {
    const int quarter = warp & 3;
    const int etid = threadIdx.x - 64;
    const int row = quarter * 32 + lane;
    int e, qt;
    decode_shrink(t, e, qt);
    const int q0 = seg[e] + qt * BN;
    const int nvalid = min(BN, seg[e + 1] - q0);
    epi_bar();   // every reader of the previous tile's buffers (which lslot may share) is done
    for (int j = etid; j < nvalid; j += 128) {
      int sl = p.slot_idx[p.perm[q0 + j] / p.k];
      if (sl < -1 || sl >= p.slots.S) {
        record_status(p.status, kDevBadSlot, kWhereGemmEpilogue);
        sl = -1;
      } else if (sl >= 0 && (p.slots.ranks[sl] <= 0 || p.slots.scal[sl] == 0.0f)) {
        sl = -1;
      }
      lslot[j] = sl;
    }
    epi_bar();
    int s_row = -1, col = 0;
    float sc = 0.0f;
    if (row < p.sa_row_off[kMaxFusedSlots]) {
      s_row = 0;
      while (p.sa_row_off[s_row + 1] <= row) ++s_row;
      col = p.coff[s_row] + row - p.sa_row_off[s_row];
      sc = p.slots.scal[s_row];
    }
    // this thread's zero columns, etid + 128 i (i < 3: the host keeps lora_rs <= 384), as bits
    uint32_t zmask = 0;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int c = etid + 128 * i;
      if (c < p.lora_rs) {
        int s2 = 0;
        while (p.coff[s2 + 1] <= c) ++s2;
        if (c - p.coff[s2] >= p.sa_row_off[s2 + 1] - p.sa_row_off[s2]) zmask |= 1u << i;
      }
    }
    if (!mbar_wait(&tfull[acc], aphase, abort_flag, p.status, kWhereGemmEpilogue)) return false;
    tc_fence_after();
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
    for (int c = 0; c < nvalid; c += 16) {   // warp-uniform bound
      uint32_t v[16];
      __syncwarp();   // tcgen05.ld is .aligned
      tmem_ld_x16(taddr + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (c + j < nvalid) {
          __nv_bfloat16* urow = p.ub_out + static_cast<size_t>(q0 + c + j) * p.lora_rs;
          if (s_row >= 0) urow[col] = __float2bfloat16_rn(lslot[c + j] == s_row ? sc * __uint_as_float(v[j]) : 0.0f);
#pragma unroll
          for (int i = 0; i < 3; ++i)
            if ((zmask >> i) & 1u) urow[etid + 128 * i] = __float2bfloat16_rn(0.0f);
        }
      }
    }
    __threadfence();
    fence_proxy_async_global();   // read next by other CTAs' TMA copies
    tc_fence_before();
    epi_bar();                    // every thread's rows are written (and lslot is free again)
    if (etid == 0) red_release_add(p.shrink_ready + t, 1);
    return true;
  };

  if (warp >= 2) pdl_wait();   // the epilogues read the previous kernel's LoRA rows and slots
  if (warp == 0) {   // ------------------------------------------------ TMA producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0;       // stages with a load in flight, and their parity
    uint32_t issued_parity = 0;
    int ok = 1;
    int npre = 0, nissued = 0;   // stages whose weight half went out before pdl_wait
    // a copy into this CTA's stage s, counted on the pair's (even CTA's) full barrier s
    auto load = [&](void* dst, const CUtensorMap* map, int s, int x, int y, uint64_t pol) {
      if constexpr (CG == 2) tma_load_2d_pair(dst, map, cluster_addr(&full[s], 0), x, y, pol);
      else tma_load_2d(dst, map, &full[s], x, y, pol);
    };
    auto issue = [&](const CUtensorMap* wmap, int wr0, int wr1, int kx, const CUtensorMap* xmap, int xrow) -> bool {
      if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, kWhereGemmProducer)) return false;
      uint8_t* a = smem + stage * STAGE;
      if (nissued++ >= npre) {
        if (leader) mbar_arrive_expect_tx(&full[stage], CG * STAGE);
        load(a, wmap, stage, kx, wr0, pol_w);
        load(a + 8192, wmap, stage, kx, wr1, pol_w);
      }
      load(a + A_BYTES, xmap, stage, kx, xrow, pol_x);
      issued_mask |= 1u << stage;
      issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
      return true;
    };
    auto weight_rows = [&](int e, int nt, int& wr0, int& wr1) {
      if (p.gated) {
        wr0 = e * p.N + nt * 64;
        wr1 = wr0 + (p.N >> 1);
      } else {
        wr0 = e * p.N + nt * 128;
        wr1 = wr0 + 64;
      }
    };
    // Weights are constants of the layer and the tile schedule comes from the expert
    // offsets, so the weight halves of the first tile's first stages go out before the
    // previous kernel (which writes the token rows) has finished.
    if (lane == 0 && cta0 >= nshrink && cta0 < total) {
      int e, nt, qt, wr0, wr1;
      decode(cta0 - nshrink, e, nt, qt);
      weight_rows(e, nt, wr0, wr1);
      npre = min(S, kFused ? lora_stage_pos(KB) : KB);   // main stages only: the LoRA stages follow later
      for (int s2 = 0; s2 < npre; ++s2) {
        uint8_t* a = smem + s2 * STAGE;
        if (leader) mbar_arrive_expect_tx(&full[s2], CG * STAGE);
        load(a, &p.tmap_w, s2, s2 * 64, wr0, pol_w);
        load(a + 8192, &p.tmap_w, s2, s2 * 64, wr1, pol_w);
        issued_mask |= 1u << s2;   // phase 0
      }
    }
    pdl_wait();
    if constexpr (!kFused) {   // lane 0 alone: no per-tile warp traffic
      if (lane == 0) {
        for (int tile = cta0; ok && tile < total; tile += ncta) {
          int e, nt, qt, wr0, wr1;
          decode(tile, e, nt, qt);
          weight_rows(e, nt, wr0, wr1);
          const int xr = seg[e] + qt * BN;
          const int xh = xr + static_cast<int>(crank) * BNH;   // this CTA's token rows
          for (int kb = 0; ok && kb < KB; ++kb) ok = issue(&p.tmap_w, wr0, wr1, kb * 64, &p.tmap_x, xh);
        }
      }
    } else {   // the whole warp: lanes gather each tile's pair slots for lane 0
      int it_tile = 0;
      for (int tile = cta0; tile < total; tile += ncta, ++it_tile) {
        if (tile < nshrink) {   // shrink tile: every active slot's A rows x the tile's token rows
          int e, qt;
          decode_shrink(tile, e, qt);
          const int xr = seg[e] + qt * BN;
          if (lane == 0) {
            tile_slot_ring[it_tile % kTileRing] = 0u;   // no LoRA stages in a shrink tile
            const int ea = p.sa_e1 ? 0 : e;
            const uint32_t bytes = static_cast<uint32_t>(p.sa_row_off[kMaxFusedSlots] + BNH) * 128u;
            for (int kb = 0; ok && kb < KB; ++kb) {
              if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, kWhereGemmProducer)) {
                ok = 0;
                break;
              }
              uint8_t* a = smem + stage * STAGE;
              mbar_arrive_expect_tx(&full[stage], bytes);
              if (p.sa_packed) {   // every slot's rows of the expert: one block of the shrink-ready A
                load(a, &p.tmap_sa[0], stage, kb * 64, ea * p.sa_R, pol_x);
              } else {
                for (int sl = 0; sl < kMaxFusedSlots; ++sl)
                  if (p.sa_row_off[sl + 1] > p.sa_row_off[sl])
                    load(a + p.sa_row_off[sl] * 128, &p.tmap_sa[sl], stage, kb * 64,
                         (sl * (p.sa_e1 ? 1 : E) + ea) * p.sa_R, pol_x);
              }
              load(a + A_BYTES, &p.tmap_x, stage, kb * 64, xr, pol_x);
              issued_mask |= 1u << stage;
              issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
              if (++stage == S) {
                stage = 0;
                phase ^= 1u;
              }
            }
          }
          if (!__shfl_sync(0xffffffffu, ok, 0)) break;
          continue;
        }
        int e, nt, qt, wr0, wr1;
        decode(tile - nshrink, e, nt, qt);
        weight_rows(e, nt, wr0, wr1);
        const int xr = seg[e] + qt * BN;
        const int xh = xr + static_cast<int>(crank) * BNH;   // this CTA's token rows
        // the tile's pair slots are loaded now (all loads in flight at once) and reduced only
        // after all but the last main stage are issued, so their latency hides behind the
        // tile's own copies
        const int nv = min(BN, seg[e + 1] - xr);
        constexpr int kSlotLoads = (BN + 31) / 32;
        int slv[kSlotLoads];
#pragma unroll
        for (int u = 0; u < kSlotLoads; ++u) {
          const int j = lane + 32 * u;
          slv[u] = j >= nv ? -1 : (nshrink > 0 ? pair_lora_slot(xr + j) : p.pair_slot[xr + j]);
        }
        const int kb_lora = lora_stage_pos(KB);
        if (lane == 0)
          for (int kb = 0; ok && kb < kb_lora - 1; ++kb) ok = issue(&p.tmap_w, wr0, wr1, kb * 64, &p.tmap_x, xh);
        unsigned lmask = 0;
#pragma unroll
        for (int u = 0; u < kSlotLoads; ++u)
          if (slv[u] >= 0 && slv[u] < kMaxFusedSlots) lmask |= 1u << slv[u];
        const unsigned smask = __reduce_or_sync(0xffffffffu, lmask);
        if (lane == 0) {
          // published before the main stage in front of the LoRA stages arrives
          // (arrive.expect_tx releases it); the MMA warp reads it after consuming that stage
          tile_slot_ring[it_tile % kTileRing] = smask;
          const int lb_off = p.lora_b_e1 ? e * p.N : 0;   // a shared B has one expert's rows
          if (ok) ok = issue(&p.tmap_w, wr0, wr1, (kb_lora - 1) * 64, &p.tmap_x, xh);
          if (ok && smask != 0u && nshrink > 0) {   // this tile's ub rows come from its shrink tile
            ok = wait_flag_geq(p.shrink_ready + tile_start[e] / (NT / CG) + qt, 1, abort_flag, p.status,
                               kWhereGemmProducer);
            fence_proxy_async_global();   // written by st.global, read next by TMA
          }
          if (p.lora_packed) {   // LoRA expand stages over the stacked ranks, per 64-column panel
            const int prow = ((p.lora_b_e1 ? 0 : e) * NT + nt) * 128;
            const int npan = (p.lora_rs + 63) >> 6;
            for (int j = 0; ok && j < npan; ++j)
              if (smask & p.lora_panel_slots[j]) ok = issue(&p.tmap_lbp, prow, prow + 64, j * 64, &p.tmap_lup, xh);
          } else {
            for (int sl = 0; ok && sl < kMaxFusedSlots; ++sl) {   // LoRA expand stages, per slot
              if (!((smask >> sl) & 1u)) continue;
              const int nkb = lora_blocks(p.slots.ranks[sl], p.lora_kb);
              for (int kb = 0; ok && kb < nkb; ++kb)
                ok = issue(&p.tmap_lb[sl], wr0 - lb_off, wr1 - lb_off, kb * 64, &p.tmap_lu, sl * p.P + xh);
            }
          }
          for (int kb = kb_lora; ok && kb < KB; ++kb) ok = issue(&p.tmap_w, wr0, wr1, kb * 64, &p.tmap_x, xh);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
    }
    pdl_trigger();   // all of this CTA's copies are issued: the next kernel may start
    if (lane == 0 && !ok) {   // drain: let every issued copy land before the CTA exits
      if (leader) {   // the pair's full barriers count both CTAs' bytes
        for (int s2 = 0; s2 < S; ++s2)
          if ((issued_mask >> s2) & 1u) mbar_wait_drain(&full[s2], (issued_parity >> s2) & 1u);
      } else {        // the odd CTA's copies are counted in the even CTA: give them time to land
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < kPeerDrainNs) {
        }
      }
    }
  } else if (warp == 1) {   // ------------------------------------------ MMA issuer (lane 0)
    constexpr uint32_t idesc = idesc_bf16_f32(128 * CG, BN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t aphase = 0;
    uint32_t dphase = 0;
    int ok = 1;
    auto consume = [&](uint32_t d, bool first, int nk = 4) -> bool {   // nk: 16-deep steps with data
      if (!mbar_wait(&full[stage], phase, abort_flag, p.status, kWhereGemmMma)) return false;
      tc_fence_after();
      const uint32_t a_addr = smem_u32(smem + stage * STAGE);
      const uint64_t ad = sw128_kmajor_desc(a_addr);
      const uint64_t bd = sw128_kmajor_desc(a_addr + A_BYTES);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (kk >= nk) break;
        if constexpr (CG == 2) umma_bf16_pair(d, ad + 2 * kk, bd + 2 * kk, idesc, (first && kk == 0) ? 0u : 1u);
        else umma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (first && kk == 0) ? 0u : 1u);
      }
      if constexpr (CG == 2) umma_commit_pair_mc(&empty[stage], 0x3);   // both CTAs' stage s is free
      else umma_commit(&empty[stage]);
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
      return true;
    };
    auto commit_all = [&](uint64_t* bar) {   // arrive on `bar` in the epilogue's CTA(s)
      if constexpr (CG == 2) umma_commit_pair_mc(bar, 0x3);
      else umma_commit(bar);
    };
    if (lane == 0 && leader) {   // the pair's MMAs are issued by its even CTA
      int it_tile = 0;
      for (int tile = cta0; ok && tile < total; tile += ncta, ++it_tile) {
        if (!mbar_wait(&tempty[acc], aphase ^ 1u, abort_flag, p.status, kWhereGemmMma)) break;
        if constexpr (kDeltaIdle) {   // the previous tile's delta has been merged out of this buffer
          if (it_tile > 0) {
            if (!mbar_wait(dfree, dphase, abort_flag, p.status, kWhereGemmMma)) break;
            dphase ^= 1u;
          }
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
        const int kb_lora = kFused ? lora_stage_pos(KB) : KB;
        for (int kb = 0; ok && kb < kb_lora; ++kb) ok = consume(d, kb == 0);
        if constexpr (kFused) {
          // the stage in front of the LoRA stages has landed, so the slot mask is published
          const unsigned smask = tile_slot_ring[it_tile % kTileRing];
          uint32_t dl = delta_acc ? tmem_base + static_cast<uint32_t>(kAccBufs * BN + acc * BN) : d;
          if constexpr (kDeltaIdle) {
            dl = tmem_base + static_cast<uint32_t>((acc ^ 1) * BN);
            if (ok && smask != 0u) {   // the idle buffer, once tile i-1's activation has left it
              const uint32_t xpar = ((static_cast<uint32_t>(it_tile + 1) >> 1) & 1u) ^ 1u;
              ok = mbar_wait(&tempty[acc ^ 1], xpar, abort_flag, p.status, kWhereGemmMma);
              tc_fence_after();
            }
          }
          bool first_delta = delta_acc;   // the delta accumulator starts fresh each tile
          if (p.lora_packed) {
            const int npan = (p.lora_rs + 63) >> 6;
            for (int j = 0; ok && j < npan; ++j) {
              if (!(smask & p.lora_panel_slots[j])) continue;
              ok = consume(dl, first_delta, min(4, (p.lora_rs - 64 * j) >> 4));
              first_delta = false;
            }
          } else {
            for (int sl = 0; ok && sl < kMaxFusedSlots; ++sl) {
              if (!((smask >> sl) & 1u)) continue;
              const int rank = p.slots.ranks[sl];
              const int nkb = lora_blocks(rank, p.lora_kb);
              for (int kb = 0; ok && kb < nkb; ++kb) {
                ok = consume(dl, first_delta, lora_ksteps(rank, kb));
                first_delta = false;
              }
            }
          }
          // the delta is complete before the tile's last main stages: the epilogue can take it
          // out of the idle buffer while they run (every tile, LoRA or not)
          if constexpr (kDeltaIdle) {
            if (ok) commit_all(dfull);
          }
        }
        for (int kb = kb_lora; ok && kb < KB; ++kb) ok = consume(d, false);
        if (!ok) break;
        commit_all(&tfull[acc]);   // both CTAs' epilogues
        if (++acc == kAccBufs) {
          acc = 0;
          aphase ^= 1u;
        }
      }
    }
  } else if constexpr (kAct) {   // --------------------------- epilogue, fused activation
    const int quarter = warp & 3;
    const int I = p.N >> 1;
    float* xchg = reinterpret_cast<float*>(lslot);   // [2][64][kXchgStride]
    int acc = 0, chunk = 0;   // chunk: the xchg buffer alternates per 16-token chunk
    uint32_t aphase = 0, dfphase = 0;
    for (int tile = cta0; tile < total; tile += ncta) {
      if (tile < nshrink) {
        if (!shrink_epilogue(tile, acc, aphase)) break;
        release(&tempty[acc]);
        if (++acc == kAccBufs) {
          acc = 0;
          aphase ^= 1u;
        }
        continue;
      }
      int e, nt, qt;
      decode(tile - nshrink, e, nt, qt);
      const int q0 = seg[e] + qt * BN;
      const int nvalid = min(BN, seg[e + 1] - q0);
      // the delta accumulator holds this tile's LoRA only if some slot was present
      unsigned lmask = 0;
      if (delta_acc) {
        for (int j = lane; j < nvalid; j += 32) {
          const int sl = nshrink > 0 ? pair_lora_slot(q0 + j) : p.pair_slot[q0 + j];
          if (sl >= 0 && sl < kMaxFusedSlots) lmask |= 1u << sl;
        }
        lmask = __reduce_or_sync(0xffffffffu, lmask);
      }
      const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
      const uint32_t tm = tmem_base + lane_base + static_cast<uint32_t>(acc * BN);
      const uint32_t td = tmem_base + lane_base +
                          static_cast<uint32_t>(kDeltaIdle ? (acc ^ 1) * BN : kAccBufs * BN + acc * BN);
      // One 16-token chunk of z = bf16(g) + bf16(delta): every lane parks its 16 values
      // (feature row = TMEM lane); then thread t computes token t / 8 of the chunk for
      // features 8 * (t % 8) .. + 8 and writes them in one 16-byte store.
      auto act_chunk = [&](int c, const float (&z)[16]) {
        float* buf = xchg + (chunk & 1) * 128 * kXchgStride;
        ++chunk;
        float* mine = buf + (quarter * 32 + lane) * kXchgStride;
#pragma unroll
        for (int j = 0; j < 16; ++j) mine[j] = z[j];
        epi_bar();   // this chunk's values are in; the other buffer is free again
        const int et = (quarter * 32 + lane);   // 0..127, any fixed numbering of the 128 threads
        const int tok = et >> 3, f8 = (et & 7) * 8;
        if (c + tok < nvalid) {
          float out8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float zg = buf[(f8 + i) * kXchgStride + tok];        // gate rows 0..63
            const float zu = buf[(64 + f8 + i) * kXchgStride + tok];   // up rows 64..127
            out8[i] = __fdividef(zg, 1.0f + __expf(-zg)) * zu;
          }
          *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(q0 + c + tok) * I + nt * 64 + f8) = pack8(out8);
        }
      };
      if constexpr (kDeltaIdle) {
        // The delta of this tile leaves the idle accumulator as soon as its MMAs are done (in
        // the middle of the tile's main loop): rounded to bf16 and held in registers as pairs,
        // so the buffer goes back to the next tile's main loop at once.
        uint32_t dpk[BN / 2];
        if (!mbar_wait(dfull, dfphase, abort_flag, p.status, kWhereGemmEpilogue)) break;
        dfphase ^= 1u;
        tc_fence_after();
        if (lmask) {
#pragma unroll
          for (int cc = 0; cc < BN / 32; ++cc) {
            uint32_t t[32];
            tmem_ld_x32(td + 32 * cc, t);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(t[2 * j]), __uint_as_float(t[2 * j + 1]));
              dpk[16 * cc + j] = *reinterpret_cast<const uint32_t*>(&v);
            }
          }
        }
        tc_fence_before();
        release(dfree);
        if (!mbar_wait(&tfull[acc], aphase, abort_flag, p.status, kWhereGemmEpilogue)) break;
        tc_fence_after();
#pragma unroll
        for (int cu = 0; cu < BN / 16; ++cu) {   // unrolled: dpk is indexed statically
          const int c = cu * 16;
          if (c >= nvalid) break;                 // warp-uniform
          uint32_t gv[16];
          __syncwarp();   // the last chunk's stores branched per lane; tcgen05.ld is .aligned
          tmem_ld_x16(tm + c, gv);
          tmem_ld_wait();
          float z[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {   // bf16(g) + bf16(delta), added in fp32
            z[j] = __bfloat162float(__float2bfloat16_rn(__uint_as_float(gv[j])));
            if (lmask) {
              const uint32_t dw = dpk[8 * cu + (j >> 1)];
              z[j] += __uint_as_float((j & 1) ? (dw & 0xffff0000u) : (dw << 16));
            }
          }
          act_chunk(c, z);
        }
      } else {
        if (!mbar_wait(&tfull[acc], aphase, abort_flag, p.status, kWhereGemmEpilogue)) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < nvalid; c += 16) {   // warp-uniform bound
          uint32_t gv[16], dv[16];
          __syncwarp();   // the last chunk's stores branched per lane; tcgen05.ld is .aligned
          tmem_ld_x16(tm + c, gv);
          if (lmask) tmem_ld_x16(td + c, dv);
          tmem_ld_wait();
          float z[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {   // bf16(g) + bf16(delta), added in fp32
            z[j] = __bfloat162float(__float2bfloat16_rn(__uint_as_float(gv[j])));
            if (lmask) z[j] += __bfloat162float(__float2bfloat16_rn(__uint_as_float(dv[j])));
          }
          act_chunk(c, z);
        }
      }
      tc_fence_before();
      release(&tempty[acc]);   // done with the accumulator
      if (++acc == kAccBufs) {
        acc = 0;
        aphase ^= 1u;
      }
    }
  } else {   // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // weight row inside the tile == TMEM lane
    const int etid = threadIdx.x - 64;     // 0..127 over the epilogue warps
    constexpr bool lora = MODE == 1;
    const int R = p.slots.R;
    const int RP8 = (R + 7) & ~7;
    // this warp's store buffers: [16 tokens][32 features] (its TMEM lane quarter), two for fp32
    const int nybuf = p.y_tma ? 2 : 1;   // as sized by the host
    float* yb2 = reinterpret_cast<float*>(
                     (reinterpret_cast<uintptr_t>(v_s + (lora ? BN * RP8 : 0)) + 127) & ~static_cast<uintptr_t>(127)) +
                 quarter * nybuf * 512;   // TMA sources start on 128-byte boundaries
    const int f4 = (lane & 7) * 4;   // the 4 features this lane stores per token row
    int ychunk = 0;                  // chunks staged so far (alternating buffers)
    int acc = 0;
    uint32_t aphase = 0;
    for (int tile = cta0; tile < total; tile += ncta) {
      if (tile < nshrink) {
        if (!shrink_epilogue(tile, acc, aphase)) break;
        release(&tempty[acc]);
        if (++acc == kAccBufs) {
          acc = 0;
          aphase ^= 1u;
        }
        continue;
      }
      int e, nt, qt;
      decode(tile - nshrink, e, nt, qt);
      const int col = nt * 128 + row;
      const int q0 = seg[e] + qt * BN;
      const int nvalid = min(BN, seg[e + 1] - q0);
      if (lora) {   // stage the tile's pair slots and scaled down-LoRA shrink values
        epi_bar();
        for (int j = etid; j < nvalid; j += 128) lslot[j] = p.pair_slot[q0 + j];
        epi_bar();
        for (int i = etid; i < nvalid * RP8; i += 128) {
          const int j = i / RP8, r = i - j * RP8;
          const int sl = lslot[j];
          v_s[i] = (sl >= 0 && r < p.slots.ranks[sl]) ? p.lora_v[static_cast<size_t>(q0 + j) * R + r] : 0.0f;
        }
        epi_bar();
      }
      if (!mbar_wait(&tfull[acc], aphase, abort_flag, p.status, kWhereGemmEpilogue)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
      int c0 = 0;
      if (!lora && p.y_tma && p.out_f32 == nullptr) {
        // bf16 output (y at wide tiles): whole 32-token chunks, each one 32 x 32 TMA store, so
        // a tile takes half the TMEM round trips and stores of 16-token chunks
#pragma unroll 1
        for (; c0 + 32 <= nvalid; c0 += 32) {
          uint32_t r[32];
          __syncwarp();
          tmem_ld_x32(taddr + c0, r);
          tmem_ld_wait();
          __nv_bfloat16* ybh = reinterpret_cast<__nv_bfloat16*>(yb2 + (ychunk++ & 1) * 512);
          if (lane == 0) bulk_wait_read_1();   // the store that last read this buffer is done
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 32; ++j) ybh[j * 32 + lane] = f2bf(__uint_as_float(r[j]));
          fence_proxy_async_smem();
          __syncwarp();
          const int fcol0 = nt * 128 + quarter * 32;
          if (lane == 0 && fcol0 < p.N) {
            tma_store_2d_hint(&p.tmap_y, ybh, fcol0, q0 + c0, l2_policy_evict_last());
            bulk_commit();
          }
        }
      }
#pragma unroll 1
      for (int c = c0; c < nvalid; c += 16) {   // warp-uniform bound
        uint32_t r[16];
        __syncwarp();   // the last chunk's stores branched per lane; tcgen05.ld is .aligned
        tmem_ld_x16(taddr + c, r);
        tmem_ld_wait();
        float val[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) val[j] = __uint_as_float(r[j]);
        if (lora && col < p.N) lora_expand_chunk(p, lslot, v_s, c, nvalid, e, col, val);
        // transpose through the warp's buffer (lane = feature on the way in).  A whole fp32
        // chunk of 16 tokens leaves as one TMA store of 16 x 32 values when the host set up the
        // output's tensor map; otherwise (bf16 tails included: their map's box is 32 tokens)
        // each lane stores 4 consecutive features of a token: 4 token rows per instruction
        float* yb = yb2 + (p.y_tma ? (ychunk++ & 1) * 512 : 0);
        if (lane == 0) bulk_wait_read_1();   // the store that last read this buffer is done
        __syncwarp();
        const bool whole = p.y_tma && p.out_f32 != nullptr && c + 16 <= nvalid;
#pragma unroll
        for (int j = 0; j < 16; ++j) yb[j * 32 + lane] = val[j];
        const int fcol0 = nt * 128 + quarter * 32;
        if (whole) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && fcol0 < p.N) {
            // wide tiles: y stays in L2 as long as it can, since the finalize reads it next
            if constexpr (BN >= 64) tma_store_2d_hint(&p.tmap_y, yb, fcol0, q0 + c, l2_policy_evict_last());
            else tma_store_2d(&p.tmap_y, yb, fcol0, q0 + c);
            bulk_commit();
          }
          continue;
        }
        __syncwarp();
        const int fcol = fcol0 + f4;
        if (fcol < p.N) {   // N is a multiple of 4, so the whole vector is in range
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tok = (lane >> 3) + 4 * i;
            if (c + tok < nvalid) {
              const float4 v = *reinterpret_cast<const float4*>(yb + tok * 32 + f4);
              const size_t off = static_cast<size_t>(q0 + c + tok) * p.N + fcol;
              if (p.out_f32 != nullptr) {
                *reinterpret_cast<float4*>(p.out_f32 + off) = v;
              } else {
                const float v4[4] = {v.x, v.y, v.z, v.w};
                *reinterpret_cast<uint2*>(p.out + off) = pack4(v4);
              }
            }
          }
        }
      }
      tc_fence_before();
      release(&tempty[acc]);   // done with the accumulator
      if (++acc == kAccBufs) {
        acc = 0;
        aphase ^= 1u;
      }
    }
  }

  bulk_wait_all();   // the epilogue's TMA stores have read their buffers and landed
  tc_fence_before();
  if constexpr (CG == 2) {   // neither CTA leaves while the pair's MMAs may touch its memory
    cluster_arrive();
    cluster_wait();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    if (*abort_flag && leader) {   // let the MMAs lane 0 already issued finish before TMEM is released
      if (lane == 0) {
        if constexpr (CG == 2) umma_commit_pair(drain);
        else umma_commit(drain);
        mbar_wait_drain(drain, 0);
      }
      __syncwarp();
    }
    tc_fence_after();
    if constexpr (CG == 2) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int BN, int MODE, int CG>
static cudaError_t launch_mode(const GemmParams& p, int grid, cudaStream_t stream, bool pdl) {
  const int smem = gemm_smem_bytes(BN, CG, p.stages, p.E, p.lora_v != nullptr ? p.slots.R : 0, p.gated == 2,
                                   p.y_tma);
  cudaError_t err =
      cudaFuncSetAttribute(grouped_gemm_kernel<BN, MODE, CG>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  grid = grid / CG * CG;   // whole clusters
  if (grid < CG) return cudaErrorInvalidValue;
  return launch_kc(grouped_gemm_kernel<BN, MODE, CG>, dim3(grid), dim3(kGemmThreads), static_cast<size_t>(smem),
                   stream, pdl, CG, p);
}

template <int BN, int CG>
static cudaError_t launch_bn(const GemmParams& p, int grid, cudaStream_t stream, bool pdl) {
  if (p.gated == 2)
    return p.lora_fused ? launch_mode<BN, 4, CG>(p, grid, stream, pdl) : launch_mode<BN, 3, CG>(p, grid, stream, pdl);
  if (p.lora_fused) return launch_mode<BN, 2, CG>(p, grid, stream, pdl);
  if (p.lora_v != nullptr) {   // the CUDA-core LoRA epilogue runs on single-CTA tiles only
    if constexpr (CG == 1) return launch_mode<BN, 1, 1>(p, grid, stream, pdl);
    else return cudaErrorInvalidValue;
  }
  return launch_mode<BN, 0, CG>(p, grid, stream, pdl);
}

cudaError_t launch_grouped_gemm(const GemmParams& p, int bn, int grid, cudaStream_t stream, bool pdl) {
  if (p.stages < 2 || p.stages > kMaxStages) return cudaErrorInvalidValue;
  if (p.cta_pair == 2) {
    const int nt = p.gated ? (p.N >> 7) : ((p.N + 127) >> 7);
    if (nt % 2 != 0) return cudaErrorInvalidValue;   // a pair covers two weight tiles
    switch (bn) {
      case 128: return launch_bn<128, 2>(p, grid, stream, pdl);
      case 256: return launch_bn<256, 2>(p, grid, stream, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (bn) {
    case 16: return launch_bn<16, 1>(p, grid, stream, pdl);
    case 32: return launch_bn<32, 1>(p, grid, stream, pdl);
    case 64: return launch_bn<64, 1>(p, grid, stream, pdl);
    case 128: return launch_bn<128, 1>(p, grid, stream, pdl);
    case 256: return launch_bn<256, 1>(p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mlk
