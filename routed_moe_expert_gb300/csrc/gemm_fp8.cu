// Grouped (per-expert) GEMM with FP8 block-scale operands on the 5th-generation tensor
// cores: TMA -> shared memory -> tcgen05.mma (kind::f8f6f4, e4m3 x e4m3 -> fp32) -> TMEM
// -> registers (block-scale promotion) -> global.
//
// For every expert e and its routed pairs q in [offsets[e], offsets[e+1]):
//     out[q, col] = sum_b sx[b][q] * sw[e][n / 128][b] * sum_{k in block b} X8[q, k] * W8[e*N + n, k]
// with n = row(col) the weight row of the output column and b the 128-wide K blocks.  X8
// and W8 are e4m3 codes, sw one float32 scale per 128 x 128 weight block and sx one per
// pair and K block: the base GEMMs of the pages' FP8 flow (sglang PR #28466, section 1
// flow (A): the FP8 flow quantises the hidden states per token group before the MoE op
// and the activation before the down GEMM; its summary ties that path to block-quantised
// weights).
//
// Orientation, tile schedule and warp roles are those of the bf16 grouped GEMM: the
// weights are the MMA "A" operand (M = 128 rows), the expert's tokens are "B" (N = BN
// columns, BN <= 64), persistent CTAs walk a static tile list, warp 0 issues TMA, warp 1
// allocates TMEM and issues the MMAs, warps 2-5 are the epilogue.  One pipeline stage is
// one K block: 128 e4m3 values = one 128-byte swizzle row per operand row, consumed by
// four MMAs of K = 32.  Because both scales change from one K block to the next, the
// MMAs of each block write a fresh partial sum into one of four TMEM buffers and the
// epilogue folds it into fp32 registers,
//     acc[j] += partial[j] * (sw * sx[j]),
// releasing the buffer as soon as it has been read, so the tensor cores run up to three
// blocks ahead of the epilogue.  After the last block the registers hold the tile's
// output, which leaves through a per-warp shared-memory transpose as 16-byte stores.
//
// gated = 1 (gate_up): tile n holds gate rows [64n, 64n+64) and up rows [N/2+64n, ...)
// and the output is gated-interleaved (column 128n + j), as in the bf16 GEMM.
//
// Every mbarrier wait is bounded (2 s); a timeout records MOE_LORA_ERR_TIMEOUT, raises a
// CTA-wide abort flag, drains the copies already issued and frees TMEM before returning.
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace mlk {

constexpr int kF8Threads = 192;
constexpr int kF8Parts = 4;                 // TMEM partial-sum buffers
constexpr int kF8AByte = 128 * 128;         // 128 weight rows x 128 e4m3 values
constexpr int kF8MaxStages = 16;
constexpr int kF8YbufFloats = 16 * 32;      // per epilogue warp: 16 tokens x 32 features

int gemm_fp8_stage_bytes(int bn) { return kF8AByte + bn * 128; }

constexpr int kF8Ring = 32;   // > kF8MaxStages: the producer runs at most that many tiles ahead

int gemm_fp8_smem_bytes(int bn, int stages, int E, int lora_R, int lora_packed) {
  // Carve-up, in order (see the kernel): 1 KB alignment slack; stage buffers; full/empty
  // barriers (2*stages), partial full/empty (2*kF8Parts), drain (1), with packed LoRA stages
  // the delta full/empty (2); tmem slot + abort flag (16 B); tile_start and seg (E+1 ints
  // each); with packed LoRA stages the tile slot-mask ring; for the LoRA epilogue BN token
  // slots then BN x RP8 floats aligned to 16 bytes; the four warps' store buffers.
  const int lora = lora_R > 0 ? bn * 4 + 16 + bn * ((lora_R + 7) / 8 * 8) * 4 : 0;
  const int lp = lora_packed ? 2 * 8 + kF8Ring * 4 : 0;
  return 1024 + stages * gemm_fp8_stage_bytes(bn) + (2 * stages + 2 * kF8Parts + 1) * 8 + 16 + 8 * (E + 1) + lp +
         lora + 16 + 4 * kF8YbufFloats * 4;
}

// Instruction descriptor, kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B e4m3 (bits 7-9 and
// 10-12 = 0), both K-major, N>>3 at bits 17-22, M>>4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T with e4m3 inputs and fp32 accumulation, cta_group::1.
MLDEV void umma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

MLDEV void f8_epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }   // the 4 epilogue warps

// Down-LoRA expand of one 16-token chunk for output feature `feat` (this thread's weight
// row): val[j] += sum_{r < ranks[s]} lora_B[s, e, feat, r] * v_s[c + j][r] for each
// token j of the chunk whose pair has slot s = lslot[c + j] >= 0.  v_s rows hold
// scaling[s] * (down-LoRA shrink), RP8 floats each, zero past the slot's rank.
MLDEV void f8_lora_expand(const GemmF8Params& p, const int* lslot, const float* v_s, int c, int nvalid, int e,
                          int feat, float (&val)[16]) {
  const int R = p.slots.R;
  const int RP8 = (R + 7) & ~7;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (c + j >= nvalid) break;
    const int sl = lslot[c + j];
    if (sl < 0) continue;
    const int rank = p.slots.ranks[sl];
    const size_t be = p.lora_b_e1 ? static_cast<size_t>(sl) : static_cast<size_t>(sl) * p.E + e;
    const __nv_bfloat16* Brow = p.lora_B + (be * p.N + feat) * static_cast<size_t>(R);
    const float* vj = v_s + (c + j) * RP8;
    float sum = 0.0f;
#pragma unroll 1
    for (int r0 = 0; r0 < rank; r0 += 8) {
      float b[8];
      if ((R & 7) == 0 && r0 + 8 <= rank) {
        unpack8(__ldg(reinterpret_cast<const uint4*>(Brow + r0)), b);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = (r0 + i < rank) ? bf2f(Brow[r0 + i]) : 0.0f;
      }
      const float4 v0 = *reinterpret_cast<const float4*>(vj + r0);
      const float4 v1 = *reinterpret_cast<const float4*>(vj + r0 + 4);
      sum += b[0] * v0.x + b[1] * v0.y + b[2] * v0.z + b[3] * v0.w + b[4] * v1.x + b[5] * v1.y + b[6] * v1.z +
             b[7] * v1.w;
    }
    val[j] += sum;
  }
}

// LP: fused LoRA expand stages from the packed B (see GemmF8Params), into a delta accumulator
// after the kF8Parts partial buffers.
template <int BN, bool LORA, bool LP>
__global__ void __launch_bounds__(kF8Threads, 1) grouped_gemm_fp8_kernel(const __grid_constant__ GemmF8Params p) {
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 64, "token tiles of 16 to 64");
  static_assert(!(LORA && LP), "one LoRA placement");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

  constexpr uint32_t STAGE = kF8AByte + BN * 128;
  constexpr uint32_t kCols = (kF8Parts + (LP ? 1 : 0)) * BN;
  constexpr uint32_t TMEM_COLS = kCols <= 32u ? 32u : kCols <= 64u ? 64u : kCols <= 128u ? 128u
                                 : kCols <= 256u ? 256u : 512u;
  constexpr uint32_t kDeltaCol = kF8Parts * BN;   // LP: the delta accumulator's first column
  constexpr int kSxLoads = (BN + 31) / 32;   // scales of the tile's tokens per lane and K block
  const int S = p.stages;
  const int E = p.E;
  const int R = p.slots.R;
  const int RP8 = (R + 7) & ~7;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE);
  uint64_t* empty = full + S;
  uint64_t* pfull = empty + S;        // [kF8Parts] partial sum ready (MMA commit)
  uint64_t* pempty = pfull + kF8Parts;   // [kF8Parts] partial sum read (128 epilogue threads)
  uint64_t* drain = pempty + kF8Parts;   // [1], used only after an abort
  uint64_t* dfull = drain + 1;           // LP: the tile's LoRA delta is complete (MMA commit)
  uint64_t* dempty = dfull + 1;          // LP: ... and read (128 epilogue threads)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1 + (LP ? 2 : 0));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* tile_start = reinterpret_cast<int*>(tmem_slot + 4);   // [E + 1]
  int* seg = tile_start + (E + 1);                           // offsets copy [E + 1]
  // LP: the i-th tile's LoRA slot mask, producer -> MMA warp
  volatile uint32_t* tile_slot_ring = reinterpret_cast<volatile uint32_t*>(seg + (E + 1));
  int* lslot = seg + (E + 1) + (LP ? kF8Ring : 0);           // [BN] (LoRA epilogue)
  float* v_s = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(lslot + (LORA ? BN : 0)) + 15) &
                                        ~static_cast<uintptr_t>(15));   // [BN][RP8] (LoRA epilogue)
  float* ybuf = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(v_s + (LORA ? BN * RP8 : 0)) + 15) &
                                         ~static_cast<uintptr_t>(15));  // [4][16][32]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta0 = static_cast<int>(blockIdx.x), ncta = static_cast<int>(gridDim.x);
  const int NT = p.N >> 7;   // 128-row weight tiles (and 128-row scale blocks) per expert
  const int KB = p.K >> 7;   // 128-wide K blocks

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < kF8Parts; ++i) {
      mbar_init(&pfull[i], 1);
      mbar_init(&pempty[i], 128);
    }
    mbar_init(drain, 1);
    if (LP) {
      mbar_init(dfull, 1);
      mbar_init(dempty, 128);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmap_w);
    tma_prefetch_desc(&p.tmap_x);
    if (LP) {
      tma_prefetch_desc(&p.tmap_lbp);
      tma_prefetch_desc(&p.tmap_lup);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) build_tile_schedule(p.offsets, E, BN, NT, seg, tile_start);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tile_start[E];

  auto decode = [&](int tile, int& e, int& nt, int& qt) {
    int lo = 0, hi = E - 1;   // last expert with tile_start <= tile (empty experts skipped)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int local = tile - tile_start[e];
    const int nq = (seg[e + 1] - seg[e] + BN - 1) / BN;
    nt = local / nq;
    qt = local - nt * nq;
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

  if (warp >= 2) pdl_wait();   // the epilogues read the previous kernel's scales and LoRA rows
  if (warp == 0) {   // ------------------------------------------------ TMA producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0;       // stages with a load in flight, and their parity
    uint32_t issued_parity = 0;
    int ok = 1;
    int npre = 0, nissued = 0;      // stages whose weight half went out before pdl_wait
    // The weights are constants of the layer and the tile schedule comes from the expert
    // offsets, so the first tile's first weight stages go out before the previous kernel
    // (which writes the token codes) has finished.
    if (lane == 0 && cta0 < total) {
      int e, nt, qt, wr0, wr1;
      decode(cta0, e, nt, qt);
      weight_rows(e, nt, wr0, wr1);
      // LP: the last main stage's expect_tx goes out only after the tile's slot mask is
      // published (that arrive releases it), so it is never issued early
      npre = min(S, LP ? KB - 1 : KB);
      for (int s2 = 0; s2 < npre; ++s2) {
        uint8_t* a = smem + s2 * STAGE;
        mbar_arrive_expect_tx(&full[s2], STAGE);
        tma_load_2d(a, &p.tmap_w, &full[s2], s2 * 128, wr0, pol_w);
        tma_load_2d(a + 8192, &p.tmap_w, &full[s2], s2 * 128, wr1, pol_w);
        issued_mask |= 1u << s2;   // phase 0
      }
    }
    pdl_wait();
    // the next stage's slot: wait for it to be free (false: abort)
    auto take_stage = [&]() -> uint8_t* {
      if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, kWhereGemmProducer)) return nullptr;
      return smem + stage * STAGE;
    };
    auto next_stage = [&]() {
      issued_mask |= 1u << stage;
      issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
    };
    // one tile's main K blocks (and, LP, its LoRA stages over the stacked ranks)
    auto tile_stages = [&](int e, int nt, int xr, unsigned smask, int it_tile) {
      int wr0, wr1;
      weight_rows(e, nt, wr0, wr1);
      for (int kb = 0; ok && kb < KB; ++kb) {
        uint8_t* a = take_stage();
        if (a == nullptr) {
          ok = 0;
          break;
        }
        // LP: published before the last main stage's expect_tx releases it to the MMA warp
        if (LP && kb == KB - 1) tile_slot_ring[it_tile % kF8Ring] = smask;
        if (nissued++ >= npre) {
          mbar_arrive_expect_tx(&full[stage], STAGE);
          tma_load_2d(a, &p.tmap_w, &full[stage], kb * 128, wr0, pol_w);
          tma_load_2d(a + 8192, &p.tmap_w, &full[stage], kb * 128, wr1, pol_w);
        }
        tma_load_2d(a + kF8AByte, &p.tmap_x, &full[stage], kb * 128, xr, pol_x);
        next_stage();
      }
      if constexpr (LP) {
        const int prow = ((p.lora_b_e1 ? 0 : e) * NT + nt) * 128;
        const int npan = (p.lora_rs + 63) >> 6;
        for (int j = 0; ok && j < npan; ++j) {
          if (!(smask & p.lora_panel_slots[j])) continue;
          uint8_t* a = take_stage();
          if (a == nullptr) {
            ok = 0;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], STAGE);
          tma_load_2d(a, &p.tmap_lbp, &full[stage], j * 64, prow, pol_w);
          tma_load_2d(a + 8192, &p.tmap_lbp, &full[stage], j * 64, prow + 64, pol_w);
          tma_load_2d(a + kF8AByte, &p.tmap_lup, &full[stage], j * 64, xr, pol_x);
          next_stage();
        }
      }
    };
    if constexpr (LP) {   // the whole warp: lanes gather each tile's pair slots for lane 0
      int it_tile = 0;
      for (int tile = cta0; tile < total; tile += ncta, ++it_tile) {
        int e, nt, qt;
        decode(tile, e, nt, qt);
        const int xr = seg[e] + qt * BN;
        const int nv = min(BN, seg[e + 1] - xr);
        unsigned lm = 0;
#pragma unroll
        for (int u = 0; u < (BN + 31) / 32; ++u) {
          const int j = lane + 32 * u;
          const int sl = j < nv ? p.pair_slot[xr + j] : -1;
          if (sl >= 0 && sl < kMaxFusedSlots) lm |= 1u << sl;
        }
        const unsigned smask = __reduce_or_sync(0xffffffffu, lm);
        if (lane == 0) tile_stages(e, nt, xr, smask, it_tile);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
    } else if (lane == 0) {
      for (int tile = cta0; ok && tile < total; tile += ncta) {
        int e, nt, qt;
        decode(tile, e, nt, qt);
        tile_stages(e, nt, seg[e] + qt * BN, 0u, 0);
      }
    }
    pdl_trigger();   // all of this CTA's copies are issued: the next kernel may start
    if (lane == 0 && !ok) {   // drain: let every issued copy land before the CTA exits
      for (int s2 = 0; s2 < S; ++s2)
        if ((issued_mask >> s2) & 1u) mbar_wait_drain(&full[s2], (issued_parity >> s2) & 1u);
    }
  } else if (warp == 1) {   // ------------------------------------------ MMA issuer (lane 0)
    constexpr uint32_t idesc = idesc_e4m3_f32(128, BN);
    constexpr uint32_t idesc_lora = idesc_bf16_f32(128, BN);
    if (lane == 0) {
      int stage = 0, part = 0;
      uint32_t phase = 0, pphase = 0, dphase = 0;
      bool ok = true;
      int it_tile = 0;
      for (int tile = cta0; ok && tile < total; tile += ncta, ++it_tile) {
        for (int kb = 0; ok && kb < KB; ++kb) {
          ok = mbar_wait(&pempty[part], pphase ^ 1u, abort_flag, p.status, kWhereGemmMma) &&
               mbar_wait(&full[stage], phase, abort_flag, p.status, kWhereGemmMma);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * STAGE);
          const uint64_t ad = sw128_kmajor_desc(a_addr);
          const uint64_t bd = sw128_kmajor_desc(a_addr + kF8AByte);
          const uint32_t d = tmem_base + static_cast<uint32_t>(part * BN);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)   // K = 32 e4m3 values = 32 bytes = 2 descriptor units
            umma_e4m3(d, ad + 2 * kk, bd + 2 * kk, idesc, kk > 0 ? 1u : 0u);
          umma_commit(&empty[stage]);   // the stage's shared memory is free
          umma_commit(&pfull[part]);    // the block's partial sum is ready
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
          if (++part == kF8Parts) {
            part = 0;
            pphase ^= 1u;
          }
        }
        if constexpr (LP) {   // the tile's LoRA stages: bf16 MMAs into the delta accumulator
          const unsigned smask = tile_slot_ring[it_tile % kF8Ring];   // published before the last main stage
          if (ok && smask != 0u) {
            ok = mbar_wait(dempty, dphase ^ 1u, abort_flag, p.status, kWhereGemmMma);   // previous delta read
            tc_fence_after();
            const uint32_t dd = tmem_base + kDeltaCol;
            const int npan = (p.lora_rs + 63) >> 6;
            bool first = true;
            for (int j = 0; ok && j < npan; ++j) {
              if (!(smask & p.lora_panel_slots[j])) continue;
              if (!mbar_wait(&full[stage], phase, abort_flag, p.status, kWhereGemmMma)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a_addr = smem_u32(smem + stage * STAGE);
              const uint64_t ad = sw128_kmajor_desc(a_addr);
              const uint64_t bd = sw128_kmajor_desc(a_addr + kF8AByte);
              const int nk = min(4, (p.lora_rs - 64 * j) >> 4);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {   // K = 16 bf16 values = 32 bytes per step
                if (kk >= nk) break;
                umma_bf16(dd, ad + 2 * kk, bd + 2 * kk, idesc_lora, (first && kk == 0) ? 0u : 1u);
              }
              first = false;
              umma_commit(&empty[stage]);
              if (++stage == S) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (ok) umma_commit(dfull);
            dphase ^= 1u;
          }
        }
      }
    }
  } else {   // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // weight row inside the tile == TMEM lane
    const int etid = threadIdx.x - 64;     // 0..127 over the epilogue warps
    float* yb = ybuf + quarter * kF8YbufFloats;
    const int f4 = (lane & 7) * 4;         // the 4 features this lane stores per token row
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int part = 0;
    uint32_t pphase = 0, dfphase = 0;
    bool ok = true;
    for (int tile = cta0; ok && tile < total; tile += ncta) {
      int e, nt, qt;
      decode(tile, e, nt, qt);
      const int q0 = seg[e] + qt * BN;
      const int nvalid = min(BN, seg[e + 1] - q0);
      unsigned lmask = 0;   // LP: the delta accumulator holds this tile's LoRA (as the producer saw it)
      if constexpr (LP) {
        for (int j = lane; j < nvalid; j += 32) {
          const int sl = p.pair_slot[q0 + j];
          if (sl >= 0 && sl < kMaxFusedSlots) lmask |= 1u << sl;
        }
        lmask = __reduce_or_sync(0xffffffffu, lmask);
      }
      if constexpr (LORA) {   // stage the tile's pair slots and scaled down-LoRA shrink values
        f8_epi_bar();
        for (int j = etid; j < nvalid; j += 128) lslot[j] = p.pair_slot[q0 + j];
        f8_epi_bar();
        for (int i = etid; i < nvalid * RP8; i += 128) {
          const int j = i / RP8, r = i - j * RP8;
          const int sl = lslot[j];
          v_s[i] = (sl >= 0 && r < p.slots.ranks[sl]) ? p.lora_v[static_cast<size_t>(q0 + j) * R + r] : 0.0f;
        }
        f8_epi_bar();
      }
      // this thread's weight row and its row of block scales
      const int n = p.gated ? (row < 64 ? nt * 64 + row : (p.N >> 1) + nt * 64 + row - 64) : nt * 128 + row;
      const float* swrow = p.w_scale + (static_cast<size_t>(e) * NT + (n >> 7)) * KB;
      float acc[BN];
#pragma unroll
      for (int j = 0; j < BN; ++j) acc[j] = 0.0f;
#pragma unroll 1
      for (int kb = 0; kb < KB; ++kb) {
        // the block's scales: token j's from lane j % 32 (zero past the tile's tokens)
        float sxl[kSxLoads];
#pragma unroll
        for (int u = 0; u < kSxLoads; ++u) {
          const int j = lane + 32 * u;
          sxl[u] = (j < nvalid) ? p.x_scale[static_cast<size_t>(kb) * p.P + q0 + j] : 0.0f;
        }
        const float sw = __ldg(swrow + kb);
        if (!mbar_wait(&pfull[part], pphase, abort_flag, p.status, kWhereGemmEpilogue)) {
          ok = false;
          break;
        }
        tc_fence_after();
        __syncwarp();   // the lanes left the barrier wait one by one: tcgen05.ld is .aligned
        uint32_t r[BN / 16][16];
#pragma unroll
        for (int c = 0; c < BN / 16; ++c)
          tmem_ld_x16(tmem_base + lane_base + static_cast<uint32_t>(part * BN + 16 * c), r[c]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&pempty[part]);   // the buffer may take the next block's MMAs
        if (++part == kF8Parts) {
          part = 0;
          pphase ^= 1u;
        }
#pragma unroll
        for (int j = 0; j < BN; ++j) {
          const float sx = __shfl_sync(0xffffffffu, sxl[j >> 5], j & 31);
          acc[j] = fmaf(__uint_as_float(r[j >> 4][j & 15]), sw * sx, acc[j]);
        }
      }
      if (!ok) break;
      if (LP && lmask) {
        if (!mbar_wait(dfull, dfphase, abort_flag, p.status, kWhereGemmEpilogue)) break;
        dfphase ^= 1u;
        tc_fence_after();
      }
      const int col = nt * 128 + row;   // output column of this thread's row
      const int fcol = nt * 128 + quarter * 32 + f4;
      // LP, gated: the logical column of this lane's 4 features (gate rows, then up rows)
      const int frow = quarter * 32 + f4;
      const int dcol = frow < 64 ? nt * 64 + frow : (p.N >> 1) + nt * 64 + frow - 64;
#pragma unroll
      for (int c = 0; c < BN; c += 16) {
        if (c >= nvalid) break;   // warp-uniform
        float val[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) val[j] = acc[c + j];
        if constexpr (LORA) f8_lora_expand(p, lslot, v_s, c, nvalid, e, col, val);
        float dv[16];   // LP: the LoRA delta of this row for the chunk's tokens
#pragma unroll
        for (int j = 0; j < 16; ++j) dv[j] = 0.0f;
        if (LP && lmask) {
          uint32_t r16[16];
          __syncwarp();   // tcgen05.ld is .aligned
          tmem_ld_x16(tmem_base + lane_base + kDeltaCol + static_cast<uint32_t>(c), r16);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) dv[j] = __uint_as_float(r16[j]);
        }
        if (LP && !p.gated) {   // the down expand: added to the fp32 sum
#pragma unroll
          for (int j = 0; j < 16; ++j) val[j] += dv[j];
        }
        // transpose through the warp's buffer: lane = feature on the way in, then each lane
        // stores 4 consecutive features of a token (4 token rows of 128 B per instruction)
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 16; ++j) yb[j * 32 + lane] = val[j];
        __syncwarp();
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
        if (LP && p.gated) {   // the gate_up delta, rounded to bf16 on its own, logical columns
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 16; ++j) yb[j * 32 + lane] = dv[j];
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tok = (lane >> 3) + 4 * i;
            if (c + tok < nvalid) {
              const float4 v = *reinterpret_cast<const float4*>(yb + tok * 32 + f4);
              const float v4[4] = {v.x, v.y, v.z, v.w};
              *reinterpret_cast<uint2*>(p.d_out + static_cast<size_t>(q0 + c + tok) * p.N + dcol) = pack4(v4);
            }
          }
        }
      }
      if (LP && lmask) {
        tc_fence_before();
        mbar_arrive(dempty);   // the delta accumulator may take the next LoRA tile
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (*abort_flag) {   // let the MMAs lane 0 already issued finish before TMEM is released
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

template <int BN, bool LORA, bool LP = false>
static cudaError_t launch_fp8_bn(const GemmF8Params& p, int grid, cudaStream_t stream, bool pdl) {
  const int smem = gemm_fp8_smem_bytes(BN, p.stages, p.E, LORA ? p.slots.R : 0, LP ? 1 : 0);
  if (smem > kMaxGemmSmem) return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(grouped_gemm_fp8_kernel<BN, LORA, LP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  return launch_k(grouped_gemm_fp8_kernel<BN, LORA, LP>, dim3(grid), dim3(kF8Threads), static_cast<size_t>(smem),
                  stream, pdl, p);
}

cudaError_t launch_grouped_gemm_fp8(const GemmF8Params& p, int bn, int grid, cudaStream_t stream, bool pdl) {
  if (p.stages < 2 || p.stages > kF8MaxStages || grid < 1) return cudaErrorInvalidValue;
  if (p.N % 128 != 0 || p.K % 128 != 0) return cudaErrorInvalidValue;
  const bool lora = p.lora_v != nullptr;
  if (p.lora_packed) {   // packed LoRA stages (32- and 64-token tiles)
    if (lora) return cudaErrorInvalidValue;
    switch (bn) {
      case 32: return launch_fp8_bn<32, false, true>(p, grid, stream, pdl);
      case 64: return launch_fp8_bn<64, false, true>(p, grid, stream, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (bn) {
    case 16: return lora ? launch_fp8_bn<16, true>(p, grid, stream, pdl) : launch_fp8_bn<16, false>(p, grid, stream, pdl);
    case 32: return lora ? launch_fp8_bn<32, true>(p, grid, stream, pdl) : launch_fp8_bn<32, false>(p, grid, stream, pdl);
    case 64: return lora ? launch_fp8_bn<64, true>(p, grid, stream, pdl) : launch_fp8_bn<64, false>(p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mlk
