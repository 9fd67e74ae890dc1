// The NVFP4 path: per-row NVFP4 quantisation of the GEMM inputs, and a grouped GEMM over
// NVFP4 expert weights on the 5th-generation tensor cores.
//
// NVFP4 stores e2m1 values (sign, 2 exponent bits with bias 1, 1 mantissa bit: 0, 0.5, 1,
// 1.5, 2, 3, 4, 6) in blocks of 16 along K that share an e4m3 scale, times one float32 scale
// per tensor (per expert for the weights, per row for the activations).  It is the format of
// the pages' NVFP4 target checkpoint (sglang PR #27329, Optimizations: the Kimi-K2.5-NVFP4
// target, "modelopt_fp4" quantisation, activations quantised per token; for NVFP4 the
// permute and the down quantisation are fused with their neighbours).
//
// An e2m1 value times an e4m3 scale has at most 5 significant bits and lies in [2^-10, 2688],
// so it is exact in f16; so is the product of two such values in the fp32 accumulator.  The
// GEMM therefore decodes each weight block in shared memory to f16 (cvt e2m1x2 -> f16x2 and
// one multiply by the block's scale, both exact), takes the inputs as the same exact f16
// values from the quantiser, runs tcgen05.mma kind::f16 (f16 x f16 -> fp32), and applies the
// two float32 tensor scales in the epilogue.
//
// Warp roles (320 threads, persistent CTAs over a static tile list as in the bf16 GEMM):
//   warp 0      TMA producer: per raw stage the packed codes of four 64-wide K blocks (128
//               weight rows x 256 values = 16 KB, rows of 128 bytes with the 128-byte swizzle:
//               a TMA copy's cost follows its row count, so short rows would cap the stream)
//               and the f16 token rows of the four blocks (BN x 64 each, 128-byte swizzle):
//               the HBM stream of the kernel;
//   warps 6+    converters, G groups of 4 warps (G = 4, 2, 1 at token tiles of 16, 32, 64):
//               group g takes the K blocks n with n % G == g, and its thread c decodes weight row
//               c of the block into a ring of f16 weight tiles (the 128-byte swizzle of the
//               tcgen05 K-major layout); its row's 4 block scales per block come from global
//               memory by cp.async into a ring in shared memory, kNv4SfAhead of its blocks ahead;
//   warp 1      tcgen05.mma issuer (M = 128 weight rows from the f16 ring, N = BN tokens from
//               the raw stage, K = 64 per stage) and TMEM owner: two tiles' accumulators, each
//               as four partial sums (k-step kk of every block into partial kk), because the
//               MMAs into one accumulator wait for each other and a block's weight stream is
//               shorter than four such waits; its commit
//               frees the f16 tile, and after a raw stage's last block the raw stage (every
//               converter read of its codes came before that block's MMAs);
//   warps 2-5   epilogue: TMEM -> registers, the four partial sums added in a fixed order,
//               times the row scale and the expert scale, the
//               optional down-LoRA expand, a shared-memory transpose, 16-byte stores.
// Every mbarrier wait is bounded (2 s); a timeout records MOE_LORA_ERR_TIMEOUT, raises a
// CTA-wide abort flag, lets the copies already issued land and frees TMEM before returning.
// Every role but the MMA issuer waits suspended (try_wait with a time hint): 22 warps share
// the SM at 16-token tiles, and spinning waiters would take the issue slots the MMA warp needs.
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace mlk {

// Converter groups (4 warps each) by token tile: group g decodes the K blocks n with n % G == g,
// so G blocks are in conversion at once; the register budget of the larger tiles' epilogue
// leaves room for fewer groups.
__host__ __device__ constexpr int nv4_groups(int bn) { return bn <= 16 ? 4 : (bn <= 32 ? 2 : 1); }
__host__ __device__ constexpr int nv4_threads(int bn) { return 192 + 128 * nv4_groups(bn); }
constexpr int kNv4AByte = 128 * 128;       // 128 weight rows x 64 f16 values
constexpr int kNv4MaxStages = 8;
constexpr int kNv4MaxRStages = 32;
constexpr int kNv4YbufFloats = 16 * 32;    // per epilogue warp: 16 tokens x 32 features
constexpr uint64_t kNv4DrainNs = 20000000ull;   // 20 ms for the copies in flight to land
constexpr int kNv4SfAhead = 8;                  // K blocks of block scales in flight per converter

int gemm_nvfp4_stage_bytes(int bn) { (void)bn; return kNv4AByte; }
int gemm_nvfp4_rstage_bytes(int bn) { return kNv4RawStageBytes + kNv4RawBlocks * bn * 128; }

int gemm_nvfp4_smem_bytes(int bn, int stages, int rstages, int E, int lora_R) {
  // Carve-up, in order (see the kernel): 1 KB alignment slack; f16 weight stages; raw stages
  // (codes, then token rows); full/empty (2*stages), raw full/empty (2*rstages), accumulator
  // full/empty (4) and drain (1) barriers; tmem slot + abort flag (16 B); tile_start and seg
  // (E+1 ints each); for the LoRA epilogue BN token slots then BN x RP8 floats aligned to 16
  // bytes; the four epilogue warps' store buffers (16-byte aligned); the converter groups' rings
  // of block scales (kNv4SfAhead x 128 words each).
  const int lora = lora_R > 0 ? bn * 4 + 16 + bn * ((lora_R + 7) / 8 * 8) * 4 : 0;
  return 1024 + stages * gemm_nvfp4_stage_bytes(bn) + rstages * gemm_nvfp4_rstage_bytes(bn) +
         (2 * stages + 2 * rstages + 5) * 8 + 16 + 8 * (E + 1) + lora + 16 + 4 * kNv4YbufFloats * 4 +
         nv4_groups(bn) * kNv4SfAhead * 128 * 4;
}

// Instruction descriptor, kind::f16 with f16 inputs: D fp32 (bits 4-5 = 1), A and B f16 (bits
// 7-9 and 10-12 = 0), both K-major, N>>3 at bits 17-22, M>>4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

MLDEV void nv4_epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }   // the 4 epilogue warps

MLDEV void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
MLDEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
MLDEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// f16x2 of the two e2m1 codes of byte b (the low nibble in the low half), exact.
MLDEV __half2 e2m1x2_to_half2(uint32_t b) {
  const __half2_raw r = __nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>(b & 0xFFu), __NV_E2M1);
  return __half2(r);
}

// Down-LoRA expand of one 16-token chunk for output feature `feat` (this thread's weight
// row): val[j] += sum_{r < ranks[s]} lora_B[s, e, feat, r] * v_s[c + j][r] for each token j
// of the chunk whose pair has slot s = lslot[c + j] >= 0; v_s rows hold scaling[s] * (the
// down-LoRA shrink), RP8 floats each, zero past the slot's rank.
MLDEV void nv4_lora_expand(const GemmNv4Params& p, const int* lslot, const float* v_s, int c, int nvalid, int e,
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

template <int BN, bool LORA>
__global__ void __launch_bounds__(nv4_threads(BN), 1) grouped_gemm_nvfp4_kernel(const __grid_constant__ GemmNv4Params p) {
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 64, "token tiles of 16 to 64");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

  constexpr uint32_t OSTAGE = kNv4AByte;                          // one f16 weight tile
  constexpr uint32_t RSTAGE = kNv4RawStageBytes + kNv4RawBlocks * BN * 128;   // codes, then token rows
  constexpr int kParts = 4;                                       // partial sums per accumulator
  constexpr uint32_t ACC_COLS = kParts * BN;                      // one tile's accumulator
  constexpr uint32_t TMEM_COLS = 2 * ACC_COLS <= 128 ? 128u : (2 * ACC_COLS <= 256 ? 256u : 512u);
  constexpr int kGxLoads = (BN + 31) / 32;   // row scales of the tile's tokens per lane
  const int S = p.stages, RS = p.rstages;
  const int E = p.E;
  const int R = p.slots.R;
  const int RP8 = (R + 7) & ~7;

  uint8_t* raw = smem + S * OSTAGE;                               // [RS][codes 4 KB | tokens BN x 128 B]
  uint64_t* full = reinterpret_cast<uint64_t*>(raw + RS * RSTAGE);
  uint64_t* empty = full + S;
  uint64_t* rfull = empty + S;
  uint64_t* rempty = rfull + RS;
  uint64_t* tfull = rempty + RS;     // [2] accumulator ready (MMA commit)
  uint64_t* tempty = tfull + 2;      // [2] accumulator read (128 epilogue threads)
  uint64_t* drain = tempty + 2;      // [1], used only after an abort
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* tile_start = reinterpret_cast<int*>(tmem_slot + 4);   // [E + 1]
  int* seg = tile_start + (E + 1);                           // offsets copy [E + 1]
  int* lslot = seg + (E + 1);                                // [BN] (LoRA epilogue)
  float* v_s = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(lslot + (LORA ? BN : 0)) + 15) &
                                        ~static_cast<uintptr_t>(15));   // [BN][RP8] (LoRA epilogue)
  float* ybuf = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(v_s + (LORA ? BN * RP8 : 0)) + 15) &
                                         ~static_cast<uintptr_t>(15));  // [4][16][32]
  uint32_t* sf_ring = reinterpret_cast<uint32_t*>(ybuf + 4 * kNv4YbufFloats);   // [G][kNv4SfAhead][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta0 = static_cast<int>(blockIdx.x), ncta = static_cast<int>(gridDim.x);
  const int NT = p.N >> 7;   // 128-row weight tiles per expert
  const int KB = p.K >> 6;   // 64-wide K blocks (one f16 weight stage each)
  const int KR = (KB + kNv4RawBlocks - 1) / kNv4RawBlocks;   // raw stages per tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 4);    // the 4 converter warps
      mbar_init(&empty[s], 1);   // the MMA commit
    }
    for (int s = 0; s < RS; ++s) {
      mbar_init(&rfull[s], 1);    // the producer's expect_tx (codes and token rows)
      mbar_init(&rempty[s], 1);   // the MMA commit after the raw stage's last block
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmap_w);
    tma_prefetch_desc(&p.tmap_x);
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
  // weight row of tile row r (0..127): gate rows then up rows when gated
  auto weight_row = [&](int nt, int r) -> int {
    if (p.gated) return r < 64 ? nt * 64 + r : (p.N >> 1) + nt * 64 + (r - 64);
    return nt * 128 + r;
  };

  if (warp >= 2) pdl_wait();   // the epilogues read the previous kernel's row scales and LoRA rows
  if (warp == 0) {   // ------------------------------------------------ TMA producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    int rs = 0;
    uint32_t rph = 0;
    int ok = 1;
    int npre = 0, nissued = 0;   // stages whose codes went out before pdl_wait
    // raw stage s2 of K blocks [4 rk, 4 rk + 4): the codes of the tile's two 64-row halves
    auto load_codes = [&](int s2, int rk, int e, int nt) {
      uint8_t* dst = raw + s2 * RSTAGE;
      const int w0 = e * p.N + weight_row(nt, 0), w1 = e * p.N + weight_row(nt, 64);
      tma_load_2d(dst, &p.tmap_w, &rfull[s2], rk * 128, w0, pol_w);
      tma_load_2d(dst + 64 * 128, &p.tmap_w, &rfull[s2], rk * 128, w1, pol_w);
    };
    // The codes are constants of the layer and the tile schedule comes from the expert
    // offsets, so the first tile's first stages' codes go out before the previous kernel (which
    // writes the token rows) ends: their bytes are registered without an arrival, which comes
    // with the token rows' copies after the wait, so no phase completes early.
    if (lane == 0 && cta0 < total) {
      int e, nt, qt;
      decode(cta0, e, nt, qt);
      npre = min(RS, KR);
      for (int s2 = 0; s2 < npre; ++s2) {
        mbar_expect_tx(&rfull[s2], kNv4RawStageBytes);
        load_codes(s2, s2, e, nt);
      }
    }
    pdl_wait();
    if (lane == 0) {
      for (int tile = cta0; ok && tile < total; tile += ncta) {
        int e, nt, qt;
        decode(tile, e, nt, qt);
        const int xr = seg[e] + qt * BN;
        for (int rk = 0; ok && rk < KR; ++rk) {
          uint8_t* dst = raw + rs * RSTAGE;
          const int nsub = min(kNv4RawBlocks, KB - kNv4RawBlocks * rk);
          if (nissued++ >= npre) {
            if (!mbar_wait_sleep(&rempty[rs], rph ^ 1u, abort_flag, p.status, kWhereGemmProducer)) {
              ok = 0;
              break;
            }
            mbar_arrive_expect_tx(&rfull[rs], kNv4RawStageBytes + nsub * BN * 128);
            load_codes(rs, rk, e, nt);
          } else {
            mbar_arrive_expect_tx(&rfull[rs], nsub * BN * 128);
          }
          for (int j = 0; j < nsub; ++j)
            tma_load_2d(dst + kNv4RawStageBytes + j * BN * 128, &p.tmap_x, &rfull[rs],
                        (kNv4RawBlocks * rk + j) * 64, xr, pol_x);
          if (++rs == RS) {
            rs = 0;
            rph ^= 1u;
          }
        }
      }
    }
    pdl_trigger();   // all of this CTA's copies are issued: the next kernel may start
    if (lane == 0 && !ok) {   // drain: let the copies in flight land before the CTA exits
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < kNv4DrainNs) {
      }
    }
  } else if (warp >= 6) {   // ------------------------------------------ converters
    constexpr int G = nv4_groups(BN);
    const int grp = (warp - 6) >> 2;              // this thread's group
    const int ct = (threadIdx.x - 192) & 127;     // the tile row this thread decodes
    const int K16 = p.K >> 4;
    uint32_t* ring = sf_ring + grp * kNv4SfAhead * 128;
    bool ok = true;
    // the block scales of block n (this thread's row, 4 e4m3 codes, one word) go by cp.async
    // into slot (n / G) % kNv4SfAhead of the group's ring, kNv4SfAhead of the group's blocks
    // before block n is decoded; a cursor walks the group's block sequence that far ahead
    int la_n = grp, la_it = -1;
    const uint8_t* la_row = nullptr;   // this thread's scale row in the lookahead tile
    auto issue_ahead = [&](int slot) {
      const int it = la_n / KB, kb = la_n - it * KB;
      const int tile = cta0 + it * ncta;
      if (tile < total) {
        if (it != la_it) {   // (the tile lookup happens once per tile)
          int e, nt, qt;
          decode(tile, e, nt, qt);
          la_row = p.w_sf + (static_cast<size_t>(e) * p.N + weight_row(nt, ct)) * K16;
          la_it = it;
        }
        cp_async4(smem_u32(ring + slot * 128 + ct), la_row + kb * 4);
        la_n += G;
      }
      cp_async_commit();   // (an empty group past the end keeps the count)
    };
#pragma unroll 1
    for (int i = 0; i < kNv4SfAhead; ++i) issue_ahead(i);
    for (int n = grp, m = 0; ok; n += G, ++m) {   // block n, the group's m-th
      const int it = n / KB, kb = n - it * KB;
      if (cta0 + it * ncta >= total) break;
      const int j = kb % kNv4RawBlocks;                         // the block's place in its raw stage
      const int rg = it * KR + kb / kNv4RawBlocks;              // its raw stage, counted over the CTA
      const int rs = rg % RS, os = n % S;
      const uint32_t rph = static_cast<uint32_t>(rg / RS) & 1u, oph = static_cast<uint32_t>(n / S) & 1u;
      const int slot = m % kNv4SfAhead;
      cp_async_wait<kNv4SfAhead - 1>();   // the block's scales have landed
      const uint32_t sfw = ring[slot * 128 + ct];
      issue_ahead(slot);                  // the group's block kNv4SfAhead further into the slot just read
      if (!mbar_wait_sleep(&rfull[rs], rph, abort_flag, p.status, kWhereGemmProducer) ||
          !mbar_wait_sleep(&empty[os], oph ^ 1u, abort_flag, p.status, kWhereGemmProducer)) {
        ok = false;
        break;
      }
      uint8_t* ost = smem + os * OSTAGE;
      // row ct of the raw stage: 128 bytes, 16-byte chunk c stored at c ^ (ct & 7)
      const uint8_t* rrow = raw + rs * RSTAGE + ct * 128;
      const uint4 c0 = *reinterpret_cast<const uint4*>(rrow + (((2 * j) ^ (ct & 7)) << 4));
      const uint4 c1 = *reinterpret_cast<const uint4*>(rrow + (((2 * j + 1) ^ (ct & 7)) << 4));
      const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      // the 4 block scales as f16 pairs {s, s}
      const __half2 s01 = __half2(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(sfw & 0xFFFFu),
                                                             __NV_E4M3));
      const __half2 s23 = __half2(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(sfw >> 16),
                                                             __NV_E4M3));
      const __half2 sc[4] = {__low2half2(s01), __high2half2(s01), __low2half2(s23), __high2half2(s23)};
      uint8_t* arow = ost + ct * 128;
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) {   // 8 f16 values (4 code bytes) per 16-byte piece
        const uint32_t w = words[pc];
        const __half2 sb = sc[pc >> 1];
        __half2 h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __hmul2(e2m1x2_to_half2(w >> (8 * i)), sb);
        uint4 v;
        v.x = *reinterpret_cast<const uint32_t*>(&h[0]);
        v.y = *reinterpret_cast<const uint32_t*>(&h[1]);
        v.z = *reinterpret_cast<const uint32_t*>(&h[2]);
        v.w = *reinterpret_cast<const uint32_t*>(&h[3]);
        *reinterpret_cast<uint4*>(arow + ((pc ^ (ct & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();   // the f16 tile is read by tcgen05.mma (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[os]);
    }
    cp_async_wait<0>();   // no scale copy is left in flight when the CTA exits
  } else if (warp == 1) {   // ------------------------------------------ MMA issuer (lane 0)
    constexpr uint32_t idesc = idesc_f16_f32(128, BN);
    if (lane == 0) {
      int os = 0, rs = 0, acc = 0;
      uint32_t oph = 0, rph = 0, aph = 0;
      bool ok = true;
      for (int tile = cta0; ok && tile < total; tile += ncta) {
        if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, p.status, kWhereGemmMma)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * ACC_COLS);
        for (int kb = 0; kb < KB; ++kb) {
          const int j = kb % kNv4RawBlocks;
          if (!mbar_wait(&full[os], oph, abort_flag, p.status, kWhereGemmMma) ||
              (j == 0 && !mbar_wait(&rfull[rs], rph, abort_flag, p.status, kWhereGemmMma))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sw128_kmajor_desc(smem_u32(smem + os * OSTAGE));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(raw + rs * RSTAGE + kNv4RawStageBytes + j * BN * 128));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)   // K = 16 f16 values = 32 bytes = 2 descriptor units
            umma_bf16(d + kk * BN, ad + 2 * kk, bd + 2 * kk, idesc, kb != 0 ? 1u : 0u);
          umma_commit(&empty[os]);    // the f16 weight tile is free
          if (j == kNv4RawBlocks - 1 || kb == KB - 1) {
            umma_commit(&rempty[rs]);   // the token rows are read (the codes were, by the converters)
            if (++rs == RS) {
              rs = 0;
              rph ^= 1u;
            }
          }
          if (++os == S) {
            os = 0;
            oph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          aph ^= 1u;
        }
      }
    }
  } else {   // -------------------------------------------------------------- epilogue (warps 2-5)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // weight row inside the tile == TMEM lane
    const int etid = threadIdx.x - 64;     // 0..127 over the epilogue warps
    float* yb = ybuf + quarter * kNv4YbufFloats;
    const int f4 = (lane & 7) * 4;         // the 4 features this lane stores per token row
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int acc = 0;
    uint32_t aph = 0;
    for (int tile = cta0; tile < total; tile += ncta) {
      int e, nt, qt;
      decode(tile, e, nt, qt);
      const int q0 = seg[e] + qt * BN;
      const int nvalid = min(BN, seg[e + 1] - q0);
      if constexpr (LORA) {   // stage the tile's pair slots and scaled down-LoRA shrink values
        nv4_epi_bar();
        for (int j = etid; j < nvalid; j += 128) lslot[j] = p.pair_slot[q0 + j];
        nv4_epi_bar();
        for (int i = etid; i < nvalid * RP8; i += 128) {
          const int j = i / RP8, r = i - j * RP8;
          const int sl = lslot[j];
          v_s[i] = (sl >= 0 && r < p.slots.ranks[sl]) ? p.lora_v[static_cast<size_t>(q0 + j) * R + r] : 0.0f;
        }
        nv4_epi_bar();
      }
      // token j's row scale from lane j % 32 (zero past the tile's tokens), the expert's scale
      float gxl[kGxLoads];
#pragma unroll
      for (int u = 0; u < kGxLoads; ++u) {
        const int j = lane + 32 * u;
        gxl[u] = (j < nvalid) ? p.x_gs[q0 + j] : 0.0f;
      }
      const float gw = __ldg(p.w_gs + e);
      if (!mbar_wait_sleep(&tfull[acc], aph, abort_flag, p.status, kWhereGemmEpilogue)) break;
      tc_fence_after();
      __syncwarp();   // the lanes left the barrier wait one by one: tcgen05.ld is .aligned
      // the four partial sums, added as (p0 + p1) + (p2 + p3)
      float r[BN / 16][16];
#pragma unroll
      for (int c = 0; c < BN / 16; ++c) {
        uint32_t q[kParts][16];
#pragma unroll
        for (int pp = 0; pp < kParts; ++pp)
          tmem_ld_x16(tmem_base + lane_base + static_cast<uint32_t>(acc * ACC_COLS + pp * BN + 16 * c), q[pp]);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          r[c][i] = (__uint_as_float(q[0][i]) + __uint_as_float(q[1][i])) +
                    (__uint_as_float(q[2][i]) + __uint_as_float(q[3][i]));
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);   // the accumulator may take the next tile's MMAs
      if (++acc == 2) {
        acc = 0;
        aph ^= 1u;
      }
      const int col = nt * 128 + row;   // output column of this thread's row
      const int fcol = nt * 128 + quarter * 32 + f4;
#pragma unroll
      for (int c = 0; c < BN; c += 16) {
        if (c >= nvalid) break;   // warp-uniform
        float val[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float gx = __shfl_sync(0xffffffffu, gxl[(c + j) >> 5], (c + j) & 31);
          val[j] = r[c >> 4][j] * __fmul_rn(gx, gw);
        }
        if constexpr (LORA) nv4_lora_expand(p, lslot, v_s, c, nvalid, e, col, val);
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

template <int BN, bool LORA>
static cudaError_t launch_nv4_bn(const GemmNv4Params& p, int grid, cudaStream_t stream, bool pdl) {
  const int smem = gemm_nvfp4_smem_bytes(BN, p.stages, p.rstages, p.E, LORA ? p.slots.R : 0);
  if (smem > kMaxGemmSmem) return cudaErrorInvalidValue;
  cudaError_t err =
      cudaFuncSetAttribute(grouped_gemm_nvfp4_kernel<BN, LORA>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  return launch_k(grouped_gemm_nvfp4_kernel<BN, LORA>, dim3(grid), dim3(nv4_threads(BN)), static_cast<size_t>(smem),
                  stream, pdl, p);
}

cudaError_t launch_grouped_gemm_nvfp4(const GemmNv4Params& p, int bn, int grid, cudaStream_t stream, bool pdl) {
  if (p.stages < 2 || p.stages > kNv4MaxStages || p.rstages < 2 || p.rstages > kNv4MaxRStages || grid < 1)
    return cudaErrorInvalidValue;
  if (p.N % 128 != 0 || p.K % 64 != 0) return cudaErrorInvalidValue;
  // The converter groups wait on the f16 stages' barriers by phase parity: a group may run up to
  // G - 1 blocks ahead of the slowest, so fewer than G stages would let two waiters of one
  // barrier be two phases apart.
  if (p.stages < nv4_groups(bn)) return cudaErrorInvalidValue;
  const bool lora = p.lora_v != nullptr;
  switch (bn) {
    case 16: return lora ? launch_nv4_bn<16, true>(p, grid, stream, pdl) : launch_nv4_bn<16, false>(p, grid, stream, pdl);
    case 32: return lora ? launch_nv4_bn<32, true>(p, grid, stream, pdl) : launch_nv4_bn<32, false>(p, grid, stream, pdl);
    case 64: return lora ? launch_nv4_bn<64, true>(p, grid, stream, pdl) : launch_nv4_bn<64, false>(p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
  }
}

// ---------------------------------------------------------------------------------
// NVFP4 quantisation of rows, one warp per row (the pages' per-token activation quantisation
// for NVFP4, fused with the permute for the gate_up input and run on the activation for the
// down input).  Per row, all float32 operations rounded to nearest:
//   g = max(amax, 1e-10) / 2688                                  (2688 = 6 * 448)
//   per 16 values: s = e4m3(amax_16 / (6 * g)), rounded to nearest even, saturated at 448
//   q = e2m1(v / (s * g)), rounded to nearest even on the e2m1 grid, saturated at 6 (0 where
//   s * g is 0)
// The row is read twice (its maximum first; the second pass hits L2).
// ---------------------------------------------------------------------------------

// Nearest e2m1 value of x (ties to the even mantissa, saturating at 6) and its 4-bit code.
// Below 1 the grid step is 0.5, in [2^e, 2^(e+1)) it is 2^(e-1): the magnitude divided by its
// step, rounded to nearest even, times the step.
MLDEV float nv4_round_e2m1(float x, uint32_t& code) {
  const float ax = fabsf(x);
  const int ex = static_cast<int>((__float_as_uint(ax) >> 23) & 0xFFu) - 127;   // floor(log2) of a normal
  const int e = ex > 0 ? (ex < 3 ? ex : 3) : 0;                                  // steps 0.5, 0.5, 1, 2
  const float step = __uint_as_float(static_cast<uint32_t>(e - 1 + 127) << 23);
  const float inv = __uint_as_float(static_cast<uint32_t>(1 - e + 127) << 23);
  float m = fminf(rintf(__fmul_rn(ax, inv)) * step, 6.0f);
  // m * 2 is one of 0, 1, 2, 3, 4, 6, 8, 12: the code's magnitude index 0..7
  const int m2 = static_cast<int>(m * 2.0f);
  const uint32_t idx = m2 <= 4 ? static_cast<uint32_t>(m2) : (m2 == 6 ? 5u : (m2 == 8 ? 6u : 7u));
  const bool neg = (__float_as_uint(x) >> 31) != 0;
  code = idx | (neg ? 8u : 0u);
  return neg ? -m : m;
}

__global__ void __launch_bounds__(256) quant_nvfp4_kernel(const __nv_bfloat16* __restrict__ src,
                                                          const int32_t* __restrict__ perm, int k, int P, int K,
                                                          float* __restrict__ g_out, __half* __restrict__ deq,
                                                          uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                          const int32_t* __restrict__ slot_idx, int32_t* slot_out) {
  pdl_wait();
  pdl_trigger();
  const int q = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (q >= P) return;
  const int t = perm != nullptr ? perm[q] / k : q;
  if (slot_out != nullptr && lane == 0) slot_out[q] = slot_idx[t];
  const uint4* s = reinterpret_cast<const uint4*>(src + static_cast<size_t>(t) * K);
  const int NB = K >> 4;   // blocks of 16 values
  float amax = 0.0f;
  for (int b = lane; b < NB; b += 32) {
    float f[16];
    unpack8(__ldg(s + 2 * b), *reinterpret_cast<float(*)[8]>(f));
    unpack8(__ldg(s + 2 * b + 1), *reinterpret_cast<float(*)[8]>(f + 8));
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float g = __fdiv_rn(fmaxf(amax, 1e-10f), 2688.0f);
  const float six_g = __fmul_rn(6.0f, g);
  if (lane == 0) g_out[q] = g;
  for (int b = lane; b < NB; b += 32) {
    float f[16];
    unpack8(__ldg(s + 2 * b), *reinterpret_cast<float(*)[8]>(f));
    unpack8(__ldg(s + 2 * b + 1), *reinterpret_cast<float(*)[8]>(f + 8));
    float ab = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(f[i]));
    const __nv_fp8_storage_t sc = __nv_cvt_float_to_fp8(__fdiv_rn(ab, six_g), __NV_SATFINITE, __NV_E4M3);
    const float sbf = __half2float(__half(__nv_cvt_fp8_to_halfraw(sc, __NV_E4M3)));
    const float eff = __fmul_rn(sbf, g);
    float qv[16];
    uint32_t cd[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (eff > 0.0f) {
        qv[i] = nv4_round_e2m1(__fdiv_rn(f[i], eff), cd[i]);
      } else {
        qv[i] = 0.0f;
        cd[i] = 0u;
      }
    }
    const size_t o = static_cast<size_t>(q) * K + static_cast<size_t>(b) * 16;
    if (deq != nullptr) {   // q * s: exact in f16
      uint32_t hw[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const __half2 h2 = __floats2half2_rn(qv[2 * i] * sbf, qv[2 * i + 1] * sbf);
        hw[i] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      uint4* d = reinterpret_cast<uint4*>(deq + o);
      d[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      d[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
    }
    if (codes != nullptr) {   // element 2i in the low nibble of byte i
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        lo |= (cd[2 * i] | (cd[2 * i + 1] << 4)) << (8 * i);
        hi |= (cd[8 + 2 * i] | (cd[8 + 2 * i + 1] << 4)) << (8 * i);
      }
      *reinterpret_cast<uint2*>(codes + o / 2) = make_uint2(lo, hi);
    }
    if (sf != nullptr) sf[static_cast<size_t>(q) * NB + b] = sc;
  }
}

cudaError_t launch_quant_nvfp4(const __nv_bfloat16* src, const int32_t* perm, int k, int P, int K, float* g,
                               __half* deq, uint8_t* codes, uint8_t* sf, cudaStream_t stream, bool pdl,
                               const int32_t* slot_idx, int32_t* slot_out) {
  if (P == 0) return cudaSuccess;
  if (K % 16 != 0) return cudaErrorInvalidValue;
  return launch_k(quant_nvfp4_kernel, dim3((P + 7) / 8), dim3(256), 0, stream, pdl, src, perm, k, P, K, g, deq, codes,
                  sf, slot_idx, slot_out);
}

// ---------------------------------------------------------------------------------
// Narrow token tiles (decode: a handful of tokens per expert).  A tile is 128 weight rows of
// one expert x up to 16 of its tokens; each of the 8 warps takes 16 of the rows.  A warp streams
// its rows' codes and scales one 256-value K region at a time (128 code bytes and 16 scale bytes
// per row) through its own ring of kNv4nRing regions in shared memory, with 16-byte cp.async
// copies issued kNv4nRing regions ahead; the stream runs on across the warp's tiles, so the
// next tile's first regions are in flight while this tile finishes.  Each thread decodes its own
// A-fragment values from the ring (cvt e2m1x2 -> f16x2, times the block's e4m3 scale: exact in
// f16) and multiplies on mma.sync m16n8k16 (f16 in, fp32 accumulate) against the tokens' f16
// rows, staged per 1024-value K chunk in shared memory in B-fragment order (one conflict-free
// 8-byte read per lane and MMA).  Within a region thread (g, t) of the warp (g = lane / 4,
// t = lane % 4) takes bytes 32t .. 32t+31 (codes 64t .. 64t+63) of rows g and g+8 (16-byte
// chunks 2t and 2t+1; chunk c of row r sits at chunk c ^ (r % 8) of its 128-byte ring row, so
// that neither the copies nor the reads conflict).  MMA step j (0..15) uses codes
// 64t + 4j .. +3: its k indices 2t, 2t+1 stand for K offsets 64t + 4j, +1 and 2t+8, 2t+9 for
// 64t + 4j + 2, +3; the tokens' B fragments take the same offsets, so the sum over K is the
// same sum.  The four codes of a step lie in 16-value block 4t + j/4 of the row: one scale.
constexpr int kNv4nThreads = 256;   // 8 warps x 16 rows = one 128-row weight tile
constexpr int kNv4nTok = 16;        // tokens per tile: two 8-token MMA column blocks
constexpr int kNv4nKC = 1024;      // K values of the token rows staged in shared memory at a time
static_assert(kNv4nKC / 4 == kNv4nThreads, "one 8-byte piece of each token row per thread");
constexpr int kNv4nPieces = kNv4nKC / 256 * 16 * 32;   // 8-byte B pieces of one 8-token block and K chunk
constexpr int kNv4nRing = 3;        // regions in flight per warp (shared-memory ring)
constexpr int kNv4nSlot = 16 * 128 + 16 * 16;   // one region of a warp's 16 rows: codes, then scales
constexpr int kNv4nSmem = 2 * kNv4nPieces * 8 + (kNv4nThreads / 32) * kNv4nRing * kNv4nSlot;

MLDEV void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// s[i] = {v, v} for v the e4m3 code in byte i of w, exact in f16
MLDEV void e4m3x4_to_half2_bcast(uint32_t w, __half2 (&s)[4]) {
  const __half2 lo(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFFu), __NV_E4M3));
  const __half2 hi(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3));
  s[0] = __low2half2(lo);
  s[1] = __high2half2(lo);
  s[2] = __low2half2(hi);
  s[3] = __high2half2(hi);
}

// f16x2 values of the 8 e2m1 codes of w: h[i] holds the codes of byte i (low nibble in the low
// half), exact
MLDEV void e2m1x8_to_half2x4(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
      "mov.b32 {c0, c1, c2, c3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, c0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, c1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, c2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, c3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

MLDEV uint32_t hmul2_bits(uint32_t a, __half2 s) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), s);
  return *reinterpret_cast<const uint32_t*>(&r);
}

MLDEV void prefetch_l2(const void* ptr) { asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr)); }

// The down-LoRA expand of one 8-token column block c of a narrow tile for this thread (tokens
// 8c + 2t + i, slots ts[i], negative: none; weight rows n0, n1), rows of R = 8 NC values:
// ls[i][half] = sum_{r < ranks[s]} lora_B[s, e, n, r] * lora_v[q, r], in order of r.  Every
// load is issued first (from a valid row for a token without a slot, whose rank counts as 0).
template <int NC>
MLDEV void nv4n_lora_expand(const GemmNv4Params& p, int e, int q0, int c, int t, int n0, int n1, const int (&ts)[2],
                            float (&ls)[2][2]) {
  const int R = 8 * NC, N = p.N;
  uint4 bw[2][2][NC];
  float4 vv[2][2 * NC];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int s = ts[i] >= 0 ? ts[i] : 0;
    const int q = q0 + (ts[i] >= 0 ? 8 * c + 2 * t + i : 0);
    const size_t be = p.lora_b_e1 ? static_cast<size_t>(s) : static_cast<size_t>(s) * p.E + e;
    const float4* vq = reinterpret_cast<const float4*>(p.lora_v + static_cast<size_t>(q) * R);
#pragma unroll
    for (int h = 0; h < 2 * NC; ++h) vv[i][h] = __ldg(vq + h);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint4* Brow = reinterpret_cast<const uint4*>(p.lora_B + (be * N + (hh == 0 ? n0 : n1)) * R);
#pragma unroll
      for (int ch = 0; ch < NC; ++ch) bw[i][hh][ch] = __ldg(Brow + ch);
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int rank = ts[i] >= 0 ? p.slots.ranks[ts[i]] : 0;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float sum = 0.0f;
#pragma unroll
      for (int ch = 0; ch < NC; ++ch) {
        float bv[8];
        unpack8(bw[i][hh][ch], bv);
        const float v8[8] = {vv[i][2 * ch].x,     vv[i][2 * ch].y,     vv[i][2 * ch].z,     vv[i][2 * ch].w,
                             vv[i][2 * ch + 1].x, vv[i][2 * ch + 1].y, vv[i][2 * ch + 1].z, vv[i][2 * ch + 1].w};
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (8 * ch + u < rank) sum = fmaf(bv[u], v8[u], sum);
      }
      ls[i][hh] = sum;
    }
  }
}

MLDEV void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

template <bool LORA>
__global__ void __launch_bounds__(kNv4nThreads, 2) grouped_gemm_nvfp4_narrow_kernel(
    const __grid_constant__ GemmNv4Params p) {
  __shared__ int tile_start[kMaxExperts + 1];
  __shared__ int seg[kMaxExperts + 1];
  // dynamic: the tile's token rows for one K chunk in B-fragment order (two 8-token blocks:
  // 8-byte piece (region r, step j, token g, t) holds K offsets 256 r + 64t + 4j .. +3), then
  // each warp's ring of regions (its 16 rows' codes, 128-byte swizzled, then their scales)
  extern __shared__ __align__(128) uint8_t nsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  uint2* sB0 = reinterpret_cast<uint2*>(nsm);
  uint2* sB1 = sB0 + kNv4nPieces;
  uint8_t* ring = nsm + 2 * kNv4nPieces * 8 + warp * kNv4nRing * kNv4nSlot;
  const uint32_t ring_s = smem_u32(ring);
  const int E = p.E, N = p.N, K = p.K;
  const int NT = N >> 7;    // 128-row weight tiles per expert
  const int NR = K >> 8;    // 256-value K regions per row
  pdl_wait();   // the f16 inputs and their row scales come from the previous kernel
  pdl_trigger();
  if (warp == 0) build_tile_schedule(p.offsets, E, kNv4nTok, NT, seg, tile_start);
  __syncthreads();
  const int total = tile_start[E];
  auto decode = [&](int tile, int& e, int& nt, int& qt) {
    int lo = 0, hi = E - 1;   // last expert with tile_start <= tile (empty experts skipped)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int local = tile - tile_start[e];
    const int nq = (seg[e + 1] - seg[e] + kNv4nTok - 1) / kNv4nTok;
    nt = local / nq;
    qt = local - nt * nq;
  };
  auto weight_row = [&](int nt, int r) {   // the weight row of row r of tile nt
    return p.gated ? (r < 64 ? nt * 64 + r : (N >> 1) + nt * 64 + r - 64) : nt * 128 + r;
  };
  // ---- the warp's stream of regions over its tiles, copied kNv4nRing regions ahead: lane l
  // copies 16-byte chunks l, l+32, l+64, l+96 of a region's 16 rows x 128 bytes (row 4i + l/8,
  // chunk l % 8) and, lanes 0..15, the 16 scale bytes of row l
  int is_tile = blockIdx.x, is_r = 0;
  const uint8_t* cbase[4];
  const uint8_t* sbase = nullptr;
  auto issue_rows = [&](int tile) {
    int e, nt, qt;
    decode(tile, e, nt, qt);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      cbase[i] = p.w_codes + (static_cast<size_t>(e) * N + weight_row(nt, warp * 16 + 4 * i + (lane >> 3))) *
                                 (K >> 1);
    sbase = p.w_sf + (static_cast<size_t>(e) * N + weight_row(nt, warp * 16 + (lane & 15))) * (K >> 4);
  };
  int islot = 0;   // ring slot of the next region copied
  auto issue_next = [&]() {
    if (is_tile < total) {
      const uint32_t dst = ring_s + static_cast<uint32_t>(islot * kNv4nSlot);
      const int c = lane & 7;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = 4 * i + (lane >> 3);
        cp_async16(dst + row * 128 + ((c ^ (row & 7)) << 4), cbase[i] + is_r * 128 + c * 16);
      }
      if (lane < 16) cp_async16(dst + 2048 + lane * 16, sbase + is_r * 16);
      if (++is_r == NR) {
        is_r = 0;
        is_tile += gridDim.x;
        if (is_tile < total) issue_rows(is_tile);
      }
    }
    cp_async_commit();   // an empty group past the end keeps one group per region
    if (++islot == kNv4nRing) islot = 0;
  };
  if (is_tile < total) issue_rows(is_tile);
#pragma unroll 1
  for (int d = 0; d < kNv4nRing; ++d) issue_next();
  int cslot = 0;   // ring slot of the next region used

  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    int e, nt, qt;
    decode(tile, e, nt, qt);
    const int q0 = seg[e] + qt * kNv4nTok;
    const int nvalid = min(kNv4nTok, seg[e + 1] - q0);
    const bool tv1 = nvalid > 8;   // the second 8-token column block has tokens (warp-uniform)
    // this thread's two weight rows (tile rows r0, r1; weight rows n0, n1)
    const int r0 = warp * 16 + g, r1 = r0 + 8;
    const int n0 = weight_row(nt, r0), n1 = weight_row(nt, r1);
    float acc0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    // the down-LoRA slots of this thread's tokens 8c + 2t + i (negative: none); their B and v
    // rows are prefetched into L2 once the first K chunk is staged and read in the epilogue
    int tslot[2][2] = {{-1, -1}, {-1, -1}};
    if constexpr (LORA) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int j = 8 * c + 2 * t + i;
          if (j < nvalid) {
            const int sl = __ldg(p.pair_slot + q0 + j);
            tslot[c][i] = sl < p.slots.S ? sl : -1;
          }
        }
      }
    }
    for (int kc0 = 0; kc0 < K; kc0 += kNv4nKC) {
      const int kcl = min(kNv4nKC, K - kc0);   // a multiple of 256
      const int npc = kcl >> 2;                 // 8-byte pieces per token row
      __syncthreads();   // every warp is done with the previous chunk's rows
      // thread c stages piece c (K offsets kc0 + 4c .. +3) of each of the tile's token rows, per
      // 8-token block all loads first; rows past the tile's tokens are not staged: their
      // accumulator columns are never stored
      if (threadIdx.x < npc) {
        const int c = threadIdx.x;
        const int so = (((c >> 6) * 16 + (c & 15)) * 8) * 4 + ((c >> 4) & 3);
        const uint2* src = reinterpret_cast<const uint2*>(p.x16 + static_cast<size_t>(q0) * K + kc0) + c;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          if (blk == 1 && !tv1) break;
          uint2* sB = blk == 0 ? sB0 : sB1;
          uint2 v[8];
#pragma unroll
          for (int tok = 0; tok < 8; ++tok)
            if (8 * blk + tok < nvalid) v[tok] = __ldg(src + static_cast<size_t>(8 * blk + tok) * (K >> 2));
#pragma unroll
          for (int tok = 0; tok < 8; ++tok)
            if (8 * blk + tok < nvalid) sB[so + tok * 4] = v[tok];
        }
      }
      __syncthreads();
      if constexpr (LORA) {
        if (kc0 == 0) {
          const int R = p.slots.R;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int sl = tslot[c][i];
              if (sl < 0) continue;
              const size_t be = p.lora_b_e1 ? static_cast<size_t>(sl) : static_cast<size_t>(sl) * E + e;
              prefetch_l2(p.lora_B + (be * N + n0) * R);
              prefetch_l2(p.lora_B + (be * N + n1) * R);
              prefetch_l2(p.lora_v + static_cast<size_t>(q0 + 8 * c + 2 * t + i) * R);
            }
          }
        }
      }
      const int nrg = kcl >> 8;
#pragma unroll 1
      for (int rl = 0; rl < nrg; ++rl) {
        cp_async_wait<kNv4nRing - 1>();   // this thread's copies of the oldest region have landed
        __syncwarp();                     // ... and every lane's
        const uint8_t* sl = ring + cslot * kNv4nSlot;
        // this thread's 32 code bytes of rows g and g+8 (chunks 2t, 2t+1; rows g and g+8 share
        // the swizzle) and the scales of its four blocks of 16
        const int x0 = ((2 * t) ^ (g & 7)) << 4, x1 = ((2 * t + 1) ^ (g & 7)) << 4;
        const uint4 cl0 = *reinterpret_cast<const uint4*>(sl + g * 128 + x0);
        const uint4 ch0 = *reinterpret_cast<const uint4*>(sl + g * 128 + x1);
        const uint4 cl1 = *reinterpret_cast<const uint4*>(sl + (g + 8) * 128 + x0);
        const uint4 ch1 = *reinterpret_cast<const uint4*>(sl + (g + 8) * 128 + x1);
        const uint32_t sw0 = *reinterpret_cast<const uint32_t*>(sl + 2048 + g * 16 + 4 * t);
        const uint32_t sw1 = *reinterpret_cast<const uint32_t*>(sl + 2048 + (g + 8) * 16 + 4 * t);
        __syncwarp();   // every lane has read the slot: it takes the next region
        issue_next();
        if (++cslot == kNv4nRing) cslot = 0;
        __half2 sc0[4], sc1[4];   // the block scales of rows g and g+8, one per 16 values
        e4m3x4_to_half2_bcast(sw0, sc0);
        e4m3x4_to_half2_bcast(sw1, sc1);
        const uint2* b0p = sB0 + rl * 16 * 32 + lane;
        const uint2* b1p = sB1 + rl * 16 * 32 + lane;
        // the region's 16 MMA steps, with the second 8-token block or without it
        auto steps = [&](auto two) {
#pragma unroll
          for (int w = 0; w < 8; ++w) {   // word w: steps 2w and 2w + 1
            const uint4& qa = w < 4 ? cl0 : ch0;
            const uint4& qb = w < 4 ? cl1 : ch1;
            const int ww = w & 3;
            uint32_t ha[4], hb[4];
            e2m1x8_to_half2x4(ww == 0 ? qa.x : ww == 1 ? qa.y : ww == 2 ? qa.z : qa.w, ha);
            e2m1x8_to_half2x4(ww == 0 ? qb.x : ww == 1 ? qb.y : ww == 2 ? qb.z : qb.w, hb);
            const __half2 s0 = sc0[w >> 1], s1 = sc1[w >> 1];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int j = 2 * w + u;
              uint32_t a[4];
              a[0] = hmul2_bits(ha[2 * u], s0);       // row g,   k 2t, 2t+1
              a[1] = hmul2_bits(hb[2 * u], s1);       // row g+8, k 2t, 2t+1
              a[2] = hmul2_bits(ha[2 * u + 1], s0);   // row g,   k 2t+8, 2t+9
              a[3] = hmul2_bits(hb[2 * u + 1], s1);   // row g+8, k 2t+8, 2t+9
              const uint2 b0 = b0p[j * 32];
              mma_f16_16816(acc0, a, b0.x, b0.y);
              if constexpr (decltype(two)::value) {
                const uint2 b1 = b1p[j * 32];
                mma_f16_16816(acc1, a, b1.x, b1.y);
              }
            }
          }
        };
        if (tv1) steps(std::true_type{});
        else steps(std::false_type{});
      }
    }
    // epilogue: accumulator (row, token) = acc_c[2 * half + i] for row g (+8 when half = 1),
    // token 8c + 2t + i; times the token's and the expert's scales, plus the down-LoRA expand
    // lsum[c][i][half] = sum_{r < ranks[s]} lora_B[s, e, n, r] * lora_v[q, r] (s = pair_slot[q]),
    // summed in order of r; for rows of 8 or 16 values all loads are issued before the sums
    float lsum[2][2][2] = {{{0.0f, 0.0f}, {0.0f, 0.0f}}, {{0.0f, 0.0f}, {0.0f, 0.0f}}};
    if constexpr (LORA) {
      const int R = p.slots.R;
      const bool al = ((reinterpret_cast<uintptr_t>(p.lora_B) | reinterpret_cast<uintptr_t>(p.lora_v)) & 15u) == 0;
      if (al && R == 16) {
        nv4n_lora_expand<2>(p, e, q0, 0, t, n0, n1, tslot[0], lsum[0]);
        if (tv1) nv4n_lora_expand<2>(p, e, q0, 1, t, n0, n1, tslot[1], lsum[1]);
      } else if (al && R == 8) {
        nv4n_lora_expand<1>(p, e, q0, 0, t, n0, n1, tslot[0], lsum[0]);
        if (tv1) nv4n_lora_expand<1>(p, e, q0, 1, t, n0, n1, tslot[1], lsum[1]);
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int sl = tslot[c][i];
            if (sl < 0) continue;
            const int q = q0 + 8 * c + 2 * t + i, rank = p.slots.ranks[sl];
            const size_t be = p.lora_b_e1 ? static_cast<size_t>(sl) : static_cast<size_t>(sl) * E + e;
            const float* vq = p.lora_v + static_cast<size_t>(q) * R;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const __nv_bfloat16* Brow = p.lora_B + (be * N + (hh == 0 ? n0 : n1)) * static_cast<size_t>(R);
              float sum = 0.0f;
              for (int r = 0; r < rank; ++r) sum = fmaf(bf2f(Brow[r]), __ldg(vq + r), sum);
              lsum[c][i][hh] = sum;
            }
          }
        }
      }
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int j = 8 * c + 2 * t + i;
        if (j >= nvalid) continue;
        const int q = q0 + j;
        const float sc = __fmul_rn(__ldg(p.x_gs + q), __ldg(p.w_gs + e));
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float val = (c == 0 ? acc0[2 * hh + i] : acc1[2 * hh + i]) * sc;
          if constexpr (LORA) val += lsum[c][i][hh];
          const int col = nt * 128 + (hh == 0 ? r0 : r1);   // the output's column order (gated: interleaved)
          const size_t off = static_cast<size_t>(q) * N + col;
          if (p.out_f32 != nullptr) p.out_f32[off] = val;
          else p.out[off] = __float2bfloat16_rn(val);
        }
      }
    }
  }
}

cudaError_t launch_grouped_gemm_nvfp4_narrow(const GemmNv4Params& p, int grid, cudaStream_t stream, bool pdl) {
  if (grid < 1 || p.N % 128 != 0 || p.K % 256 != 0 || p.w_codes == nullptr || p.x16 == nullptr ||
      (reinterpret_cast<uintptr_t>(p.w_codes) & 15u) != 0 || (reinterpret_cast<uintptr_t>(p.w_sf) & 15u) != 0)
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(grouped_gemm_nvfp4_narrow_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kNv4nSmem);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(grouped_gemm_nvfp4_narrow_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kNv4nSmem);
  if (err != cudaSuccess) return err;
  if (p.lora_v != nullptr)
    return launch_k(grouped_gemm_nvfp4_narrow_kernel<true>, dim3(grid), dim3(kNv4nThreads), kNv4nSmem, stream, pdl, p);
  return launch_k(grouped_gemm_nvfp4_narrow_kernel<false>, dim3(grid), dim3(kNv4nThreads), kNv4nSmem, stream, pdl, p);
}

}  // namespace mlk
