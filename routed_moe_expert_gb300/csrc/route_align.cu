// Fused routing + expert alignment, one launch.
//
// Phase 1: each warp selects the top-k experts of 4 tokens at a time (warp arg-max
//          rounds, ties to the lower expert id, the 4 tokens interleaved) and the routing
//          weights; each CTA counts its pairs per expert in shared memory.
// Phase 2: (grid barrier) per expert, an exclusive prefix of the per-CTA counts over
//          the CTAs in order; (grid barrier) every CTA scans the expert totals into
//          expert_offsets, then scatters its own pairs, in ascending expanded index,
//          to perm / inv_perm.  Because every CTA owns a contiguous token range and
//          the per-CTA bases are prefixes in CTA order, the permutation is the unique
//          "by expert, then by expanded index" order.
//
// Stage references: sglang PR #27329 "Experimental fast LoRA path", Optimizations
// ("topk + FlashInfer routed-pack in a single launch", "JIT MoE-align"); the routing
// methods of the vLLM API page "fused_moe/experts/trtllm_lora_moe"
// (_supports_routing_method: Renormalize, DeepSeekV3).
//
// With more than one CTA the kernel is launched cooperatively (all CTAs resident), and
// each grid barrier is a bounded spin: after 2 s it records MOE_LORA_ERR_TIMEOUT in the
// status word and the kernel returns.
#include "common.cuh"
#include "kernels.h"

namespace mlk {

constexpr int kRouteThreads = 512;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kInvalidId = 0x7fffffff;
constexpr int kRouteIdsInSmem = 3072;   // pairs per CTA kept in shared memory for the scatter
constexpr int kScatterMaxE = 384;       // per-warp expert cursors fit in shared memory up to here
constexpr int kRouteClusterMax = 8;     // CTAs of the single-cluster routing (portable size)

// sigma(z) = 1 / (1 + exp(-z)) in float32, one IEEE rounding per operation, with exp
// evaluated by Cody-Waite reduction (W. J. Cody and W. Waite, "Software Manual for the
// Elementary Functions", 1980): n = rint(x log2 e), r = (x - n*C1) - n*C2 where C1 =
// 355/512 is short enough that n*C1 is exact and C1 + C2 = ln 2, then exp(r) from the
// degree-7 Taylor polynomial in Horner form and an exact scaling by 2^n.  The input is
// clamped to [-86, 88] so 2^n stays a normal float.  Written out operation by operation
// (no contraction into fused multiply-adds) because the DeepSeekV3 key s + bias decides
// which experts win, and the host-side checker evaluates the same sequence.
MLDEV float sigmoid_key_f32(float z) {
  float x = -z;
  x = fminf(fmaxf(x, -86.0f), 88.0f);
  const float n = rintf(__fmul_rn(x, 0x1.715476p+0f));          // log2(e)
  float r = __fsub_rn(x, __fmul_rn(n, 0x1.63p-1f));             // 355/512
  r = __fsub_rn(r, __fmul_rn(n, -0x1.bd0106p-13f));             // ln 2 - 355/512
  float p = 1.0f / 5040.0f;
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 720.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 120.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 24.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 6.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 2.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  const float two_n = __int_as_float((static_cast<int>(n) + 127) << 23);
  const float e = __fmul_rn(p, two_n);
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
}

// Unsigned integer whose order is the float order of finite and infinite keys; 0 is left
// free as "no candidate".  -0 is folded to +0 first so that +-0 compare equal.
MLDEV uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);   // never 0 for a non-NaN key
}

MLDEV float from_order_key(uint32_t v) {
  return __uint_as_float((v & 0x80000000u) ? (v & 0x7fffffffu) : ~v);
}

MLDEV float load_logit(const __nv_bfloat16* row, int e) {
  float l = bf2f(row[e]);
  return (l != l) ? -INFINITY : l;   // NaN logits never win
}

// Grid-wide barrier for a cooperative launch; bounded spin.
MLDEV bool grid_barrier(uint32_t* ctr, uint32_t target, uint32_t* status, volatile int* ok_s) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1u);
    const uint64_t t0 = globaltimer_ns();
    int ok = 1;
    while (ld_acquire_gpu(ctr) < target) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        ok = 0;
        record_status(status, kDevTimeout, kWhereRouteBarrier);
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    *ok_s = ok;
  }
  __syncthreads();
  return *ok_s != 0;
}

// Exclusive scan of in[0..n) into out[0..n) (n <= 2 * kRouteThreads); returns the total.
MLDEV int block_exclusive_scan(const int* in, int* out, int n, int* warp_sums) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i0 = 2 * tid;
  const int a = (i0 < n) ? in[i0] : 0;
  const int b = (i0 + 1 < n) ? in[i0 + 1] : 0;
  const int s = a + b;
  int incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < kRouteWarps) ? warp_sums[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += y;
    }
    if (lane < kRouteWarps) warp_sums[lane] = wi - w;   // exclusive warp prefix
    if (lane == kRouteWarps - 1) warp_sums[kRouteWarps] = wi;
  }
  __syncthreads();
  const int excl = warp_sums[warp] + incl - s;
  if (i0 < n) out[i0] = excl;
  if (i0 + 1 < n) out[i0 + 1] = excl + a;
  const int total = warp_sums[kRouteWarps];
  __syncthreads();
  return total;
}

// Renormalize selection key: the 16-bit order key of the bf16 logit (NaN as -inf, -0 as +0)
// above 0xFFFF - e, so one unsigned maximum picks the largest logit and, among equal
// logits, the lowest expert id.  Never 0 ("no candidate").
MLDEV uint32_t packed_logit_key(const __nv_bfloat16* row, int e) {
  uint32_t u = static_cast<uint32_t>(__bfloat16_as_ushort(row[e]));
  if ((u & 0x7fffu) > 0x7f80u) u = 0xff80u;   // NaN -> -inf
  if (u == 0x8000u) u = 0u;                    // -0 -> +0
  const uint32_t o = (u & 0x8000u) ? (~u & 0xffffu) : (u | 0x8000u);
  return (o << 16) | (0xffffu - static_cast<uint32_t>(e));
}

MLDEV float packed_key_logit(uint32_t v) {
  const uint32_t o = v >> 16;
  const uint32_t u = (o & 0x8000u) ? (o & 0x7fffu) : (~o & 0xffffu);
  return __uint_as_float(u << 16);
}

// Top-k of the tokens [t0, t1): each warp runs kTPW tokens in lockstep, writes ids and
// weights, records the CTA-local pair ids in ids_s and counts pairs per expert in hist_s.
// Routing errors (an expert id out of range) are recorded in `err`: the status word, or a
// per-CTA shared word that the cluster kernel publishes once.
template <int EPL, int METHOD, int kTPW>
MLDEV void select_topk(const RouteParams& p, int t0, int t1, int* ids_s, int* hist_s, uint32_t* err) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int E = p.E, k = p.k;
  if constexpr (METHOD == 2) {
    // routing given from outside: each pair's global expert and bf16 weight come packed;
    // experts outside the local range (and invalid ids, which are also reported) go to
    // the last bucket
    for (int tb = t0 + warp * kTPW; tb < t1; tb += kRouteWarps * kTPW) {
#pragma unroll
      for (int u = 0; u < kTPW; ++u) {
        const int t = tb + u;
        if (t >= t1 || lane >= k) continue;
        const size_t pp = static_cast<size_t>(t) * k + lane;
        const uint32_t word = static_cast<uint32_t>(p.packed[pp]);
        const int gid = static_cast<int>(word >> 16);
        int e = gid - p.local_offset;
        if (gid >= p.ext_experts) {
          record_status(err, kDevBadSlot, kWhereRouteExpert);
          e = E - 1;
        } else if (e < 0 || e >= E - 1) {
          e = E - 1;
        }
        const int pl = (t - t0) * k + lane;   // pair index local to this CTA
        if (pl < kRouteIdsInSmem) ids_s[pl] = e;
        p.ids[pp] = e;
        p.weights[pp] = __uint_as_float((word & 0xffffu) << 16);
        atomicAdd(&hist_s[e], 1);
      }
    }
  } else if constexpr (METHOD == 0) {
    // Renormalize: packed (logit, id) keys are all distinct, so a round is one hardware
    // maximum over the lanes' list heads and the one lane holding it shifts its list.
    for (int tb = t0 + warp * kTPW; tb < t1; tb += kRouteWarps * kTPW) {
      uint32_t sk[kTPW][EPL];   // this lane's packed keys, descending; 0 = empty
      int my_id[kTPW];
      float my_key[kTPW];
#pragma unroll
      for (int u = 0; u < kTPW; ++u) {
        const int t = tb + u;
        my_id[u] = kInvalidId;
        my_key[u] = -INFINITY;
        const __nv_bfloat16* row = p.logits + static_cast<size_t>(t) * E;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const int e = lane + 32 * i;
          sk[u][i] = (t < t1 && e < E) ? packed_logit_key(row, e) : 0u;
        }
#pragma unroll
        for (int pass = 0; pass < EPL; ++pass) {   // odd-even transposition sort
#pragma unroll
          for (int i = pass & 1; i + 1 < EPL; i += 2) {
            const uint32_t a = sk[u][i], b = sk[u][i + 1];
            sk[u][i] = max(a, b);
            sk[u][i + 1] = min(a, b);
          }
        }
      }
      for (int j = 0; j < k; ++j) {
        uint32_t wmax[kTPW];
#pragma unroll
        for (int u = 0; u < kTPW; ++u) wmax[u] = __reduce_max_sync(0xffffffffu, sk[u][0]);
#pragma unroll
        for (int u = 0; u < kTPW; ++u) {
          if (wmax[u] != 0u && sk[u][0] == wmax[u]) {   // pop this lane's head
#pragma unroll
            for (int i = 0; i + 1 < EPL; ++i) sk[u][i] = sk[u][i + 1];
            sk[u][EPL - 1] = 0u;
          }
          if (lane == j && wmax[u] != 0u) {
            my_id[u] = static_cast<int>(0xffffu - (wmax[u] & 0xffffu));
            my_key[u] = packed_key_logit(wmax[u]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kTPW; ++u) {
        const int t = tb + u;
        if (t >= t1) break;   // uniform across the warp
        const float kmax = __shfl_sync(0xffffffffu, my_key[u], 0);
        const float ex = (lane < k) ? expf(my_key[u] - kmax) : 0.0f;
        float sum = ex;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        const float wv = ex / sum;
        if (lane < k) {
          const int pl = (t - t0) * k + lane;   // pair index local to this CTA
          if (pl < kRouteIdsInSmem) ids_s[pl] = my_id[u];
          p.ids[static_cast<size_t>(t) * k + lane] = my_id[u];
          p.weights[static_cast<size_t>(t) * k + lane] = wv;
          atomicAdd(&hist_s[my_id[u]], 1);
        }
      }
    }
  } else {
  // ---------------- phase 1: top-k per token; each warp runs kTPW tokens in lockstep.
  // Keys are mapped to unsigned integers whose order is the float order (-0 folded to +0,
  // so +-0 tie like equal floats).  Each lane first sorts its EPL (key, id) entries
  // (descending key, ascending id); a selection round is then: the warp maximum of the
  // lanes' heads (one hardware reduction), the lowest id holding it (a second one), and
  // the winning lane shifts its list.
  for (int tb = t0 + warp * kTPW; tb < t1; tb += kRouteWarps * kTPW) {
    uint32_t sk[kTPW][EPL];   // this lane's keys, sorted; 0 = empty
    int si[kTPW][EPL];        // their expert ids
    int my_id[kTPW];
    float my_key[kTPW];
#pragma unroll
    for (int u = 0; u < kTPW; ++u) {
      const int t = tb + u;
      my_id[u] = kInvalidId;
      my_key[u] = -INFINITY;
      const __nv_bfloat16* row = p.logits + static_cast<size_t>(t) * E;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        uint32_t ok = 0u;
        if (t < t1 && e < E) {
          const float l = load_logit(row, e);
          ok = order_key(METHOD == 1 ? __fadd_rn(sigmoid_key_f32(l), p.bias[e]) : l);
        }
        sk[u][i] = ok;
        si[u][i] = e;
      }
      // odd-even transposition sort, EPL passes: descending key; equal keys keep the
      // lower id first (ids start ascending and a swap needs a strictly larger key)
#pragma unroll
      for (int pass = 0; pass < EPL; ++pass) {
#pragma unroll
        for (int i = pass & 1; i + 1 < EPL; i += 2) {
          if (sk[u][i + 1] > sk[u][i]) {
            const uint32_t tk = sk[u][i];
            sk[u][i] = sk[u][i + 1];
            sk[u][i + 1] = tk;
            const int ti = si[u][i];
            si[u][i] = si[u][i + 1];
            si[u][i + 1] = ti;
          }
        }
      }
    }
    for (int j = 0; j < k; ++j) {
      uint32_t wmax[kTPW];
#pragma unroll
      for (int u = 0; u < kTPW; ++u) wmax[u] = __reduce_max_sync(0xffffffffu, sk[u][0]);
      uint32_t win[kTPW];
#pragma unroll
      for (int u = 0; u < kTPW; ++u)
        win[u] = __reduce_min_sync(0xffffffffu, (sk[u][0] == wmax[u] && sk[u][0] != 0u)
                                                    ? static_cast<uint32_t>(si[u][0]) : 0xffffffffu);
#pragma unroll
      for (int u = 0; u < kTPW; ++u) {
        const int w = static_cast<int>(win[u]);
        if (win[u] != 0xffffffffu && (w & 31) == lane) {   // pop this lane's head
#pragma unroll
          for (int i = 0; i + 1 < EPL; ++i) {
            sk[u][i] = sk[u][i + 1];
            si[u][i] = si[u][i + 1];
          }
          sk[u][EPL - 1] = 0u;
        }
        if (lane == j) {
          my_id[u] = w;
          my_key[u] = from_order_key(wmax[u]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kTPW; ++u) {
      const int t = tb + u;
      if (t >= t1) break;   // uniform across the warp
      const __nv_bfloat16* row = p.logits + static_cast<size_t>(t) * E;
      float wv;
      if (METHOD == 1) {
        const float s = (lane < k) ? sigmoid_key_f32(load_logit(row, my_id[u])) : 0.0f;
        float sum = s;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        wv = s / sum * p.rsf;
      } else {
        const float kmax = __shfl_sync(0xffffffffu, my_key[u], 0);
        const float ex = (lane < k) ? expf(my_key[u] - kmax) : 0.0f;
        float sum = ex;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        wv = ex / sum;
      }
      if (lane < k) {
        const int pl = (t - t0) * k + lane;   // pair index local to this CTA
        if (pl < kRouteIdsInSmem) ids_s[pl] = my_id[u];
        p.ids[static_cast<size_t>(t) * k + lane] = my_id[u];
        p.weights[static_cast<size_t>(t) * k + lane] = wv;
        atomicAdd(&hist_s[my_id[u]], 1);
      }
    }
  }
  }
}

// Scatter the pairs of tokens [t0, t1) to perm / inv_perm in ascending expanded index;
// cursor_s[e] holds the first permuted slot of this CTA's pairs of expert e.  wcnt is
// scratch of kRouteWarps * kScatterMaxE ints.
MLDEV void scatter_pairs(const RouteParams& p, int t0, int t1, const int* ids_s, int* cursor_s, int* wcnt) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E, k = p.k;
  // ---------------- scatter this CTA's pairs in ascending expanded index.  The pairs are
  // split into one contiguous chunk per warp; per-warp expert counts and their prefix over
  // warps (in warp order) give each warp its own cursors, and inside a warp 32 pairs at a
  // time get their rank among equal experts from ballots over the expert-id bits.
  const int p0 = t0 * k, p1 = max(t0, t1) * k;
  const int npairs = p1 - p0;
  const bool parallel = npairs <= kRouteIdsInSmem && E <= kScatterMaxE;
  const int chunk = parallel ? (npairs + kRouteWarps - 1) / kRouteWarps : npairs;
  if (parallel) {
    for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) wcnt[i] = 0;
    __syncthreads();
    for (int pl = tid; pl < npairs; pl += kRouteThreads) atomicAdd(&wcnt[(pl / chunk) * E + ids_s[pl]], 1);
    __syncthreads();
    for (int e = tid; e < E; e += kRouteThreads) {   // prefix over warps, in warp order
      int run = cursor_s[e];
      for (int w = 0; w < kRouteWarps; ++w) {
        const int c0 = wcnt[w * E + e];
        wcnt[w * E + e] = run;
        run += c0;
      }
    }
    __syncthreads();
  }
  if (parallel || warp == 0) {
    int* cur = parallel ? wcnt + warp * E : cursor_s;
    const int lo = parallel ? min(npairs, warp * chunk) : 0;
    const int hi = parallel ? min(npairs, lo + chunk) : npairs;
    int nbits = 0;
    while ((1 << nbits) < E) ++nbits;
    for (int pb = lo; pb < hi; pb += 32) {
      const int pl = pb + lane;
      const bool valid = pl < hi;
      const int e = valid ? (pl < kRouteIdsInSmem ? ids_s[pl] : p.ids[p0 + pl]) : -1;
      unsigned grp = __ballot_sync(0xffffffffu, valid);   // lanes with the same expert id
      for (int b = 0; b < nbits; ++b) {
        const unsigned ones = __ballot_sync(0xffffffffu, valid && ((e >> b) & 1));
        grp &= ((e >> b) & 1) ? ones : ~ones;
      }
      const int rank = __popc(grp & ((1u << lane) - 1u));
      const int q = valid ? cur[e] + rank : 0;
      __syncwarp();
      if (valid && rank == 0) cur[e] += __popc(grp);
      __syncwarp();
      if (valid) {
        p.perm[q] = p0 + pl;
        p.inv[p0 + pl] = (p.packed != nullptr && e == E - 1) ? -1 : q;   // dropped pair (method 2)
      }
    }
  }
}

template <int EPL, int METHOD>
__global__ void __launch_bounds__(kRouteThreads) route_align_kernel(const RouteParams p) {
  constexpr int kTPW = EPL <= 4 ? 4 : (EPL <= 8 ? 2 : 1);   // tokens per warp, in lockstep
  __shared__ int hist_s[kMaxExperts];
  __shared__ int cursor_s[kMaxExperts];
  __shared__ int warp_sums[kRouteWarps + 1];
  __shared__ int ok_s;
  __shared__ int ids_s[kRouteIdsInSmem];   // this CTA's expert ids, when they fit
  __shared__ int wcnt[kRouteWarps * kScatterMaxE];   // per-warp expert cursors

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, c = blockIdx.x;
  const int E = p.E;

  for (int e = tid; e < E; e += kRouteThreads) hist_s[e] = 0;
  __syncthreads();

  const int t0 = c * p.tokens_per_cta;
  const int t1 = min(p.T, t0 + p.tokens_per_cta);

  select_topk<EPL, METHOD, kTPW>(p, t0, t1, ids_s, hist_s, p.status);
  __syncthreads();

  pdl_trigger();   // the permute may launch now; it waits for this kernel to finish

  // ---------------- phase 2: expert offsets and per-CTA bases
  if (G > 1) {
    for (int e = tid; e < E; e += kRouteThreads) p.hist[c * E + e] = hist_s[e];
    if (!grid_barrier(p.barrier, static_cast<uint32_t>(G), p.status, &ok_s)) return;
    // warp per expert: prefix of the per-CTA counts in CTA order
    const int m = (G + 31) / 32;
    for (int e = c * kRouteWarps + warp; e < E; e += G * kRouteWarps) {
      int loc = 0;
      for (int i = 0; i < m; ++i) {
        const int cc = lane * m + i;
        if (cc < G) loc += __ldcg(&p.hist[cc * E + e]);
      }
      int incl = loc;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      int run = incl - loc;
      for (int i = 0; i < m; ++i) {
        const int cc = lane * m + i;
        if (cc < G) {
          p.base[cc * E + e] = run;
          run += __ldcg(&p.hist[cc * E + e]);
        }
      }
      if (lane == 31) p.total[e] = incl;
    }
    if (!grid_barrier(p.barrier, 2u * static_cast<uint32_t>(G), p.status, &ok_s)) return;
    for (int e = tid; e < E; e += kRouteThreads) hist_s[e] = __ldcg(&p.total[e]);
    __syncthreads();
  }
  const int total = block_exclusive_scan(hist_s, cursor_s, E, warp_sums);
  if (c == 0) {
    for (int e = tid; e < E; e += kRouteThreads) p.offsets[e] = cursor_s[e];
    if (tid == 0) p.offsets[E] = total;
  }
  if (G > 1) {
    for (int e = tid; e < E; e += kRouteThreads) cursor_s[e] += __ldcg(&p.base[c * E + e]);
  }
  __syncthreads();

  scatter_pairs(p, t0, t1, ids_s, cursor_s, wcnt);
}

// ---------------------------------------------------------------------------------
// Up to kRouteClusterMax CTAs of one thread-block cluster (up to 512 tokens): the same
// top-k and scatter, with the per-CTA expert counts exchanged through distributed shared
// memory between two cluster barriers instead of global scratch and grid barriers.  Every
// CTA reads all CTAs' counts (C x E loads), so each forms the expert offsets itself and
// its own per-expert base, the prefix of the counts of the CTAs before it.
// ---------------------------------------------------------------------------------

MLDEV int ld_dsmem(const int* local, uint32_t rank) {   // the same variable in CTA `rank`
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  int v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}


template <int EPL, int METHOD>
__global__ void __launch_bounds__(kRouteThreads) route_cluster_kernel(const RouteParams p) {
  __shared__ int hist_s[kMaxExperts];
  __shared__ int cursor_s[kMaxExperts];
  __shared__ int warp_sums[kRouteWarps + 1];
  __shared__ int ids_s[kRouteIdsInSmem];
  __shared__ int wcnt[kRouteWarps * kScatterMaxE];   // expert totals and bases, then scatter cursors
  __shared__ int err_s;                               // this CTA's first routing error (0: none)

  const int tid = threadIdx.x;
  const int C = gridDim.x;   // the grid is one cluster
  const uint32_t c = cluster_ctarank();
  const int E = p.E;

  for (int e = tid; e < E; e += kRouteThreads) hist_s[e] = 0;
  if (tid == 0) err_s = 0;
  // Launched behind the previous forward's last kernel: nothing global is read or written
  // before it has finished.
  pdl_wait();
  __syncthreads();
  const int t0 = static_cast<int>(c) * p.tokens_per_cta;
  const int t1 = min(p.T, t0 + p.tokens_per_cta);
  select_topk<EPL, METHOD, 1>(p, t0, t1, ids_s, hist_s, reinterpret_cast<uint32_t*>(&err_s));
  pdl_trigger();   // the permute may launch now; it waits for this kernel to finish

  cluster_arrive();   // this CTA's counts are final ...
  cluster_wait();     // ... and so are everyone's
  // This forward's status word starts here, written once: the first CTA's error, or 0.
  // Every later kernel touches it only after its own griddepcontrol.wait.
  if (c == 0 && tid == 0) {
    uint32_t w = 0;
    for (int cc = 0; cc < C; ++cc) {
      const uint32_t v = static_cast<uint32_t>(ld_dsmem(&err_s, static_cast<uint32_t>(cc)));
      if (w == 0) w = v;
    }
    *p.status = w;
  }
  int* tot_s = wcnt;          // [E] expert totals over the cluster
  int* base_s = wcnt + E;     // [E] pairs of the CTAs before this one
  for (int e = tid; e < E; e += kRouteThreads) {
    int base = 0, tot = 0;
    for (int cc = 0; cc < C; ++cc) {
      const int v = ld_dsmem(&hist_s[e], static_cast<uint32_t>(cc));
      base += (cc < static_cast<int>(c)) ? v : 0;
      tot += v;
    }
    tot_s[e] = tot;
    base_s[e] = base;
  }
  cluster_arrive();   // done reading the other CTAs' counts (waited for before exit)
  __syncthreads();
  const int total = block_exclusive_scan(tot_s, cursor_s, E, warp_sums);
  if (c == 0) {
    for (int e = tid; e < E; e += kRouteThreads) p.offsets[e] = cursor_s[e];
    if (tid == 0) p.offsets[E] = total;
  }
  for (int e = tid; e < E; e += kRouteThreads) cursor_s[e] += base_s[e];
  __syncthreads();
  scatter_pairs(p, t0, t1, ids_s, cursor_s, wcnt);
  cluster_wait();     // no CTA leaves while another may still read its counts
}

int route_cluster_ctas(int T) {
  if (T > kRouteClusterMax * 64) return 0;
  int c = (T + 15) / 16;
  if (c > kRouteClusterMax) c = kRouteClusterMax;
  return c < 1 ? 1 : c;
}

template <int EPL, int METHOD>
static cudaError_t launch_cluster_epl(const RouteParams& p, int ctas, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, route_cluster_kernel<EPL, METHOD>, p);
}

template <int METHOD>
static cudaError_t launch_cluster_method(const RouteParams& p, int ctas, cudaStream_t stream, bool pdl);

static int epl_for(int E) { return E <= 128 ? 4 : E <= 256 ? 8 : E <= 384 ? 12 : E <= 512 ? 16 : 32; }

template <int EPL, int METHOD>
static cudaError_t launch_epl(const RouteParams& p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = grid > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, route_align_kernel<EPL, METHOD>, p);
}

template <int METHOD>
static cudaError_t launch_method(const RouteParams& p, int grid, cudaStream_t stream) {
  if (METHOD == 2) return launch_epl<4, METHOD>(p, grid, stream);   // no candidate lists
  switch (epl_for(p.E)) {
    case 4: return launch_epl<4, METHOD>(p, grid, stream);
    case 8: return launch_epl<8, METHOD>(p, grid, stream);
    case 12: return launch_epl<12, METHOD>(p, grid, stream);
    case 16: return launch_epl<16, METHOD>(p, grid, stream);
    default: return launch_epl<32, METHOD>(p, grid, stream);
  }
}

int route_max_coop_ctas(int E) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  cudaError_t err;
  // every instantiation has the same block size and static shared memory; use the widest
  switch (epl_for(E)) {
    case 4: err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_align_kernel<4, 1>, kRouteThreads, 0); break;
    case 8: err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_align_kernel<8, 1>, kRouteThreads, 0); break;
    case 12: err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_align_kernel<12, 1>, kRouteThreads, 0); break;
    case 16: err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_align_kernel<16, 1>, kRouteThreads, 0); break;
    default: err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_align_kernel<32, 1>, kRouteThreads, 0); break;
  }
  if (err != cudaSuccess || per_sm < 1) return 1;
  const int n = sms * per_sm;
  return n < kMaxRouteCtas ? n : kMaxRouteCtas;
}

cudaError_t launch_route_align(const RouteParams& p, int grid, cudaStream_t stream) {
  if (p.method == 2) return launch_method<2>(p, grid, stream);
  return p.method == 1 ? launch_method<1>(p, grid, stream) : launch_method<0>(p, grid, stream);
}

template <int METHOD>
static cudaError_t launch_cluster_method(const RouteParams& p, int ctas, cudaStream_t stream, bool pdl) {
  if (METHOD == 2) return launch_cluster_epl<4, METHOD>(p, ctas, stream, pdl);
  switch (epl_for(p.E)) {
    case 4: return launch_cluster_epl<4, METHOD>(p, ctas, stream, pdl);
    case 8: return launch_cluster_epl<8, METHOD>(p, ctas, stream, pdl);
    case 12: return launch_cluster_epl<12, METHOD>(p, ctas, stream, pdl);
    case 16: return launch_cluster_epl<16, METHOD>(p, ctas, stream, pdl);
    default: return launch_cluster_epl<32, METHOD>(p, ctas, stream, pdl);
  }
}

cudaError_t launch_route_cluster(const RouteParams& p, int ctas, cudaStream_t stream, bool pdl) {
  if (ctas < 1 || ctas > kRouteClusterMax) return cudaErrorInvalidValue;
  if (p.method == 2) return launch_cluster_method<2>(p, ctas, stream, pdl);
  return p.method == 1 ? launch_cluster_method<1>(p, ctas, stream, pdl)
                       : launch_cluster_method<0>(p, ctas, stream, pdl);
}

}  // namespace mlk
