// attention_tc.cu - causal grouped-query attention on tcgen05 (sm_103a), hd = 64.
//
// o[b,t,h,:] = sum_{j visible} softmax_j(q[b,h,t].k[b,h/g,j] / sqrt(hd)) v[b,h/g,j]
// with j visible iff valid_start[b] <= j <= t ("model.py" (SmolLM2-135M)
// section 4: scaled scores, triu(1) causal mask plus the padding mask, softmax,
// probs @ v; query head h reads key/value head h // g as in the "SmolLM3"
// page's "Grouped-query attention").  Rows with no visible key produce 0.
//
// One CTA owns (sequence b, kv head, a tile of 128 query tokens) and GH <= 3
// query heads of that kv head.  Each K tile [64 keys x 64] and V^T tile
// [64 x 64 keys] is loaded once by TMA into shared memory and serves all GH
// heads: K/V are never expanded per query head.  Per (kv tile, head) "slot":
//   S = Q_h K^T        tcgen05.mma, M=128 N=64 K=64, fp32 in TMEM
//   P = exp2(S*c - m)  four softmax warps, one query row per thread (no
//                      cross-thread reductions); P is written as packed f16
//                      over S's own TMEM columns
//   O_h += P V         tcgen05.mma with A (= P) read from TMEM, M=128 N=64 K=64
// The CTA is serial (S, softmax, P V, next S) and small - 256 TMEM columns
// (O for GH heads + one S tile) and ~100 KB of shared memory - so two CTAs
// share an SM and the tensor core works for one while the other's softmax
// runs (and one's prologue/epilogue overlaps the other's main loop).
// The running max is updated lazily: O_h is rescaled in TMEM only when a row's
// max grows by more than 2^8 (otherwise P may exceed 1 by up to 256, exact in
// the fp32 sums and within f16 range), the FlashAttention-4 idea.
// Warp 0 issues TMA, warp 1 allocates TMEM and one lane issues every MMA,
// warps 2..5 do the softmax and the final normalisation.  All waits are
// bounded (status word + abort flag, copies and MMAs drained before exit).
#include <math.h>

#include "common.cuh"
#include "prims.cuh"

namespace smol {

namespace {

constexpr int kBQ = 128;      // query rows per tile (UMMA M)
constexpr int kBK = 64;       // keys per KV tile
constexpr int kHD = 64;
constexpr int kNS = 3;        // K / V^T pipeline stages
constexpr int kThreads = 192;   // producer, MMA, one softmax warpgroup

template <int GH>
struct AtCfg {
  static constexpr int Q_BYTES = kBQ * kHD * 2;         // one head: [128][64] f16
  static constexpr int K_BYTES = kBK * kHD * 2;         // [64 keys][64]
  static constexpr int VT_BYTES = kHD * kBK * 2;        // [64 dims][64 keys]
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + GH * Q_BYTES;
  static constexpr int OFF_VT = OFF_K + kNS * K_BYTES;
  static constexpr int OFF_BAR = OFF_VT + kNS * VT_BYTES;
  static constexpr int SMEM_RAW = 1024 + OFF_BAR + 256;
  // at least 80 KB so that no third CTA (whose TMEM allocation would wait) joins two on an SM
  static constexpr int SMEM = SMEM_RAW < 81920 ? 81920 : SMEM_RAW;
  static constexpr int TMEM_S = GH * kHD;               // S (and P over its first 32 columns)
  static constexpr int TMEM_COLS = 256;
  static_assert(GH >= 1 && GH <= 3, "O accumulators and one S tile in 256 columns");
  static_assert(SMEM <= 116736, "two CTAs per SM");
};

struct AtParams {
  f16 *o;                   // [B, T, H*hd]
  const int *valid_start;
  int B, T, H, KV, G, GH, n_hsub;
  float scale_log2;
  int *status;
};

enum : int {
  kAtTimeoutLoad = 0x201,
  kAtTimeoutMma = 0x202,
  kAtTimeoutSoftmax = 0x203,
  kAtTimeoutDrain = 0x204,
};

// 2^x with the hardware approximation (flushes subnormal results to zero;
// 2^(-inf) = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void at_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

template <int GH>
__global__ void __launch_bounds__(kThreads, 2)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmVt, const AtParams p) {
  using C = AtCfg<GH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + C::OFF_Q;
  uint8_t *sK = smem + C::OFF_K;
  uint8_t *sVt = smem + C::OFF_VT;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *q_full = bars;
  uint64_t *kv_full = bars + 1;              // [kNS]
  uint64_t *kv_empty = bars + 1 + kNS;       // [kNS]
  uint64_t *s_full = bars + 1 + 2 * kNS;     // S(s) computed
  uint64_t *p_full = s_full + 1;             // P(s) written (128 arrivals)
  uint64_t *s_free = s_full + 2;             // P(s) V done: S/P columns free, O_h current
  uint64_t *o_done = s_full + 3;             // every MMA of the CTA complete
  uint64_t *drain = s_full + 4;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.T;
  // blocks are launched in linear order (x fastest): the query tile is the
  // slow index, descending, so every sequence's longest causal tiles start
  // first and the short ones fill the tail (longest-processing-time order)
  const int q0 = (gridDim.y - 1 - blockIdx.y) * kBQ;
  const int groups = p.KV * p.n_hsub;
  const int b = blockIdx.x / groups;
  const int kvh = (blockIdx.x - b * groups) / p.n_hsub;
  const int hsub = blockIdx.x - b * groups - kvh * p.n_hsub;
  const int h_first = kvh * p.G + hsub * GH;
  const int vs = p.valid_start ? min(max(p.valid_start[b], 0), T) : 0;
  const int last_q = min(q0 + kBQ - 1, T - 1);
  const int j_hi = last_q / kBK;
  const int j_lo = min(vs / kBK, j_hi);          // an all-padding tile still runs one (masked) tile
  const int ntiles = j_hi - j_lo + 1;
  const int nslots = ntiles * GH;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(s_free, 1);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVt);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------- TMA producer
      int dummy = 0;
      long long issued = 0;                       // kv stages issued (for the drain)
      bool ok = true;
      mbar_arrive_expect_tx(q_full, GH * C::Q_BYTES);
      for (int h = 0; h < GH; ++h)
        tma_load_2d(sQ + h * C::Q_BYTES, &tmQ, q_full, 0, ((b * p.H) + h_first + h) * T + q0);
      for (int it = 0; it < ntiles && ok; ++it) {
        const int j = j_lo + it, st = it % kNS;
        if (!mbar_wait_bounded(&kv_empty[st], ((it / kNS) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&kv_full[st], C::K_BYTES + C::VT_BYTES);
        tma_load_2d(sK + st * C::K_BYTES, &tmK, &kv_full[st], 0, (b * p.KV + kvh) * T + j * kBK);
        tma_load_2d(sVt + st * C::VT_BYTES, &tmVt, &kv_full[st], j * kBK, (b * p.KV + kvh) * kHD);
        ++issued;
      }
      // wait (bounded) until every copy this thread issued has landed
      if (!mbar_wait_bounded(q_full, 0, reinterpret_cast<volatile int *>(&dummy)))
        at_status(p.status, kAtTimeoutDrain);
      if (!ok) {
        at_status(p.status, kAtTimeoutLoad);
        *abort_flag = 1;
        const long long first = issued > kNS ? issued - kNS : 0;
        for (long long i = first; i < issued; ++i)
          if (!mbar_wait_bounded(&kv_full[i % kNS], (uint32_t)((i / kNS) & 1),
                                 reinterpret_cast<volatile int *>(&dummy)))
            at_status(p.status, kAtTimeoutDrain);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------- MMA issuer
      constexpr uint32_t kIdesc = idesc_f16_f32(kBQ, 64);   // both MMAs: M=128, N=64
      bool ok = mbar_wait_bounded(q_full, 0, abort_flag), any = false;
      for (int s = 0; s < nslots && ok; ++s) {
        const int it = s / GH, h = s - it * GH, st = it % kNS;
        // S(s) = Q_h K_j^T over S's columns, once P(s-1) V has read them
        if (s > 0 && !mbar_wait_bounded(s_free, (s - 1) & 1, abort_flag)) { ok = false; break; }
        if (h == 0 && !mbar_wait_bounded(&kv_full[st], (it / kNS) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after_sync();
        const uint64_t a = sdesc_kmajor_sw128(smem_u32(sQ + h * C::Q_BYTES));
        const uint64_t bk = sdesc_kmajor_sw128(smem_u32(sK + st * C::K_BYTES));
#pragma unroll
        for (int k = 0; k < kHD / 16; ++k)
          umma_f16(tmem + C::TMEM_S, a + 2 * k, bk + 2 * k, kIdesc, k > 0);
        any = true;
        umma_commit(s_full);
        // O_h += P(s) V_j once the softmax has written P(s)
        if (!mbar_wait_bounded(p_full, s & 1, abort_flag)) { ok = false; break; }
        tc_fence_after_sync();
        const uint64_t bv = sdesc_kmajor_sw128(smem_u32(sVt + st * C::VT_BYTES));
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)   // 16 keys of P = 8 TMEM columns per MMA
          umma_f16_tmem_a(tmem + h * kHD, tmem + C::TMEM_S + k * 8, bv + 2 * k, kIdesc, (it | k) != 0);
        umma_commit(s_free);
        if (h == GH - 1) umma_commit(&kv_empty[st]);
      }
      if (ok) {
        umma_commit(o_done);
      } else {
        at_status(p.status, kAtTimeoutMma);
        *abort_flag = 1;
        if (any) {
          umma_commit(drain);
          int dummy = 0;
          if (!mbar_wait_bounded(drain, 0, reinterpret_cast<volatile int *>(&dummy)))
            at_status(p.status, kAtTimeoutDrain);
        }
      }
    }
  } else {
    // ---------------------------------------------- softmax: warps 2..5, one
    // query row per thread, all 64 keys of every tile
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;              // query row within the tile
    const int t = q0 + r;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    float m[GH], l[GH];                             // running max (exp2 domain) and sum
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
    bool alive = true;
    for (int s = 0; s < nslots; ++s) {
      const int it = s / GH, h = s - it * GH;
      const int k0 = (j_lo + it) * kBK;             // first key of this tile
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(s_full, s & 1, abort_flag))) {
        alive = false;
        break;
      }
      tc_fence_after_sync();
      const bool need_mask = (k0 + kBK - 1 > q0) || (k0 < vs);
      uint32_t sv[64];
      tmem_ld32(lane_base + C::TMEM_S, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld32(lane_base + C::TMEM_S + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_ld_wait();
      // eight independent max chains (a single chain is latency-bound)
      float mc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) mc[q] = -INFINITY;
      const int hi = t - k0, lo = vs - k0;          // keys k0+e visible iff lo <= e <= hi
      if (need_mask) {
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (e <= hi && e >= lo) mc[e & 7] = fmaxf(mc[e & 7], __uint_as_float(sv[e]));
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) mc[e & 7] = fmaxf(mc[e & 7], __uint_as_float(sv[e]));
      }
      float mxa = fmaxf(fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3])), fmaxf(fmaxf(mc[4], mc[5]), fmaxf(mc[6], mc[7])));
      mxa = (mxa == -INFINITY) ? -INFINITY : mxa * sl2;   // into the exp2 domain
      float mh = m[h];
      float alpha = 1.f;
      const bool resc = (mh != -INFINITY) && (mxa > mh + 8.f);
      if (resc) {
        alpha = ex2_approx(mh - mxa);
        l[h] *= alpha;
        mh = mxa;
      } else if (mh == -INFINITY) {
        mh = mxa;                                   // first visible key(s) of this row
      }
      m[h] = mh;
      if (__any_sync(0xffffffffu, resc)) {
        // O_h holds every earlier P V (the MMA issued S(s) only after the
        // previous P V completed); rescale in TMEM.  tcgen05.ld/st are
        // warp-collective: every lane takes part, alpha = 1 where the row's
        // max did not move
        uint32_t ov[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          tmem_ld32(lane_base + h * kHD + half * 32, ov);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(lane_base + h * kHD + half * 32, ov);
        }
      }
      const float mu = (mh == -INFINITY) ? 0.f : mh;
      // p = 2^(s*c - m) as f16, packed two keys per TMEM column over S's first 32 columns
      uint32_t pk[32];
      float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // eight partial sums
      if (need_mask) {
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          const float x0 = (e <= hi && e >= lo) ? fmaf(__uint_as_float(sv[e]), sl2, -mu) : -INFINITY;
          const float x1 = (e + 1 <= hi && e + 1 >= lo) ? fmaf(__uint_as_float(sv[e + 1]), sl2, -mu) : -INFINITY;
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          ps[e & 7] += p0;
          ps[(e + 1) & 7] += p1;
          pk[e >> 1] = pack_f16x2(p0, p1);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(sv[e]), sl2, -mu));
          const float p1 = ex2_approx(fmaf(__uint_as_float(sv[e + 1]), sl2, -mu));
          ps[e & 7] += p0;
          ps[(e + 1) & 7] += p1;
          pk[e >> 1] = pack_f16x2(p0, p1);
        }
      }
      tmem_st32(lane_base + C::TMEM_S, pk);
      tmem_st_wait();                               // P (and any O rescale) visible to the MMA
      l[h] += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      tc_fence_before_sync();
      mbar_arrive(p_full);
    }
    // ------------------------------------------------ normalise and store
    if (alive && !__all_sync(0xffffffffu, mbar_wait_bounded(o_done, 0, abort_flag))) alive = false;
    if (!alive) {
      if (lane == 0) at_status(p.status, kAtTimeoutSoftmax);
      *abort_flag = 1;
    } else {
      tc_fence_after_sync();
      const bool row_ok = t < T;
      const long long ldo = (long long)p.H * kHD;
#pragma unroll 1
      for (int h = 0; h < GH; ++h) {
        const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t ov[32];
          tmem_ld32(lane_base + h * kHD + half * 32, ov);
          tmem_ld_wait();
          if (row_ok) {
            f16 *dst = p.o + ((long long)b * T + t) * ldo + (long long)(h_first + h) * kHD + half * 32;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float *f = reinterpret_cast<const float *>(&ov[8 * q]);
              const uint4 w = make_uint4(pack_f16x2(f[0] * inv, f[1] * inv), pack_f16x2(f[2] * inv, f[3] * inv),
                                         pack_f16x2(f[4] * inv, f[5] * inv), pack_f16x2(f[6] * inv, f[7] * inv));
              *reinterpret_cast<uint4 *>(dst + 8 * q) = w;
            }
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int GH>
cudaError_t launch_gh(const AttnParams &a, const CUtensorMap &tq, const CUtensorMap &tk,
                      const CUtensorMap &tv, cudaStream_t st) {
  using C = AtCfg<GH>;
  auto kern = attn_tc_kernel<GH>;
  cudaError_t e = ensure_smem_attr<attn_tc_kernel<GH>>(C::SMEM);
  if (e != cudaSuccess) return e;
  AtParams p{};
  p.o = a.o;
  p.valid_start = a.valid_start;
  p.B = a.B; p.T = a.T; p.H = a.H; p.KV = a.KV;
  p.G = a.H / a.KV;
  p.GH = GH;
  p.n_hsub = p.G / GH;
  p.scale_log2 = a.scale_log2;
  p.status = a.status;
  dim3 grid((unsigned)(a.B * a.KV * p.n_hsub), (unsigned)cdiv(a.T, kBQ), 1u);
  kern<<<grid, kThreads, C::SMEM, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

bool attention_tc_supported(int hd, int H, int KV) {
  const int G = H / KV;
  return hd == kHD && (G == 1 || G == 2 || G == 3 || G == 4 || G == 6 || G == 8);
}

cudaError_t launch_attention_tc(const AttnParams &a, cudaStream_t st) {
  if (!attention_tc_supported(a.hd, a.H, a.KV) || a.v_t == nullptr) return cudaErrorInvalidConfiguration;
  CUtensorMap tq, tk, tv;
  if (!get_tmap_f16(&tq, a.q, (uint64_t)a.B * a.H * a.T, kHD, kHD, kBQ)) return cudaErrorInvalidValue;
  if (!get_tmap_f16(&tk, a.k, (uint64_t)a.B * a.KV * a.T, kHD, kHD, kBK)) return cudaErrorInvalidValue;   // [64 keys] boxes
  // V^T: rows are (b, kv head, dim), columns are keys; columns >= T read as zero
  if (!get_tmap_f16(&tv, a.v_t, (uint64_t)a.B * a.KV * kHD, a.T, a.T_pad, kHD)) return cudaErrorInvalidValue;
  const int G = a.H / a.KV;
  switch (G) {
    case 1: return launch_gh<1>(a, tq, tk, tv, st);
    case 2: return launch_gh<2>(a, tq, tk, tv, st);
    case 3: return launch_gh<3>(a, tq, tk, tv, st);
    case 4: return launch_gh<2>(a, tq, tk, tv, st);   // two CTAs per group of four
    case 6: return launch_gh<3>(a, tq, tk, tv, st);   // two CTAs per group of six
    case 8: return launch_gh<2>(a, tq, tk, tv, st);   // four CTAs per group of eight
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace smol
