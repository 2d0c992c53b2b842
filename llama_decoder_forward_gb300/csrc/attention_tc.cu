// attention_tc.cu - causal grouped-query attention on tcgen05 (sm_103a), hd = 64.
//
// o[b,t,h,:] = sum_{j visible} softmax_j(q[b,h,t].k[b,h/g,j] / sqrt(hd)) v[b,h/g,j]
// with j visible iff valid_start[b] <= j <= t ("model.py" (SmolLM2-135M)
// section 4: scaled scores, triu(1) causal mask plus the padding mask, softmax,
// probs @ v; query head h reads key/value head h // g as in the "SmolLM3"
// page's "Grouped-query attention").  Rows with no visible key produce 0.
// A block with a sliding window w (the "SmolLM3" page, "A sliding window the
// 3B checkpoints leave off") also hides keys j <= t - w: the CTA starts at the
// tile of its first query's window and masks per row.  An optional key mask
// (the additive 0 / -inf attention_mask of "model.py" section 4, as bytes)
// hides further keys; every tile then takes the masked path.
//
// One CTA owns (sequence b, kv head, a tile of 128 query tokens) and the GH
// query heads of that kv head.  Each K tile [128 keys x 64] and V^T tile
// [64 x 128 keys] is loaded once by TMA into shared memory and serves all GH
// heads: K/V are never expanded per query head.  Per (kv tile, head):
//   S = Q_h K^T        tcgen05.mma, M=128 N=128 K=64, fp32 in TMEM (two S buffers,
//                      so the MMA for the next head runs while this one's softmax does)
//   P = exp2(S*c - m)  eight softmax warps, one query row per thread per half tile; P is
//                      written as packed f16 into the S buffer's own TMEM columns
//   O_h += P V         tcgen05.mma with A (= P) read from TMEM, M=128 N=64 K=128, fp32
//                      accumulator in TMEM; shared memory only feeds Q, K and V^T
// The running max is updated lazily: O_h is rescaled in TMEM only when a row's
// max grows by more than 2^8 (otherwise P may exceed 1 by up to 256, exact in
// the fp32 sums and within f16 range), the FlashAttention-4 idea.
// Warp 0 issues TMA, warp 1 allocates TMEM and one lane issues every MMA,
// warps 2..9 (two groups of four, each taking half of every tile's keys) do
// the softmax and the final normalisation.  All waits are
// bounded (status word + abort flag, copies and MMAs drained before exit).
#include <math.h>

#include "common.cuh"
#include "prims.cuh"

namespace smol {

namespace {

constexpr int kBQ = 128;      // query rows per tile (UMMA M)
constexpr int kBK = 128;      // keys per KV tile
constexpr int kHD = 64;
constexpr int kThreads = 320;   // producer, MMA, two softmax warpgroups

template <int GH>
struct AtCfg {
  static constexpr int Q_BYTES = kBQ * kHD * 2;         // one head: [128][64] f16
  static constexpr int K_BYTES = kBK * kHD * 2;         // [128 keys][64]
  static constexpr int VT_SUB = kHD * 64 * 2;           // [64 dims][64 keys]
  static constexpr int VT_BYTES = 2 * VT_SUB;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + GH * Q_BYTES;
  static constexpr int OFF_VT = OFF_K + 2 * K_BYTES;
  static constexpr int OFF_RED = OFF_VT + 2 * VT_BYTES;  // [2][2][128] row maxes, [2][4][128] row sums
  static constexpr int OFF_STG = OFF_RED + (2 * 2 * 128 + 2 * 4 * 128) * 4;   // output staging:
  static constexpr int STG_WARP = 32 * 32 * 2;          // [head][softmax warp][32 rows][32 f16]
  static constexpr int OFF_BAR = OFF_STG + GH * 8 * STG_WARP;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
  static constexpr int TMEM_S = 256;                    // S buffers at columns 256 + sb*128;
                                                        // P (f16) overwrites columns 0..63 of its S
  static_assert(GH >= 1 && GH * kHD <= 256, "O accumulators must fit below the S buffers");
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

struct AtParams {
  f16 *o;                   // [B, T, H*hd]
  const int *valid_start;
  int B, T, H, KV, G, GH, n_hsub;
  float scale_log2;
  int window;               // > 0: query t sees keys j > t - window only
  const uint8_t *key_mask;  // [B, T] or nullptr: key j of sequence b hidden where 0
  int Tk, q_off;            // keys per sequence; key index of query 0
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

// AND of `pred` over the 256 softmax threads (named barrier 1); also a
// barrier between the two softmax warpgroups.
__device__ __forceinline__ bool softmax_and(bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)pred)
      : "memory");
  return out != 0;
}

// max(a, b, c) in one instruction (three-input max of sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void at_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// KM: the launch carries a key mask (a separate instantiation, so the
// unmasked kernel is exactly the code without it).
template <int GH, bool KM>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmVt, const __grid_constant__ CUtensorMap tmO,
                   const AtParams p) {
  using C = AtCfg<GH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + C::OFF_Q;
  uint8_t *sK = smem + C::OFF_K;
  uint8_t *sVt = smem + C::OFF_VT;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *q_full = bars;
  uint64_t *kv_full = bars + 1;     // [2]
  uint64_t *kv_empty = bars + 3;    // [2]
  uint64_t *s_full = bars + 5;      // [2] S(s) computed
  uint64_t *s_free = bars + 7;      // [2] PV(s) done: the S/P columns may be overwritten
  uint64_t *p_full = bars + 9;      // [2] P(s) written into TMEM
  uint64_t *o_ready = bars + 13;    // [GH]
  uint64_t *drain = bars + 13 + GH;
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
  const int Tk = p.Tk, qo = p.q_off;              // query t is key qo + t
  const int vs = p.valid_start ? min(max(p.valid_start[b], 0), Tk) : 0;
  const int last_q = min(q0 + kBQ - 1, T - 1);
  const int j_hi = (qo + last_q) / kBK;
  // lowest key any query of the tile sees (padding start; window start of the first query)
  const int key_lo = p.window > 0 ? max(vs, qo + q0 - p.window + 1) : vs;
  const int j_lo = min(key_lo / kBK, j_hi);      // an all-padding tile still runs one (masked) tile
  const int ntiles = j_hi - j_lo + 1;
  const int nslots = ntiles * GH;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 1);
      mbar_init(&p_full[i], 256);
    }
    for (int h = 0; h < GH; ++h) mbar_init(&o_ready[h], 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVt);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) griddep_launch_dependents();
  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------- TMA producer
      griddep_wait();                             // q, k and V^T come from the preceding kernel
      int dummy = 0;
      long long issued = 0;                       // kv stages issued (for the drain)
      bool ok = true;
      mbar_arrive_expect_tx(q_full, GH * C::Q_BYTES);
      for (int h = 0; h < GH; ++h)
        tma_load_2d(sQ + h * C::Q_BYTES, &tmQ, q_full, 0, ((b * p.H) + h_first + h) * T + q0);
      for (int it = 0; it < ntiles && ok; ++it) {
        const int j = j_lo + it, st = it & 1;
        if (!mbar_wait_bounded(&kv_empty[st], ((it >> 1) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&kv_full[st], C::K_BYTES + C::VT_BYTES);
        tma_load_2d(sK + st * C::K_BYTES, &tmK, &kv_full[st], 0, (b * p.KV + kvh) * Tk + j * kBK);
        tma_load_2d(sVt + st * C::VT_BYTES, &tmVt, &kv_full[st], j * kBK, (b * p.KV + kvh) * kHD);
        tma_load_2d(sVt + st * C::VT_BYTES + C::VT_SUB, &tmVt, &kv_full[st], j * kBK + 64,
                    (b * p.KV + kvh) * kHD);
        ++issued;
      }
      // wait (bounded) until every copy this thread issued has landed
      if (!mbar_wait_bounded(q_full, 0, reinterpret_cast<volatile int *>(&dummy)))
        at_status(p.status, kAtTimeoutDrain);
      if (!ok) {
        at_status(p.status, kAtTimeoutLoad);
        *abort_flag = 1;
        const long long first = issued > 2 ? issued - 2 : 0;
        for (long long i = first; i < issued; ++i)
          if (!mbar_wait_bounded(&kv_full[i & 1], (uint32_t)((i >> 1) & 1),
                                 reinterpret_cast<volatile int *>(&dummy)))
            at_status(p.status, kAtTimeoutDrain);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------- MMA issuer
      constexpr uint32_t kIdescS = idesc_f16_f32(kBQ, kBK);
      constexpr uint32_t kIdescO = idesc_f16_f32(kBQ, kHD);
      bool ok = mbar_wait_bounded(q_full, 0, abort_flag), any = false;
      for (int s = 0; s <= nslots && ok; ++s) {
        if (s < nslots) {
          // S(s) = Q_h K_j^T into S buffer s & 1
          const int it = s / GH, h = s - it * GH, sb = s & 1;
          if (!mbar_wait_bounded(&s_free[sb], ((s >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
          if (h == 0 && !mbar_wait_bounded(&kv_full[it & 1], (it >> 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after_sync();
          const uint64_t a = sdesc_kmajor_sw128(smem_u32(sQ + h * C::Q_BYTES));
          const uint64_t bk = sdesc_kmajor_sw128(smem_u32(sK + (it & 1) * C::K_BYTES));
#pragma unroll
          for (int k = 0; k < kHD / 16; ++k)
            umma_f16(tmem + C::TMEM_S + sb * kBK, a + 2 * k, bk + 2 * k, kIdescS, k > 0);
          any = true;
          umma_commit(&s_full[sb]);
        }
        if (s >= 1) {
          // O_h += P(s-1) V_j
          const int ps = s - 1, it = ps / GH, h = ps - it * GH, pb = ps & 1;
          if (!mbar_wait_bounded(&p_full[pb], (ps >> 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after_sync();
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
            const uint64_t bv = sdesc_kmajor_sw128(smem_u32(sVt + (it & 1) * C::VT_BYTES + kb * C::VT_SUB));
#pragma unroll
            for (int k = 0; k < 4; ++k)   // 16 keys of P = 8 TMEM columns per MMA
              umma_f16_tmem_a(tmem + h * kHD, tmem + C::TMEM_S + pb * kBK + (kb * 4 + k) * 8, bv + 2 * k,
                              kIdescO, (it | kb | k) != 0);
          }
          umma_commit(&s_free[pb]);
          umma_commit(&o_ready[h]);
          if (h == GH - 1) umma_commit(&kv_empty[it & 1]);
        }
      }
      if (!ok) {
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
    griddep_wait();                               // o is written below
    // ---------------------------------------------- softmax: warps 2..5 take keys
    // 0..63 of every tile (group 0), warps 6..9 keys 64..127 (group 1); one
    // query row per thread.  The groups exchange partial row maxes in shared
    // memory at a named-barrier reduction that also ANDs their health, so a
    // bounded wait that gives up in one group stops both together.
    const int quarter = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;              // query row within the tile
    const int t = q0 + r;
    const int tk = qo + t;                          // this row's own key index
    const int row_lo = p.window > 0 ? max(vs, tk - p.window + 1) : vs;   // this row's first visible key
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    float *red_max = reinterpret_cast<float *>(smem + C::OFF_RED);          // [2][2][128]
    float *red_sum = red_max + 2 * 2 * 128;                                   // [2][4][128]
    float m[GH], l[GH];                             // running max (shared value), partial sums
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
    bool alive = true;
    // visibility of this group's 64 keys under the caller's key mask (bit e =
    // key k0 + e), read once per key tile and shared by its GH head slots
    unsigned long long vis = ~0ull;
    int vis_it = -1;
    const uint8_t *kmask = KM ? p.key_mask + (long long)b * T : nullptr;
    for (int s = 0; s < nslots; ++s) {
      const int it = s / GH, h = s - it * GH, sb = s & 1;
      const int k0 = (j_lo + it) * kBK + grp * 64;  // first key of this group's half tile
      if (KM && it != vis_it) {
        vis = 0ull;
#pragma unroll 8
        for (int e = 0; e < 64; ++e)
          if (k0 + e < T && __ldg(kmask + k0 + e)) vis |= 1ull << e;
        vis_it = it;
      }
      const bool ok = alive && __all_sync(0xffffffffu, mbar_wait_bounded(&s_full[sb], (s >> 1) & 1, abort_flag));
      const bool need_mask = KM || (k0 + 63 > qo + q0) || (k0 < vs) || (p.window > 0 && k0 <= qo + last_q - p.window);
      uint32_t sv[64];
      float mx = -INFINITY;
      if (ok) {
        tc_fence_after_sync();
        const uint32_t s_col = lane_base + C::TMEM_S + sb * kBK + grp * 64;
        tmem_ld32(s_col, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_ld_wait();
        // eight independent max chains (a single chain is latency-bound)
        float mc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mc[q] = -INFINITY;
        if (need_mask) {
          const int hi = tk - k0, lo = row_lo - k0;
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e <= hi && e >= lo && (!KM || ((vis >> e) & 1ull))) mc[e & 7] = fmaxf(mc[e & 7], __uint_as_float(sv[e]));
        } else {
#pragma unroll
          for (int e = 0; e < 64; e += 2)
            mc[(e >> 1) & 7] = fmax3(mc[(e >> 1) & 7], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
        }
        mx = fmaxf(fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3])), fmaxf(fmaxf(mc[4], mc[5]), fmaxf(mc[6], mc[7])));
      }
      red_max[((s & 1) * 2 + grp) * 128 + r] = mx;
      tc_fence_before_sync();                       // both groups' S reads precede any P write
      alive = softmax_and(ok);
      tc_fence_after_sync();
      if (!alive) break;
      float mxa = fmaxf(mx, red_max[((s & 1) * 2 + (grp ^ 1)) * 128 + r]);
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
        // O_h must hold every earlier P V before it is rescaled; each group
        // rescales its 32 of the head's 64 columns
        if (__all_sync(0xffffffffu, mbar_wait_bounded(&o_ready[h], (it - 1) & 1, abort_flag))) {
          tc_fence_after_sync();
          uint32_t ov[32];
          tmem_ld32(lane_base + h * kHD + grp * 32, ov);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(lane_base + h * kHD + grp * 32, ov);
          tmem_st_wait();
        } else {
          alive = false;
        }
      }
      if (!alive) continue;                         // the next reduction stops both groups
      const float mu = (mh == -INFINITY) ? 0.f : mh;
      // p = 2^(s*c - m) as f16, packed two keys per TMEM column into the first
      // 64 columns of this S buffer (this group's 64 keys -> 32 columns)
      uint32_t pk[32];
      float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // eight partial sums
      if (need_mask) {
        // keys k0+e visible iff lo <= e <= hi (causal, padding and window limits)
        const int hi = tk - k0, lo = row_lo - k0;
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          const float x0 = (e <= hi && e >= lo && (!KM || ((vis >> e) & 1ull)))
                               ? fmaf(__uint_as_float(sv[e]), sl2, -mu)
                               : -INFINITY;
          const float x1 = (e + 1 <= hi && e + 1 >= lo && (!KM || ((vis >> (e + 1)) & 1ull)))
                               ? fmaf(__uint_as_float(sv[e + 1]), sl2, -mu)
                               : -INFINITY;
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
      tmem_st32(lane_base + C::TMEM_S + sb * kBK + grp * 32, pk);
      tmem_st_wait();
      l[h] += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      tc_fence_before_sync();
      mbar_arrive(&p_full[sb]);
    }
    // ------------------------------------------------ normalise and store
#pragma unroll
    for (int h = 0; h < GH; ++h) red_sum[(grp * 4 + h) * 128 + r] = l[h];
    alive = softmax_and(alive);
    if (!alive) {
      if (lane == 0) at_status(p.status, kAtTimeoutSoftmax);
      *abort_flag = 1;
    } else {
      const bool row_ok = t < T;
      const bool warp_rows_ok = q0 + quarter * 32 + 31 < T;   // all 32 rows of this warp exist
      const long long ldo = (long long)p.H * kHD;
#pragma unroll 1
      for (int h = 0; h < GH; ++h) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&o_ready[h], (ntiles - 1) & 1, abort_flag))) {
          if (lane == 0) at_status(p.status, kAtTimeoutSoftmax);
          *abort_flag = 1;
          break;
        }
        tc_fence_after_sync();
        const float lt = red_sum[h * 128 + r] + red_sum[(4 + h) * 128 + r];
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        uint32_t ov[32];
        tmem_ld32(lane_base + h * kHD + grp * 32, ov);
        tmem_ld_wait();
        uint4 w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float *f = reinterpret_cast<const float *>(&ov[8 * q]);
          w[q] = make_uint4(pack_f16x2(f[0] * inv, f[1] * inv), pack_f16x2(f[2] * inv, f[3] * inv),
                            pack_f16x2(f[4] * inv, f[5] * inv), pack_f16x2(f[6] * inv, f[7] * inv));
        }
        if (warp_rows_ok) {
          // the warp's 32 rows x 32 columns go out as one TMA box (a lane per
          // row would make every store instruction 32 separate row segments)
          uint8_t *stg = smem + C::OFF_STG + (h * 8 + (warp - 2)) * C::STG_WARP;
#pragma unroll
          for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4 *>(stg + lane * 64 + q * 16) = w[q];
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmO, stg, (h_first + h) * kHD + grp * 32, b * T + q0 + quarter * 32);
            bulk_commit_group();
          }
        } else if (row_ok) {
          f16 *dst = p.o + ((long long)b * T + t) * ldo + (long long)(h_first + h) * kHD + grp * 32;
#pragma unroll
          for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4 *>(dst + 8 * q) = w[q];
        }
      }
    }
    if (lane == 0) bulk_wait_group_read<0>();     // the staging blocks are read before the CTA exits
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int GH, bool KM>
cudaError_t launch_ghk(const AttnParams &a, const CUtensorMap &tq, const CUtensorMap &tk,
                      const CUtensorMap &tv, const CUtensorMap &to, cudaStream_t st) {
  using C = AtCfg<GH>;
  auto kern = attn_tc_kernel<GH, KM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  AtParams p{};
  p.o = a.o;
  p.valid_start = a.valid_start;
  p.B = a.B; p.T = a.T; p.H = a.H; p.KV = a.KV;
  p.G = a.H / a.KV;
  p.GH = GH;
  p.n_hsub = p.G / GH;
  p.scale_log2 = a.scale_log2;
  p.window = a.window;
  p.key_mask = a.key_mask;
  p.Tk = a.Tk > 0 ? a.Tk : a.T;
  p.q_off = a.q_off;
  p.status = a.status;
  dim3 grid((unsigned)(a.B * a.KV * p.n_hsub), (unsigned)cdiv(a.T, kBQ), 1u);
  // as a programmatic dependent: CTAs set up barriers and TMEM while the
  // preceding kernel drains, and wait for it before touching its outputs
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, to, p);
}

template <int GH>
cudaError_t launch_gh(const AttnParams &a, const CUtensorMap &tq, const CUtensorMap &tk,
                      const CUtensorMap &tv, const CUtensorMap &to, cudaStream_t st) {
  return a.key_mask ? launch_ghk<GH, true>(a, tq, tk, tv, to, st) : launch_ghk<GH, false>(a, tq, tk, tv, to, st);
}

}  // namespace

bool attention_tc_supported(int hd, int H, int KV) {
  const int G = H / KV;
  return hd == kHD && (G == 1 || G == 2 || G == 3 || G == 4 || G == 6 || G == 8);
}

cudaError_t launch_attention_tc(const AttnParams &a, cudaStream_t st) {
  if (!attention_tc_supported(a.hd, a.H, a.KV) || a.v_t == nullptr) return cudaErrorInvalidConfiguration;
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_f16(&tq, a.q, (uint64_t)a.B * a.H * a.T, kHD, kHD, kBQ)) return cudaErrorInvalidValue;
  const int Tk = a.Tk > 0 ? a.Tk : a.T;
  if (Tk < a.T || a.q_off < 0 || a.q_off + a.T > Tk) return cudaErrorInvalidValue;
  if (!make_tmap_f16(&tk, a.k, (uint64_t)a.B * a.KV * Tk, kHD, kHD, kBK)) return cudaErrorInvalidValue;
  // V^T: rows are (b, kv head, dim), columns are keys; columns >= Tk read as zero
  if (!make_tmap_f16(&tv, a.v_t, (uint64_t)a.B * a.KV * kHD, Tk, a.T_pad, kHD)) return cudaErrorInvalidValue;
  // output rows [B*T, H*hd]: a softmax warp's 32 rows x 32 columns per box
  if (!make_tmap_2d(&to, a.o, (uint64_t)a.B * a.T, (uint64_t)a.H * kHD, (uint64_t)a.H * kHD, 32, 32, false))
    return cudaErrorInvalidValue;
  const int G = a.H / a.KV;
  switch (G) {
    case 1: return launch_gh<1>(a, tq, tk, tv, to, st);
    case 2: return launch_gh<2>(a, tq, tk, tv, to, st);
    case 3: return launch_gh<3>(a, tq, tk, tv, to, st);
    case 4: return launch_gh<4>(a, tq, tk, tv, to, st);
    case 6: return launch_gh<3>(a, tq, tk, tv, to, st);   // two CTAs per group of six
    case 8: return launch_gh<4>(a, tq, tk, tv, to, st);
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace smol
