// attention_tc.cu - causal grouped-query attention on tcgen05 (sm_103a), hd = 64.
//
// o[b,t,h,:] = sum_{j visible} softmax_j(q[b,h,t].k[b,h/g,j] / sqrt(hd)) v[b,h/g,j]
// with j visible iff valid_start[b] <= j <= t ("model.py" (SmolLM2-135M)
// section 4: scaled scores, triu(1) causal mask plus the padding mask, softmax,
// probs @ v; query head h reads key/value head h // g as in the "SmolLM3"
// page's "Grouped-query attention").  Rows with no visible key produce 0.
//
// One CTA owns (sequence b, query head h, 256 query tokens as two 128-row
// tiles A and B) and reads K/V of kv head h // g: never expanded per query
// head (the g heads of a group read the same K/V tiles, from L2).  Per
// 128-key tile j and query tile X:
//   S_X = Q_X K_j^T    tcgen05.mma M=128 N=128 K=64 into S_X (TMEM, fp32)
//   P_X = exp2(S*c-m)  softmax warpgroup X: one query row per thread, all 128
//                      keys (no reduction across threads); P as packed f16 over
//                      S_X's own TMEM columns
//   O_X += P_X V_j     tcgen05.mma with A (= P_X) read from TMEM, M=128 N=64 K=128
// The two tiles ping-pong: while warpgroup A turns S_A into P_A, the tensor
// core computes S_B or P_B V, and the other way round.  The running max is
// updated lazily: O_X is rescaled in TMEM only when a row's max grows by more
// than 2^8 (otherwise P may exceed 1 by up to 256, exact in the fp32 sums and
// within f16 range), the FlashAttention-4 idea.  Warp 0 issues TMA, warp 1
// allocates TMEM and one lane issues every MMA, warps 2..5 / 6..9 are the two
// softmax warpgroups.  All waits are bounded (status word + abort flag, copies
// and MMAs drained before exit).
#include <math.h>

#include "common.cuh"
#include "prims.cuh"

namespace smol {

namespace {

constexpr int kBQ = 128;      // query rows per tile (UMMA M)
constexpr int kBK = 128;      // keys per KV tile
constexpr int kHD = 64;
constexpr int kNS = 3;        // K / V^T pipeline stages
constexpr int kThreads = 320; // producer, MMA, two softmax warpgroups

struct AtCfg {
  static constexpr int Q_BYTES = kBQ * kHD * 2;         // one tile: [128][64] f16
  static constexpr int K_BYTES = kBK * kHD * 2;         // [128 keys][64]
  static constexpr int VT_SUB = kHD * 64 * 2;           // [64 dims][64 keys]
  static constexpr int VT_BYTES = 2 * VT_SUB;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_VT = OFF_K + kNS * K_BYTES;
  static constexpr int OFF_BAR = OFF_VT + kNS * VT_BYTES;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
  // TMEM columns: S_A 0..127, S_B 128..255 (P over their first 64), O_A 256.., O_B 320..
  static constexpr int TMEM_O = 256;
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

struct AtParams {
  f16 *o;                   // [B, T, H*hd]
  const int *valid_start;
  int B, T, H, KV, G;
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

// max(a, b, c) in one instruction (three-input max of sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void at_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// KV-tile range [lo, hi] of a 128-row query tile starting at q0 (hi < lo: the
// tile has no rows).
__device__ __forceinline__ void tile_range(int q0, int T, int vs, int &lo, int &hi) {
  if (q0 >= T) {
    lo = 0;
    hi = -1;
    return;
  }
  hi = min(q0 + kBQ - 1, T - 1) / kBK;
  lo = min(vs / kBK, hi);          // an all-padding tile still runs one (masked) tile
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmVt, const AtParams p) {
  using C = AtCfg;
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
  uint64_t *s_full = bars + 1 + 2 * kNS;     // [2] S_X(j) computed
  uint64_t *p_full = s_full + 2;             // [2] P_X(j) written (128 arrivals)
  uint64_t *s_free = s_full + 4;             // [2] P_X(j) V done: S_X free, O_X current
  uint64_t *o_done = s_full + 6;             // [2] every MMA of tile X complete
  uint64_t *drain = s_full + 8;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.T;
  // blocks are launched in linear order (x fastest): the query pair is the
  // slow index, descending, so the longest causal rows start first
  const int q0 = (gridDim.y - 1 - blockIdx.y) * (2 * kBQ);
  const int b = blockIdx.x / p.H, h = blockIdx.x - b * p.H;
  const int kvh = h / p.G;
  const int vs = p.valid_start ? min(max(p.valid_start[b], 0), T) : 0;
  int lo[2], hi[2];
  tile_range(q0, T, vs, lo[0], hi[0]);
  tile_range(q0 + kBQ, T, vs, lo[1], hi[1]);
  const int j_lo = hi[1] >= lo[1] ? min(lo[0], lo[1]) : lo[0];
  const int j_hi = max(hi[0], hi[1]);
  const int ntiles = j_hi - j_lo + 1;            // KV tiles loaded (>= 1: tile A has rows)

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 128);
      mbar_init(&s_free[x], 1);
      mbar_init(&o_done[x], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVt);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
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
      mbar_arrive_expect_tx(q_full, 2 * C::Q_BYTES);
      for (int x = 0; x < 2; ++x)                 // rows past T (tile B of the tail) read other rows
        tma_load_2d(sQ + x * C::Q_BYTES, &tmQ, q_full, 0, (b * p.H + h) * T + q0 + x * kBQ);
      for (int it = 0; it < ntiles && ok; ++it) {
        const int j = j_lo + it, st = it % kNS;
        if (!mbar_wait_bounded(&kv_empty[st], ((it / kNS) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&kv_full[st], C::K_BYTES + C::VT_BYTES);
        tma_load_2d(sK + st * C::K_BYTES, &tmK, &kv_full[st], 0, (b * p.KV + kvh) * T + j * kBK);
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
      constexpr uint32_t kIdescS = idesc_f16_f32(kBQ, kBK);
      constexpr uint32_t kIdescO = idesc_f16_f32(kBQ, kHD);
      bool ok = mbar_wait_bounded(q_full, 0, abort_flag), any = false;
      int n_pv[2] = {0, 0};                       // P V products issued per query tile
      auto active = [&](int x, int j) { return j >= lo[x] && j <= hi[x]; };
      // S_X(j) = Q_X K_j^T into S_X (j's K tile is in stage (j - j_lo) % kNS)
      auto issue_s = [&](int x, int j) {
        const int st = (j - j_lo) % kNS;
        const uint64_t a = sdesc_kmajor_sw128(smem_u32(sQ + x * C::Q_BYTES));
        const uint64_t bk = sdesc_kmajor_sw128(smem_u32(sK + st * C::K_BYTES));
#pragma unroll
        for (int k = 0; k < kHD / 16; ++k)
          umma_f16(tmem + x * kBK, a + 2 * k, bk + 2 * k, kIdescS, k > 0);
        umma_commit(&s_full[x]);
        any = true;
      };
      // the tiles' first S
      if (ok && !mbar_wait_bounded(&kv_full[0], 0, abort_flag)) ok = false;
      if (ok) {
        tc_fence_after_sync();
        for (int x = 0; x < 2; ++x)
          if (active(x, j_lo)) issue_s(x, j_lo);
      }
      // Per KV tile j, per query tile X: P_X(j) V_j as soon as softmax X has
      // written P_X(j), then right away S_X(j+1) - so the tensor core turns to
      // X's next scores while the other tile's softmax is still running (ping-pong).
      for (int it = 0; it < ntiles && ok; ++it) {
        const int j = j_lo + it, st = it % kNS;
        bool next_ready = false;
#pragma unroll 1
        for (int x = 0; x < 2 && ok; ++x) {
          if (active(x, j)) {
            if (!mbar_wait_bounded(&p_full[x], n_pv[x] & 1, abort_flag)) { ok = false; break; }
            tc_fence_after_sync();
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
              const uint64_t bv = sdesc_kmajor_sw128(smem_u32(sVt + st * C::VT_BYTES + kb * C::VT_SUB));
#pragma unroll
              for (int k = 0; k < 4; ++k)   // 16 keys of P = 8 TMEM columns per MMA
                umma_f16_tmem_a(tmem + C::TMEM_O + x * kHD, tmem + x * kBK + (kb * 4 + k) * 8, bv + 2 * k,
                                kIdescO, (j > lo[x]) || kb || k);
            }
            umma_commit(&s_free[x]);
            if (j == hi[x]) umma_commit(&o_done[x]);
            ++n_pv[x];
          }
          if (active(x, j + 1)) {
            if (!next_ready) {
              if (!mbar_wait_bounded(&kv_full[(it + 1) % kNS], ((it + 1) / kNS) & 1, abort_flag)) { ok = false; break; }
              next_ready = true;
            }
            // S_X shares its columns with P_X: the P V just issued must be done
            if (n_pv[x] > 0 && !mbar_wait_bounded(&s_free[x], (n_pv[x] - 1) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after_sync();
            issue_s(x, j + 1);
          }
        }
        if (!ok) break;
        umma_commit(&kv_empty[st]);               // both tiles' P V of block j issued
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
    // ---------------------------------------------- softmax warpgroup x (warps
    // 2..5: tile A, 6..9: tile B), one query row per thread, all 128 keys
    const int x = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;              // query row within the tile
    const int t = q0 + x * kBQ + r;
    const int tq0 = q0 + x * kBQ;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t s_col = lane_base + x * kBK;
    const uint32_t o_col = lane_base + C::TMEM_O + x * kHD;
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;                   // running max (exp2 domain) and sum
    bool alive = true;
    int n = 0;
    for (int j = lo[x]; j <= hi[x]; ++j, ++n) {
      const int k0 = j * kBK;                       // first key of this tile
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&s_full[x], n & 1, abort_flag))) {
        alive = false;
        break;
      }
      tc_fence_after_sync();
      const bool need_mask = (k0 + kBK - 1 > tq0) || (k0 < vs);
      const int hi_e = t - k0, lo_e = vs - k0;      // keys k0+e visible iff lo_e <= e <= hi_e
      // pass 1, the row max: the 128 scores in four loads in flight, one wait
      float mx;
      {
        uint32_t sv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(s_col + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]));
        tmem_ld_wait();
        float mc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (need_mask) {
#pragma unroll
          for (int e = 0; e < 128; ++e)
            if (e <= hi_e && e >= lo_e) mc[e & 3] = fmaxf(mc[e & 3], __uint_as_float(sv[e]));
        } else {
#pragma unroll
          for (int e = 0; e < 128; e += 2)
            mc[(e >> 1) & 3] = fmax3(mc[(e >> 1) & 3], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
        }
        mx = fmax3(fmaxf(mc[0], mc[1]), mc[2], mc[3]);
      }
      const float mxa = (mx == -INFINITY) ? -INFINITY : mx * sl2;   // into the exp2 domain
      float alpha = 1.f;
      const bool resc = (m != -INFINITY) && (mxa > m + 8.f);
      if (resc) {
        alpha = ex2_approx(m - mxa);
        l *= alpha;
        m = mxa;
      } else if (m == -INFINITY) {
        m = mxa;                                    // first visible key(s) of this row
      }
      if (__any_sync(0xffffffffu, resc)) {
        // O_X holds every earlier P V (S_X(j) was issued after P_X(j-1) V had
        // completed); rescale it in TMEM.  tcgen05.ld/st are warp-collective:
        // every lane takes part, alpha = 1 where the row's max did not move
        uint32_t ov[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          tmem_ld32(o_col + 32 * half, ov);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(o_col + 32 * half, ov);
        }
      }
      const float mu = (m == -INFINITY) ? 0.f : m;
      // pass 2: p = 2^(s*c - m) as f16 pairs over S_X's first 64 columns, in
      // two halves of 64 keys (half h -> columns 32h..32h+31, over scores
      // already read)
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t sv[64];
        tmem_ld32(s_col + 64 * hf, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(s_col + 64 * hf + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_ld_wait();
        uint32_t pk[32];
        if (need_mask) {
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            const int ee = 64 * hf + e;
            const float x0 = (ee <= hi_e && ee >= lo_e) ? fmaf(__uint_as_float(sv[e]), sl2, -mu) : -INFINITY;
            const float x1 = (ee + 1 <= hi_e && ee + 1 >= lo_e) ? fmaf(__uint_as_float(sv[e + 1]), sl2, -mu) : -INFINITY;
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            ps[(e >> 1) & 3] += p0 + p1;
            pk[e >> 1] = pack_f16x2(p0, p1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            const float p0 = ex2_approx(fmaf(__uint_as_float(sv[e]), sl2, -mu));
            const float p1 = ex2_approx(fmaf(__uint_as_float(sv[e + 1]), sl2, -mu));
            ps[(e >> 1) & 3] += p0 + p1;
            pk[e >> 1] = pack_f16x2(p0, p1);
          }
        }
        tmem_st32(s_col + 32 * hf, pk);
      }
      tmem_st_wait();                               // P (and any O rescale) visible to the MMA
      l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
      tc_fence_before_sync();
      mbar_arrive(&p_full[x]);
    }
    // ------------------------------------------------ normalise and store
    if (hi[x] >= lo[x]) {
      if (alive && !__all_sync(0xffffffffu, mbar_wait_bounded(&o_done[x], 0, abort_flag))) alive = false;
      if (!alive) {
        if (lane == 0) at_status(p.status, kAtTimeoutSoftmax);
        *abort_flag = 1;
      } else {
        tc_fence_after_sync();
        const bool row_ok = t < T;
        const long long ldo = (long long)p.H * kHD;
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t ov[32];
          tmem_ld32(o_col + 32 * half, ov);
          tmem_ld_wait();
          if (row_ok) {
            f16 *dst = p.o + ((long long)b * T + t) * ldo + (long long)h * kHD + half * 32;
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
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_at(const AttnParams &a, const CUtensorMap &tq, const CUtensorMap &tk,
                      const CUtensorMap &tv, cudaStream_t st) {
  using C = AtCfg;
  constexpr auto kern = attn_tc_kernel;
  cudaError_t e = ensure_smem_attr<kern>(C::SMEM);
  if (e != cudaSuccess) return e;
  AtParams p{};
  p.o = a.o;
  p.valid_start = a.valid_start;
  p.B = a.B; p.T = a.T; p.H = a.H; p.KV = a.KV;
  p.G = a.H / a.KV;
  p.scale_log2 = a.scale_log2;
  p.status = a.status;
  dim3 grid((unsigned)(a.B * a.H), (unsigned)cdiv(a.T, 2 * kBQ), 1u);
  kern<<<grid, kThreads, C::SMEM, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

bool attention_tc_supported(int hd, int H, int KV) { return hd == kHD && KV > 0 && H % KV == 0; }

cudaError_t launch_attention_tc(const AttnParams &a, cudaStream_t st) {
  if (!attention_tc_supported(a.hd, a.H, a.KV) || a.v_t == nullptr) return cudaErrorInvalidConfiguration;
  CUtensorMap tq, tk, tv;
  if (!get_tmap_f16(&tq, a.q, (uint64_t)a.B * a.H * a.T, kHD, kHD, kBQ)) return cudaErrorInvalidValue;
  if (!get_tmap_f16(&tk, a.k, (uint64_t)a.B * a.KV * a.T, kHD, kHD, kBK)) return cudaErrorInvalidValue;
  // V^T: rows are (b, kv head, dim), columns are keys; columns >= T read as zero
  if (!get_tmap_f16(&tv, a.v_t, (uint64_t)a.B * a.KV * kHD, a.T, a.T_pad, kHD)) return cudaErrorInvalidValue;
  return launch_at(a, tq, tk, tv, st);
}

}  // namespace smol
