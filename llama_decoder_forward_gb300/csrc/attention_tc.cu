// attention_tc.cu - causal grouped-query attention on tcgen05 (sm_103a), hd 64 or 128.
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
// hides further keys: each key tile gets the mask as one additive row of 0 and
// -inf, the same for every query row, added to S.  With a KV cache
// in front (prefill on top of a cache), query t is key q_off + t of a longer
// key sequence.
//
// One CTA owns (sequence b, kv head, a tile of 128 query tokens) and GH query
// heads of that kv head.  Each K tile [128 keys x hd] and V^T tile [hd x 128
// keys] is loaded once by TMA into shared memory and serves all GH heads: K/V
// are never expanded per query head.  Per (kv tile, head):
//   S = Q_h K^T        tcgen05.mma, M=128 N=128 K=hd, fp32 in TMEM (two S buffers
//                      taken in turn by the heads)
//   P = exp2(S*c - m)  a softmax warpgroup, one query row per thread,
//                      all 128 keys of the tile (no exchange between warps); P is
//                      written as f16 into the head's shared-memory P buffer, in the
//                      swizzled K-major layout of an MMA operand, and the S buffer is
//                      released as soon as it has been read
//   O_h += P [V | 1]   tcgen05.mma, M=128 N=hd+16 K=128: the hd value columns plus a
//                      constant row of ones appended to V^T, so column hd of the
//                      accumulator is the row sum of the very f16 P that weights V
// The tensor pipe is fed by three issuing warps: an issue of tcgen05.mma takes
// a fixed ~110 cycles of its issuing thread whatever N is (measured), so one
// thread issuing all twelve small MMAs of a (tile, head) would leave the pipe
// idle; several warps' MMAs run concurrently.  Warp 1 issues every S MMA, warps
// 2 and 3 the P V MMAs of alternate (tile, head) slots.
// The running max is updated lazily: O_h is rescaled in TMEM only when a row's
// max grows by more than 2^8 (otherwise P may exceed 1 by up to 256, exact in
// the fp32 sums and within f16 range), the FlashAttention-4 idea.
// Warp 0 issues TMA (and, with a key mask, turns the tile's mask bytes into
// its additive row).  Warps 4.. form two softmax warpgroups (one when GH = 1) that
// take the (tile, head) slots in turn; a head's running row max passes from
// one to the other through shared memory.  All waits are bounded (status
// word + abort flag, copies and MMAs drained before exit).
#include <math.h>

#include "common.cuh"
#include "prims.cuh"

namespace smol {

namespace {

constexpr int kBQ = 128;      // query rows per tile (UMMA M)
constexpr int kBK = 128;      // keys per KV tile
constexpr int kNST = 2;       // K/V stages
constexpr int kTmemS = 256;   // S buffers at TMEM columns 256 and 384

// HD = head dim (64 or 128).  Q and K tiles are HD/64 swizzled sub-tiles of
// 64 columns; a V^T half tile holds the HD value rows and 16 constant rows.
template <int HD, int GH>
struct AtCfg {
  static constexpr int NO = HD + 16;                    // accumulator columns per head: HD values, the row sum, 15 zero
  static constexpr int NSUB = HD / 64;                  // 64-column sub-tiles of a Q or K tile
  static constexpr int NG = (GH == 1 && HD == 64) ? 1 : 2;   // softmax warpgroups, taking the slots in turn
  static constexpr int THREADS = 128 * (1 + NG);        // one control warpgroup + NG softmax warpgroups
  static constexpr int Q_BYTES = kBQ * HD * 2;          // one head: NSUB x [128 rows][64] f16
  static constexpr int K_BYTES = kBK * HD * 2;          // NSUB x [128 keys][64]
  static constexpr int VT_TMA = HD * 128;               // [HD dims][64 keys], written by TMA
  static constexpr int VT_SUB = NO * 128;               // + [16 rows][64 keys]: a row of ones, 15 of zeros
  static constexpr int VT_BYTES = 2 * VT_SUB;           // keys 0..63 and 64..127 of the tile
  static constexpr int P_SUB = kBQ * 128;               // [128 rows][64 keys] f16
  static constexpr int P_BYTES = 2 * P_SUB;             // one head's P, also its output staging
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + GH * Q_BYTES;
  static constexpr int OFF_VT = OFF_K + kNST * K_BYTES;
  static constexpr int OFF_P = OFF_VT + kNST * VT_BYTES;
  static constexpr int OFF_MASK = OFF_P + GH * P_BYTES;   // [kNST][128] key-mask bias (0 or -inf) per key
  static constexpr int OFF_MANY = OFF_MASK + kNST * kBK * 4;  // [kNST] the tile hides some key (int)
  static constexpr int OFF_MST = OFF_MANY + 16;         // [GH][128] running row max per head
  static constexpr int OFF_BAR = OFF_MST + GH * 128 * 4;
  static constexpr int NBAR = 1 + 4 * kNST + 4 + 5 * GH + 3;
  static constexpr int SMEM = 1024 + OFF_BAR + NBAR * 8 + 16;
  static_assert(GH >= 1 && GH * NO <= kTmemS, "O accumulators must fit below the S buffers");
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

struct AtParams {
  f16 *o;                   // [B, T, H*hd]
  const int *valid_start;
  const int *seq_order;     // [B] or nullptr: sequence of the CTAs' sequence slot
  const uint8_t *key_mask;  // [B, T] or nullptr: key j of sequence b hidden where 0
  int B, T, H, KV, G, GH, n_hsub;
  float scale_log2;
  int window;               // > 0: query t sees keys j > t - window only
  int Tk, q_off;            // keys per sequence; key index of query 0
  unsigned long long wait_ns;   // limit of the bounded waits (drains keep 1 s)
  int *status;
  int *done_out;            // or nullptr: +1 at done_out[b * T / 128 + query tile] when written
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

// (a0, a1) * b + c on the packed two-lane fp32 pipe path (one instruction).
__device__ __forceinline__ float2 ffma2(float a0, float a1, float b, float c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %4};\n\t"
      "mov.b64 rc, {%5, %5};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
  return d;
}

// (a0 + b0, a1 + b1) on the packed two-lane fp32 path (one instruction).
__device__ __forceinline__ float2 fadd2(float a0, float a1, float b0, float b1) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
  return d;
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

template <int HD, int GH, bool KM>
__global__ void __launch_bounds__(AtCfg<HD, GH>::THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmVt, const __grid_constant__ CUtensorMap tmO,
                   const AtParams p) {
  using C = AtCfg<HD, GH>;
  constexpr int NO = C::NO;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + C::OFF_Q;
  uint8_t *sK = smem + C::OFF_K;
  uint8_t *sVt = smem + C::OFF_VT;
  uint8_t *sP = smem + C::OFF_P;
  float *sBias = reinterpret_cast<float *>(smem + C::OFF_MASK);
  int *sBiasAny = reinterpret_cast<int *>(smem + C::OFF_MANY);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1;                // [kNST] K of a tile landed
  uint64_t *k_empty = k_full + kNST;          // [kNST] every head's S of the tile done
  uint64_t *v_full = k_empty + kNST;          // [kNST] V^T of a tile (and its key-mask row) landed
  uint64_t *v_empty = v_full + kNST;          // [kNST] every head's P V of the tile done (GH commits)
  uint64_t *s_full = v_empty + kNST;          // [2] S computed
  uint64_t *s_free = s_full + 2;              // [2] S read by its softmax warpgroup (128 arrivals)
  // [GH][2] P of the head written for tiles of even / odd index (128 arrivals).
  // Split by tile parity so that each barrier has one waiter that sees every
  // phase: a P V warp takes a given head only every other tile, and a parity
  // wait two phases behind would pass early.
  uint64_t *p_full = s_free + 2;
  uint64_t *pv_done = p_full + 2 * GH;        // [GH][2] P V of the head done, per tile parity
  uint64_t *m_ready = pv_done + 2 * GH;       // [GH] running max of the head's rows stored (128 arrivals)
  uint64_t *drain = m_ready + GH;             // [3] one per MMA-issuing warp (warps 1, 2, 3)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 3);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.T;
  // blocks are launched in linear order (x fastest): the query tile is the
  // slow index, descending, so every sequence's longest causal tiles start
  // first and the short ones fill the tail (longest-processing-time order)
  const int q0 = (gridDim.y - 1 - blockIdx.y) * kBQ;
  const int groups = p.KV * p.n_hsub;
  const int bslot = blockIdx.x / groups;
  const int b = p.seq_order ? p.seq_order[bslot] : bslot;   // the sequence (longest first with an order)
  const int kvh = (blockIdx.x - bslot * groups) / p.n_hsub;
  const int hsub = blockIdx.x - bslot * groups - kvh * p.n_hsub;
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
    for (int i = 0; i < kNST; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], GH);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
    }
    for (int h = 0; h < GH; ++h) {
      mbar_init(&p_full[2 * h], 128);
      mbar_init(&p_full[2 * h + 1], 128);
      mbar_init(&pv_done[2 * h], 1);
      mbar_init(&pv_done[2 * h + 1], 1);
      mbar_init(&m_ready[h], 128);
    }
    for (int i = 0; i < 3; ++i) mbar_init(&drain[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVt);
    tma_prefetch_desc(&tmO);
  }
  // the constant rows under each V^T half tile: row 64 all ones (its product
  // with P is the row sum of P), rows 65..79 zero; TMA never writes them
  for (int i = threadIdx.x; i < kNST * 2 * 16 * 8; i += C::THREADS) {
    const int sub = i >> 7, row = (i >> 3) & 15, ch = i & 7;
    const uint32_t w = row == 0 ? 0x3c003c00u : 0u;
    *reinterpret_cast<uint4 *>(sVt + sub * C::VT_SUB + C::VT_TMA + row * 128 + ch * 16) = make_uint4(w, w, w, w);
  }
  fence_proxy_async_smem();
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
    // ---------------------------------------------------- TMA producer
    // K of a tile is released once its S MMAs are done and V only after its
    // P V MMAs, so K runs one tile ahead: K(0), K(1), V(0), K(2), V(1), ...
    griddep_wait();                               // q, k and V^T come from the preceding kernel
    int nk = 0, nv = 0;                           // K and V tiles issued (for the drain)
    bool ok = true;
    // with a key mask: this lane's bytes of the next V tile's keys, loaded a
    // tile ahead so that their latency stays off the V loads
    const uint8_t *km = KM ? p.key_mask + (long long)b * T : nullptr;
    uint32_t mb[4] = {0u, 0u, 0u, 0u};
    if constexpr (KM) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int key = j_lo * kBK + 32 * w + lane;
        mb[w] = key < T ? km[key] : 0u;
      }
    }
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, GH * C::Q_BYTES);
      for (int h = 0; h < GH; ++h)
        for (int qs = 0; qs < C::NSUB; ++qs)
          tma_load_2d(sQ + h * C::Q_BYTES + qs * (kBQ * 128), &tmQ, q_full, qs * 64,
                      ((b * p.H) + h_first + h) * T + q0);
    }
    for (int it = -1; it < ntiles && ok; ++it) {
      const int ik = it + 1;                      // K tile issued in this step
      if (ik < ntiles) {
        const int st = ik % kNST;
        if (lane == 0) {
          ok = mbar_wait_bounded(&k_empty[st], ((ik / kNST) & 1) ^ 1, abort_flag, p.wait_ns);
          if (ok) {
            mbar_arrive_expect_tx(&k_full[st], C::K_BYTES);
            for (int ks = 0; ks < C::NSUB; ++ks)
              tma_load_2d(sK + st * C::K_BYTES + ks * (kBK * 128), &tmK, &k_full[st], ks * 64,
                          (b * p.KV + kvh) * Tk + (j_lo + ik) * kBK);
            ++nk;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      if (it < 0) continue;
      const int j = j_lo + it, st = it % kNST;
      if (lane == 0) ok = mbar_wait_bounded(&v_empty[st], ((it / kNST) & 1) ^ 1, abort_flag, p.wait_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if constexpr (KM) {
        // the tile's key mask as one additive row (0 visible, -inf hidden; the
        // same for every query row): key j*128 + 32w + e is bit e of word w,
        // and lane 0 writes the row (or only marks a tile that hides no key)
        uint32_t bits[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) bits[w] = __ballot_sync(0xffffffffu, mb[w] != 0u);
        if (it + 1 < ntiles) {
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int key = (j + 1) * kBK + 32 * w + lane;
            mb[w] = key < T ? km[key] : 0u;
          }
        }
        if (lane == 0) {
          const int any = (bits[0] & bits[1] & bits[2] & bits[3]) != ~0u;
          sBiasAny[st] = any;
          if (any) {
            float4 *row = reinterpret_cast<float4 *>(sBias + st * kBK);
#pragma unroll
            for (int e4 = 0; e4 < kBK / 4; ++e4) {
              const uint32_t nib = bits[e4 >> 3] >> ((e4 & 7) * 4);
              row[e4] = make_float4((nib & 1u) ? 0.f : -INFINITY, (nib & 2u) ? 0.f : -INFINITY,
                                    (nib & 4u) ? 0.f : -INFINITY, (nib & 8u) ? 0.f : -INFINITY);
            }
          }
        }
      }
      if (lane == 0) {
        // the arrive below also releases the mask row to the softmax warps
        mbar_arrive_expect_tx(&v_full[st], 2 * C::VT_TMA);
        tma_load_2d(sVt + st * C::VT_BYTES, &tmVt, &v_full[st], j * kBK, (b * p.KV + kvh) * HD);
        tma_load_2d(sVt + st * C::VT_BYTES + C::VT_SUB, &tmVt, &v_full[st], j * kBK + 64,
                    (b * p.KV + kvh) * HD);
        ++nv;
      }
    }
    if (lane == 0) {
      // wait (bounded) until every copy this thread issued has landed
      if (!mbar_wait_drain(q_full, 0)) at_status(p.status, kAtTimeoutDrain);
      if (!ok) {
        at_status(p.status, kAtTimeoutLoad);
        *abort_flag = 1;
        for (int i = nk > kNST ? nk - kNST : 0; i < nk; ++i)
          if (!mbar_wait_drain(&k_full[i % kNST], (uint32_t)((i / kNST) & 1)))
            at_status(p.status, kAtTimeoutDrain);
        for (int i = nv > kNST ? nv - kNST : 0; i < nv; ++i)
          if (!mbar_wait_drain(&v_full[i % kNST], (uint32_t)((i / kNST) & 1)))
            at_status(p.status, kAtTimeoutDrain);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------- S = Q_h K^T issuer
      constexpr uint32_t kIdescS = idesc_f16_f32(kBQ, kBK);
      bool ok = mbar_wait_bounded(q_full, 0, abort_flag, p.wait_ns), any = false;
      for (int s = 0; s < nslots && ok; ++s) {
        const int it = s / GH, h = s - it * GH, sb = s & 1, st = it % kNST;
        if (!mbar_wait_bounded(&s_free[sb], ((s >> 1) & 1) ^ 1, abort_flag, p.wait_ns)) { ok = false; break; }
        if (h == 0 && !mbar_wait_bounded(&k_full[st], (it / kNST) & 1, abort_flag, p.wait_ns)) { ok = false; break; }
        tc_fence_after_sync();
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          // k step k: sub-tile k / 4, +32 bytes per 16 columns inside it
          const uint64_t a = sdesc_kmajor_sw128(smem_u32(sQ + h * C::Q_BYTES + (k >> 2) * (kBQ * 128)));
          const uint64_t bk = sdesc_kmajor_sw128(smem_u32(sK + st * C::K_BYTES + (k >> 2) * (kBK * 128)));
          umma_f16(tmem + kTmemS + sb * kBK, a + 2 * (k & 3), bk + 2 * (k & 3), kIdescS, k > 0);
        }
        any = true;
        umma_commit(&s_full[sb]);
        if (h == GH - 1) umma_commit(&k_empty[st]);   // every head's S of the tile issued
      }
      if (!ok) {
        at_status(p.status, kAtTimeoutMma);
        *abort_flag = 1;
        if (any) {
          // wait for this warp's MMAs already issued before TMEM is freed
          umma_commit(&drain[warp - 1]);
          if (!mbar_wait_drain(&drain[warp - 1], 0)) at_status(p.status, kAtTimeoutDrain);
        }
      }
    }
  } else if (warp < 4) {
    if (lane == 0) {
      // ---------------------------------------------------- O_h += P_h [V | 1] issuer
      // warp 2 takes the even slots, warp 3 the odd ones.  A head's P V MMAs of
      // consecutive tiles never overlap even when issued from different warps:
      // P of the next tile is written only after the previous P V is done.
      constexpr uint32_t kIdescO = idesc_f16_f32(kBQ, NO);
      const int par = warp - 2;
      bool ok = true, any = false;
      for (int s = par; s < nslots && ok; s += 2) {
        const int it = s / GH, h = s - it * GH, st = it % kNST;
        if (!mbar_wait_bounded(&p_full[2 * h + (it & 1)], (it >> 1) & 1, abort_flag, p.wait_ns)) { ok = false; break; }
        if (!mbar_wait_bounded(&v_full[st], (it / kNST) & 1, abort_flag, p.wait_ns)) { ok = false; break; }
        tc_fence_after_sync();
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint64_t ap = sdesc_kmajor_sw128(smem_u32(sP + h * C::P_BYTES + kb * C::P_SUB));
          const uint64_t bv = sdesc_kmajor_sw128(smem_u32(sVt + st * C::VT_BYTES + kb * C::VT_SUB));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_f16(tmem + h * NO, ap + 2 * k, bv + 2 * k, kIdescO, (it | kb | k) != 0);
        }
        any = true;
        umma_commit(&pv_done[2 * h + (it & 1)]);
        umma_commit(&v_empty[st]);
      }
      if (!ok) {
        at_status(p.status, kAtTimeoutMma);
        *abort_flag = 1;
        if (any) {
          // wait for this warp's MMAs already issued before TMEM is freed
          umma_commit(&drain[warp - 1]);
          if (!mbar_wait_drain(&drain[warp - 1], 0)) at_status(p.status, kAtTimeoutDrain);
        }
      }
    }
  } else {
    griddep_wait();                               // o is written below
    // ---------------------------------------------- softmax warpgroup g: slots g, g + NG, ...
    const int g = (warp - 4) >> 2;
    const int quarter = warp & 3;                   // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;              // query row within the tile
    const int t = q0 + r;
    const int tk = qo + t;                          // this row's own key index
    const int row_lo = p.window > 0 ? max(vs, tk - p.window + 1) : vs;   // this row's first visible key
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float *m_state = reinterpret_cast<float *>(smem + C::OFF_MST);      // [GH][128]
    const float sl2 = p.scale_log2;
    bool alive = true;
    for (int s = g; s < nslots; s += C::NG) {
      const int it = s / GH, h = s - it * GH, sb = s & 1, st = it % kNST;
      const int k0 = (j_lo + it) * kBK;             // first key of the tile
      const bool need_mask =
          (k0 + kBK - 1 > qo + q0) || (k0 < vs) || (p.window > 0 && k0 <= qo + last_q - p.window);
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&s_full[sb], (s >> 1) & 1, abort_flag, p.wait_ns))) {
        alive = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t sv[128];
      const uint32_t s_col = lane_base + kTmemS + sb * kBK;
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_col + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]));
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(&s_free[sb]);                     // the S buffer may be overwritten now
      if constexpr (KM) {
        // the tile's key-mask row, published with its V^T: s + (-inf) = -inf
        // hides a key, s + 0 leaves it (every row reads the same 128 values)
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&v_full[st], (it / kNST) & 1, abort_flag, p.wait_ns))) {
          alive = false;
          break;
        }
        const float4 *row = reinterpret_cast<const float4 *>(sBias + st * kBK);
        if (sBiasAny[st])
#pragma unroll
        for (int e4 = 0; e4 < kBK / 4; ++e4) {
          const float4 bb = row[e4];
          const float2 x = fadd2(__uint_as_float(sv[4 * e4]), __uint_as_float(sv[4 * e4 + 1]), bb.x, bb.y);
          const float2 y = fadd2(__uint_as_float(sv[4 * e4 + 2]), __uint_as_float(sv[4 * e4 + 3]), bb.z, bb.w);
          sv[4 * e4] = __float_as_uint(x.x);
          sv[4 * e4 + 1] = __float_as_uint(x.y);
          sv[4 * e4 + 2] = __float_as_uint(y.x);
          sv[4 * e4 + 3] = __float_as_uint(y.y);
        }
      }
      // keys hidden by the causal, padding and window limits become -inf in
      // place, so one code path serves masked and unmasked tiles
      if (need_mask) {
        const int hi = tk - k0, lo = row_lo - k0;   // keys k0+e visible iff lo <= e <= hi
#pragma unroll
        for (int e = 0; e < kBK; ++e)
          if (!(e <= hi && e >= lo)) sv[e] = 0xff800000u;
      }
      // row max; eight independent chains
      float mc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) mc[q] = -INFINITY;
#pragma unroll
      for (int e = 0; e < kBK; e += 2)
        mc[(e >> 1) & 7] = fmax3(mc[(e >> 1) & 7], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
      const float mx = fmaxf(fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3])),
                             fmaxf(fmaxf(mc[4], mc[5]), fmaxf(mc[6], mc[7])));
      const float mxa = (mx == -INFINITY) ? -INFINITY : mx * sl2;   // into the exp2 domain
      // the head's running max (exp2 domain), left by whichever warpgroup took
      // its previous tile
      float m = -INFINITY;
      if (it > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&m_ready[h], (it - 1) & 1, abort_flag, p.wait_ns))) {
          alive = false;
          break;
        }
        m = m_state[h * 128 + r];
      }
      float alpha = 1.f;
      const bool resc = (m != -INFINITY) && (mxa > m + 8.f);
      if (resc) {
        alpha = ex2_approx(m - mxa);
        m = mxa;
      } else if (m == -INFINITY) {
        m = mxa;                                    // first visible key(s) of this row
      }
      // publish the max at once, so that the group taking the head's next tile
      // can start its exponents.  pv_done is one barrier per (head, tile
      // parity), and whoever waits for tile i's P V below has itself waited
      // for tile i - 2's (a head's tiles alternate between the two groups, or
      // all go to one), so no parity wait runs two phases behind its barrier.
      m_state[h * 128 + r] = m;
      mbar_arrive(&m_ready[h]);
      // P V of the head's previous tile must be done: it reads the P buffer,
      // and a rescale of O must not race its accumulation
      if (it > 0 && !__all_sync(0xffffffffu, mbar_wait_bounded(&pv_done[2 * h + ((it - 1) & 1)], ((it - 1) >> 1) & 1,
                                                              abort_flag, p.wait_ns))) {
        alive = false;
        break;
      }
      if (__any_sync(0xffffffffu, resc)) {
        // O_h (and its row-sum column) *= alpha, sixteen columns at a time
        tc_fence_after_sync();
        const uint32_t o_col = lane_base + h * NO;
#pragma unroll 1
        for (int c = 0; c < NO; c += 16) {
          uint32_t ov[16];
          tmem_ld16(o_col + c, ov);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st16(o_col + c, ov);
        }
        tmem_st_wait();
      }
      const float mu = (m == -INFINITY) ? 0.f : m;
      // p = 2^(s*c - m) as f16, eight keys per 16-byte chunk of the row, in the
      // 128-byte swizzled layout (chunk c of row r at r*128 + 16*(c ^ (r & 7)))
      uint8_t *pbuf = sP + h * C::P_BYTES;
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        uint8_t *row_base = pbuf + kb * C::P_SUB + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int e0 = kb * 64 + c * 8;
          uint32_t pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 x = ffma2(__uint_as_float(sv[e0 + 2 * q]), __uint_as_float(sv[e0 + 2 * q + 1]), sl2, -mu);
            pk[q] = pack_f16x2(ex2_approx(x.x), ex2_approx(x.y));
          }
          *reinterpret_cast<uint4 *>(row_base + ((c ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      fence_proxy_async_smem();                     // P visible to the tensor core
      tc_fence_before_sync();                       // and the rescale's TMEM stores ordered before it
      mbar_arrive(&p_full[2 * h + (it & 1)]);
    }
    // ------------------------------------------------ normalise and store
    // each head is finished by the warpgroup that took its last tile
#pragma unroll 1
    for (int h = 0; h < GH; ++h) {
      if (((ntiles - 1) * GH + h) % C::NG != g) continue;
      if (alive &&
          !__all_sync(0xffffffffu, mbar_wait_bounded(&pv_done[2 * h + ((ntiles - 1) & 1)], ((ntiles - 1) >> 1) & 1,
                                                     abort_flag, p.wait_ns)))
        alive = false;
      if (!alive) break;
      tc_fence_after_sync();
      uint32_t ov[32], os[16];
      const uint32_t o_col = lane_base + h * NO;
      tmem_ld16(o_col + HD, os);
      tmem_ld_wait();
      const float lt = __uint_as_float(os[0]);
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const bool row_ok = t < T;
      const bool warp_rows_ok = q0 + quarter * 32 + 31 < T;   // all 32 rows of this warp exist
      f16 *dst = p.o + ((long long)b * T + t) * ((long long)p.H * HD) + (long long)(h_first + h) * HD;
#pragma unroll 1
      for (int j = 0; j < C::NSUB; ++j) {
        // the warp's 32 rows x 64 columns j*64.. staged in sub-tile j of the
        // head's (now free) P buffer, swizzled
        uint8_t *stg = sP + h * C::P_BYTES + j * C::P_SUB + quarter * 32 * 128;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          tmem_ld32(o_col + j * 64 + 32 * half, ov);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float *f = reinterpret_cast<const float *>(&ov[8 * q]);
            const uint4 w = make_uint4(pack_f16x2(f[0] * inv, f[1] * inv), pack_f16x2(f[2] * inv, f[3] * inv),
                                       pack_f16x2(f[4] * inv, f[5] * inv), pack_f16x2(f[6] * inv, f[7] * inv));
            const int c = half * 4 + q;
            if (warp_rows_ok)
              *reinterpret_cast<uint4 *>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) = w;
            else if (row_ok)
              *reinterpret_cast<uint4 *>(dst + j * 64 + 8 * c) = w;
          }
        }
        if (warp_rows_ok) {
          // one TMA box per warp and 64 columns (a lane per row would make
          // every store instruction 32 separate row segments)
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmO, stg, (h_first + h) * HD + j * 64, b * T + q0 + quarter * 32);
            bulk_commit_group();
          }
        }
      }
    }
    if (!alive) {
      if (lane == 0) at_status(p.status, kAtTimeoutSoftmax);
      *abort_flag = 1;
    }
    // the staging is read before the CTA exits; with a completion flag the
    // stores must also be complete
    if (lane == 0) {
      if (p.done_out) bulk_wait_group<0>();
      else bulk_wait_group_read<0>();
    }
  }

  if (p.done_out) __threadfence();                // every lane's direct row stores
  tc_fence_before_sync();
  __syncthreads();
  if (p.done_out && threadIdx.x == 0) {
    fence_proxy_async_global();
    flag_add_release(p.done_out + b * (T / kBQ) + q0 / kBQ, 1);
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int HD, int GH, bool KM>
cudaError_t launch_ghk(const AttnParams &a, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &to, cudaStream_t st) {
  using C = AtCfg<HD, GH>;
  auto kern = attn_tc_kernel<HD, GH, KM>;
  cudaError_t e = ensure_smem_attr<attn_tc_kernel<HD, GH, KM>>(C::SMEM);
  if (e != cudaSuccess) return e;
  AtParams p{};
  p.o = a.o;
  p.valid_start = a.valid_start;
  p.seq_order = a.seq_order;
  p.key_mask = a.key_mask;
  p.B = a.B; p.T = a.T; p.H = a.H; p.KV = a.KV;
  p.G = a.H / a.KV;
  p.GH = GH;
  p.n_hsub = p.G / GH;
  p.scale_log2 = a.scale_log2;
  p.window = a.window;
  p.Tk = a.Tk > 0 ? a.Tk : a.T;
  p.q_off = a.q_off;
  p.wait_ns = a.wait_ns ? a.wait_ns : kWaitTimeoutNs;
  p.status = a.status;
  p.done_out = (a.done_out && a.T % kBQ == 0 && (a.Tk <= 0 || a.Tk == a.T)) ? a.done_out : nullptr;
  dim3 grid((unsigned)(a.B * a.KV * p.n_hsub), (unsigned)cdiv(a.T, kBQ), 1u);
  // as a programmatic dependent: CTAs set up barriers and TMEM while the
  // preceding kernel drains, and wait for it before touching its outputs
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, to, p);
}

template <int HD, int GH>
cudaError_t launch_gh(const AttnParams &a, const CUtensorMap &tq, const CUtensorMap &tk,
                      const CUtensorMap &tv, const CUtensorMap &to, cudaStream_t st) {
  return a.key_mask ? launch_ghk<HD, GH, true>(a, tq, tk, tv, to, st)
                    : launch_ghk<HD, GH, false>(a, tq, tk, tv, to, st);
}

}  // namespace

int attention_tc_ctas_per_tile(int hd, int H, int KV) {
  if (!attention_tc_supported(hd, H, KV)) return 0;
  const int G = H / KV;
  const int GH = hd == 128 ? 1 : (G % 3 == 0 ? 3 : (G % 2 == 0 ? 2 : 1));
  return KV * (G / GH);
}

bool attention_tc_supported(int hd, int H, int KV) {
  return (hd == 64 || hd == 128) && KV > 0 && H >= KV && H % KV == 0;
}

cudaError_t launch_attention_tc(const AttnParams &a, cudaStream_t st) {
  if (!attention_tc_supported(a.hd, a.H, a.KV) || a.v_t == nullptr) return cudaErrorInvalidConfiguration;
  const int HDv = a.hd;
  CUtensorMap tq, tk, tv, to;
  if (!get_tmap_f16(&tq, a.q, (uint64_t)a.B * a.H * a.T, HDv, HDv, kBQ)) return cudaErrorInvalidValue;
  const int Tk = a.Tk > 0 ? a.Tk : a.T;
  if (Tk < a.T || a.q_off < 0 || a.q_off + a.T > Tk) return cudaErrorInvalidValue;
  if (a.key_mask && Tk != a.T) return cudaErrorInvalidValue;
  if (!get_tmap_f16(&tk, a.k, (uint64_t)a.B * a.KV * Tk, HDv, HDv, kBK)) return cudaErrorInvalidValue;
  // V^T: rows are (b, kv head, dim), columns are keys; columns >= Tk read as zero
  if (!get_tmap_f16(&tv, a.v_t, (uint64_t)a.B * a.KV * HDv, Tk, a.T_pad, HDv)) return cudaErrorInvalidValue;
  // output rows [B*T, H*hd]: a softmax warp's 32 rows x 64 columns per box, swizzled
  if (!get_tmap_2d(&to, a.o, (uint64_t)a.B * a.T, (uint64_t)a.H * HDv, (uint64_t)a.H * HDv, 64, 32, true))
    return cudaErrorInvalidValue;
  const int G = a.H / a.KV;
  if (HDv == 128) return launch_gh<128, 1>(a, tq, tk, tv, to, st);   // one query head per CTA
  // the group's heads split over G / GH CTAs: three heads per CTA where G is
  // a multiple of 3, two where it is even, else one (groups of 5 and 7)
  if (G % 3 == 0) return launch_gh<64, 3>(a, tq, tk, tv, to, st);
  if (G % 2 == 0) return launch_gh<64, 2>(a, tq, tk, tv, to, st);
  return launch_gh<64, 1>(a, tq, tk, tv, to, st);
}

}  // namespace smol
