// decode.cu - one KV-cache decode step on B sequences ("model.py"
// (SmolLM2-135M) section 4, the past_key_value branch: the new token's q and
// k are rotated at position past_len, k and v are concatenated after the
// cached ones, and with a single new token no causal mask applies; section 7
// generate slices the RoPE rows at past_len).
//
// Per layer: QKV GEMM (rstd, RoPE at cache_len[b], k/v written to k_new/v_new)
// -> split-K decode attention over cache_len[b] cached keys plus the new key
// -> O GEMM + residual -> gate/up GEMM + SwiGLU -> down GEMM + residual.
// Then the tied head.  The GEMMs are the tcgen05 kernel of gemm.cu with M = B.
//
// Decode attention is bound by HBM bandwidth (it streams the cache).  One CTA
// owns (sequence b, kv head, a chunk of kChunk keys) and all g query heads of
// that kv head, so each cached key/value is read once for the whole group.
// One thread fetches the chunk's K and V rows with two bulk copies (the TMA
// engine) into shared memory, so the whole chunk is in flight at once while
// other CTAs on the SM compute.  Keys are then spread over lane groups of hd/8
// lanes (16-byte reads, 8 dims per lane); each lane group takes 4 keys per
// step, reduces the q.k partial dots with shuffles and updates an online
// softmax in the exp2 domain.  Partial (max, sum, output) triples are merged inside the
// warp, then across warps in shared memory, then across chunks by the last
// CTA of the (b, kv head) pair (an atomic arrival counter, no waiting).
#include <math.h>

#include "decode.cuh"
#include "profile.cuh"
#include "prims.cuh"

namespace smol {

constexpr int kChunk = 256;        // keys per CTA
constexpr int kDecWarps = 4;       // warps per CTA

struct DecWs {
  size_t status, x, h, q, o, a, ssq_a, ssq_b, part_m, part_l, part_o, counters, total;
  int max_splits;
};

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static DecWs dec_ws(const smol_config *c, int B) {
  DecWs W{};
  const size_t d = c->hidden, hd = c->head_dim, H = c->n_heads, KV = c->n_kv_heads,
               I = c->intermediate;
  W.max_splits = (int)cdiv(c->max_pos, kChunk);
  size_t o = 0;
  W.status = o; o += 1024;
  W.x = o; o = align_up(o + B * d * 2, 1024);
  W.h = o; o = align_up(o + B * d * 2, 1024);
  W.q = o; o = align_up(o + B * H * hd * 2, 1024);
  W.o = o; o = align_up(o + B * H * hd * 2, 1024);
  W.a = o; o = align_up(o + B * I * 2, 1024);
  W.ssq_a = o; o = align_up(o + B * 4, 1024);
  W.ssq_b = o; o = align_up(o + B * 4, 1024);
  W.part_m = o; o = align_up(o + (size_t)B * H * W.max_splits * 4, 1024);
  W.part_l = o; o = align_up(o + (size_t)B * H * W.max_splits * 4, 1024);
  W.part_o = o; o = align_up(o + (size_t)B * H * W.max_splits * hd * 4, 1024);
  W.counters = o; o = align_up(o + (size_t)B * KV * 4, 1024);
  W.total = o;
  return W;
}

size_t decode_ws_bytes(const smol_config *cfg, int B) { return dec_ws(cfg, B).total; }

struct DecAttnParams {
  const f16 *q;             // [B, H, hd] (already rotated)
  const bf16 *k_cache, *v_cache;   // this layer: [B, KV, S_max, hd]
  const bf16 *k_new, *v_new;       // this layer: [B, KV, hd]
  const int *cache_len;
  f16 *o;                   // [B, H * hd], the O projection's f16 operand
  float *part_m, *part_l, *part_o; // [B, H, max_splits] and [B, H, max_splits, hd]
  int *counters;            // [B, KV], zero between layers
  int B, H, KV, S_max, max_pos, max_splits;
  float scale_log2;
  int *status;              // workspace status word (bounded wait)
  int layer;                // layer index (row offset into the whole-cache tensor maps)
};

// Launches `kern` as a programmatic dependent of the preceding kernel in the
// stream (it calls griddep_wait() before touching that kernel's outputs).
template <typename Kern, typename... Args>
static cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, int smem, cudaStream_t st,
                              const Args &...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Writes this CTA's (max, sum, output) triple for each head of the group and,
// if it is the last CTA of its (sequence, kv head) to finish, merges all the
// chunks' triples into the attention output.  red_m/red_l/red_o hold the
// per-warp triples ([NW][GM], [NW][GM], [NW][GM][HD]) in shared memory.
template <int HD, int GM, int NW>
__device__ __forceinline__ void chunk_partial_and_combine(const DecAttnParams &p, int b, int kvh,
                                                          int split, int nsplit, const float *red_m,
                                                          const float *red_l, const float *red_o,
                                                          int *s_last) {
  const int G = p.H / p.KV;
  const long long row = (long long)b * p.KV + kvh;
  const long long pbase = (long long)b * p.H + kvh * G;   // first head of the group
  for (int t = threadIdx.x; t < G * HD; t += blockDim.x) {
    const int g = t / HD, dim = t - g * HD;
    float M = -INFINITY;
    for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w * GM + g]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float Ls = 0.f, Os = 0.f;
    for (int w = 0; w < NW; ++w) {
      const float f = exp2f(red_m[w * GM + g] - Mu);
      Ls += red_l[w * GM + g] * f;
      Os += red_o[(w * GM + g) * HD + dim] * f;
    }
    const long long ps = (pbase + g) * p.max_splits + split;
    if (dim == 0) {
      p.part_m[ps] = M;
      p.part_l[ps] = Ls;
    }
    p.part_o[ps * HD + dim] = Os;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(p.counters + row, 1);
    *s_last = (prev == nsplit - 1);
  }
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  for (int t = threadIdx.x; t < G * HD; t += blockDim.x) {
    const int g = t / HD, dim = t - g * HD;
    const long long ps0 = (pbase + g) * p.max_splits;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, __ldcg(p.part_m + ps0 + s));
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float Ls = 0.f, Os = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float f = exp2f(__ldcg(p.part_m + ps0 + s) - Mu);
      Ls += __ldcg(p.part_l + ps0 + s) * f;
      Os += __ldcg(p.part_o + (ps0 + s) * HD + dim) * f;
    }
    p.o[(pbase + g) * HD + dim] = __float2half_rn(Ls > 0.f ? Os / Ls : 0.f);
  }
  if (threadIdx.x == 0) p.counters[row] = 0;        // ready for the next layer
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *ptr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(ptr)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *ptr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(ptr)));
}
// Splits x into bf16 hi + lo with hi + lo == x to about 16 significant bits.
__device__ __forceinline__ void split_bf16(float x, float &hi, float &lo) {
  hi = __bfloat162float(__float2bfloat16_rn(x));
  lo = x - hi;
}

// Decode attention on tensor cores (hd = 64).  One CTA = (sequence, kv head,
// 256-key chunk); 2-D TMA (128-byte swizzle) brings the chunk's K and V rows
// into shared memory; each of the 4 warps takes 64 keys with mma.sync
// m16n8k16 (bf16, the cache's type).  The g query heads of the group occupy
// A rows 0..g-1 as the bf16 "hi" part of q and rows 8..8+g-1 as the "lo"
// remainder, so one MMA yields both halves and their sum (in the same
// thread) carries q to ~16 bits; the probabilities P are split the same way
// for P V.  Keys past the chunk's valid range are masked (V rows zeroed so
// unused cache slots cannot inject NaN).
template <int GM>
__global__ void __launch_bounds__(128) decode_attn_mma_kernel(const __grid_constant__ CUtensorMap tmK,
                                                              const __grid_constant__ CUtensorMap tmV,
                                                              const DecAttnParams p) {
  constexpr int HD = 64, NW = 4;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t *dsm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t *sK = dsm;                     // [256 keys][128 B], 16-byte chunks swizzled by key & 7
  uint8_t *sV = dsm + kChunk * 128;
  uint64_t *kv_bar = reinterpret_cast<uint64_t *>(dsm + 2 * kChunk * 128);
  int *s_last = reinterpret_cast<int *>(kv_bar + 1);
  float *red_m = reinterpret_cast<float *>(kv_bar + 2);     // [NW][GM]
  float *red_l = red_m + NW * GM;                            // [NW][GM]
  float *red_o = red_l + NW * GM;                            // [NW][GM][HD]

  const int G = p.H / p.KV;
  const int b = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int Lb = p.cache_len[b];
  const int lmax = min(p.S_max, p.max_pos - 1);
  Lb = Lb < 0 ? 0 : (Lb > lmax ? lmax : Lb);
  const int n_keys = Lb + 1;
  const int nsplit = (n_keys + kChunk - 1) / kChunk;
  if (split >= nsplit) return;
  const int k_begin = split * kChunk;
  const int n_valid = min(kChunk, n_keys - k_begin);
  const long long row = (long long)b * p.KV + kvh;

  if (threadIdx.x == 0) {
    mbar_init(kv_bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // the cache is an input of the step, not written by any kernel of it: its
    // chunk is requested before waiting for the preceding kernel
    const int y = static_cast<int>(((long long)p.layer * p.B + b) * p.KV + kvh) * p.S_max + k_begin;
    mbar_arrive_expect_tx(kv_bar, 2 * kChunk * 128);
    tma_load_2d(sK, &tmK, kv_bar, 0, y);
    tma_load_2d(sV, &tmV, kv_bar, 0, y);
    griddep_launch_dependents();
  }
  griddep_wait();                                  // q, k_new, v_new, partials, counters
  // q as A fragments (rows r < G: hi; rows r + 8: lo), built while the copy flies
  const int r = lane >> 2, c2 = (lane & 3) * 2;
  uint32_t qa[4][4];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    if (r < G) {
      const f16 *qr = p.q + ((long long)b * p.H + kvh * G + r) * HD + kk * 16 + c2;
      const float2 lo2 = unpack_f16x2(*reinterpret_cast<const uint32_t *>(qr));
      const float2 hi2 = unpack_f16x2(*reinterpret_cast<const uint32_t *>(qr + 8));
      float h0, l0, h1, l1, h2, l2, h3, l3;
      split_bf16(lo2.x, h0, l0);
      split_bf16(lo2.y, h1, l1);
      split_bf16(hi2.x, h2, l2);
      split_bf16(hi2.y, h3, l3);
      qa[kk][0] = pack_bf16x2(h0, h1);
      qa[kk][1] = pack_bf16x2(l0, l1);
      qa[kk][2] = pack_bf16x2(h2, h3);
      qa[kk][3] = pack_bf16x2(l2, l3);
    } else {
      qa[kk][0] = qa[kk][1] = qa[kk][2] = qa[kk][3] = 0u;
    }
  }
  {
    int no_abort = 0;
    const bool landed = mbar_wait_bounded(kv_bar, 0, &no_abort);
    if (!__syncthreads_and(landed)) {
      if (threadIdx.x == 0) atomicCAS(p.status, 0, kDevTimeoutProducer);
      mbar_wait_bounded(kv_bar, 0, &no_abort);   // (bounded) drain before exiting
      return;
    }
  }
  // the new token's key/value into its slot; zero V rows past the valid keys
  if (Lb >= k_begin && Lb < k_begin + kChunk) {
    const int slot = Lb - k_begin;
    if (threadIdx.x < 8) {
      const int c = threadIdx.x;
      *reinterpret_cast<uint4 *>(sK + slot * 128 + ((c ^ (slot & 7)) << 4)) =
          reinterpret_cast<const uint4 *>(p.k_new + row * HD)[c];
      *reinterpret_cast<uint4 *>(sV + slot * 128 + ((c ^ (slot & 7)) << 4)) =
          reinterpret_cast<const uint4 *>(p.v_new + row * HD)[c];
    }
  }
  for (int i = n_valid * 8 + threadIdx.x; i < kChunk * 8; i += blockDim.x)
    reinterpret_cast<uint4 *>(sV)[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();

  const int kw0 = warp * 64;                       // this warp's first key (chunk-relative)
  float mw = -INFINITY, lw = 0.f;
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  if (kw0 < n_valid) {                             // warp-uniform
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = kw0 + j * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int chunk = kk * 2 + ((lane >> 3) & 1);
        uint32_t bk[4];
        ldsm_x4(bk, sK + key * 128 + ((chunk ^ (key & 7)) << 4));
        mma_bf16_16816(s[2 * j], qa[kk], bk[0], bk[1]);
        mma_bf16_16816(s[2 * j + 1], qa[kk], bk[2], bk[3]);
      }
    }
    // head r's score = hi row + lo row; mask keys past the valid range
    float sc[8][2];
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = kw0 + 8 * j + c2 + e;
        const float v = key < n_valid ? (s[j][e] + s[j][2 + e]) * p.scale_log2 : -INFINITY;
        sc[j][e] = v;
        mx = fmaxf(mx, v);
      }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mu = (mx == -INFINITY) ? 0.f : mx;
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sc[j][0] = exp2f(sc[j][0] - mu);
      sc[j][1] = exp2f(sc[j][1] - mu);
      sum += sc[j][0] + sc[j][1];
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    mw = mx;
    lw = sum;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      float h0, l0, h1, l1, h2, l2, h3, l3;
      split_bf16(sc[2 * kk][0], h0, l0);
      split_bf16(sc[2 * kk][1], h1, l1);
      split_bf16(sc[2 * kk + 1][0], h2, l2);
      split_bf16(sc[2 * kk + 1][1], h3, l3);
      const uint32_t a[4] = {pack_bf16x2(h0, h1), pack_bf16x2(l0, l1), pack_bf16x2(h2, h3),
                             pack_bf16x2(l2, l3)};
#pragma unroll
      for (int nd = 0; nd < 4; ++nd) {
        const int key = kw0 + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int chunk = nd * 2 + (lane >> 4);
        uint32_t bv[4];
        ldsm_x4_t(bv, sV + key * 128 + ((chunk ^ (key & 7)) << 4));
        mma_bf16_16816(o[2 * nd], a, bv[0], bv[1]);
        mma_bf16_16816(o[2 * nd + 1], a, bv[2], bv[3]);
      }
    }
  }
  // this warp's triple for head r (lanes 4r..4r+3), output dims 8i + c2 + e
  if (r < G) {
    if ((lane & 3) == 0) {
      red_m[warp * GM + r] = mw;
      red_l[warp * GM + r] = lw;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      red_o[(warp * GM + r) * HD + 8 * i + c2] = o[i][0] + o[i][2];
      red_o[(warp * GM + r) * HD + 8 * i + c2 + 1] = o[i][1] + o[i][3];
    }
  }
  __syncthreads();
  chunk_partial_and_combine<HD, GM, NW>(p, b, kvh, split, nsplit, red_m, red_l, red_o, s_last);
}


// GM: compile-time bound on the group size g = H / KV (arrays are sized GM).
template <int HD, int GM>
__global__ void __launch_bounds__(kDecWarps * 32) decode_attn_kernel(const DecAttnParams p) {
  if (threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();
  extern __shared__ __align__(128) uint8_t dsm[];
  bf16 *sK = reinterpret_cast<bf16 *>(dsm);          // [kChunk][HD]
  bf16 *sV = sK + kChunk * HD;                       // [kChunk][HD]
  uint64_t *kv_bar = reinterpret_cast<uint64_t *>(sV + kChunk * HD);
  constexpr int LPK = HD / 8;            // lanes per key
  constexpr int KPW = 32 / LPK;          // keys per warp step (per lane group: 1)
  constexpr int NB = 4;                  // keys per lane group per step
  const int G = p.H / p.KV;
  const int b = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPK, sub = lane % LPK;   // key group in the warp, dim chunk

  int Lb = p.cache_len[b];
  const int lmax = min(p.S_max, p.max_pos - 1);
  Lb = Lb < 0 ? 0 : (Lb > lmax ? lmax : Lb);
  const int n_keys = Lb + 1;                       // cached keys + the new one
  const int nsplit = (n_keys + kChunk - 1) / kChunk;
  if (split >= nsplit) return;
  const int k_begin = split * kChunk;
  const int k_end = min(k_begin + kChunk, n_keys);

  // q for the G heads of this kv head: 8 dims per lane, pre-scaled into exp2 domain
  float qv[GM][8];
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    if (g < G) {
      const uint4 u = *reinterpret_cast<const uint4 *>(p.q + ((long long)b * p.H + kvh * G + g) * HD + sub * 8);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_f16x2(w[e]);
        qv[g][2 * e] = f.x * p.scale_log2;
        qv[g][2 * e + 1] = f.y * p.scale_log2;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) qv[g][e] = 0.f;   // heads beyond the group are never written
    }
  }
  float m[GM], l[GM], acc[GM][8];
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
  }

  const long long row = (long long)b * p.KV + kvh;
  const bf16 *kc = p.k_cache + row * p.S_max * HD;
  const bf16 *vc = p.v_cache + row * p.S_max * HD;
  const bf16 *kn = p.k_new + row * HD;
  const bf16 *vn = p.v_new + row * HD;

  // the chunk's cached rows [k_begin, min(k_end, Lb)) arrive by bulk copy; the
  // new key (index Lb), if it falls in this chunk, is copied by the threads
  const int n_cached = max(0, min(k_end, Lb) - k_begin);
  if (threadIdx.x == 0) {
    mbar_init(kv_bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (n_cached > 0) {
      const uint32_t bytes = static_cast<uint32_t>(n_cached) * HD * 2;
      mbar_arrive_expect_tx(kv_bar, 2 * bytes);
      bulk_load(sK, kc + (long long)k_begin * HD, bytes, kv_bar);
      bulk_load(sV, vc + (long long)k_begin * HD, bytes, kv_bar);
    } else {
      mbar_arrive(kv_bar);
    }
  }
  if (Lb >= k_begin && Lb < k_end) {
    const int slot = Lb - k_begin;
    for (int i = threadIdx.x; i < HD / 8; i += blockDim.x) {
      reinterpret_cast<uint4 *>(sK + slot * HD)[i] = reinterpret_cast<const uint4 *>(kn)[i];
      reinterpret_cast<uint4 *>(sV + slot * HD)[i] = reinterpret_cast<const uint4 *>(vn)[i];
    }
  }
  {
    int no_abort = 0;
    const bool landed = mbar_wait_bounded(kv_bar, 0, &no_abort);
    if (!__syncthreads_and(landed)) {
      if (threadIdx.x == 0) atomicCAS(p.status, 0, kDevTimeoutProducer);
      // wait (bounded) once more for the copies before the CTA exits
      mbar_wait_bounded(kv_bar, 0, &no_abort);
      return;
    }
  }

  const int step = kDecWarps * KPW * NB;           // keys per CTA step
  // The trip count depends on the warp only: every lane runs every iteration,
  // so the full-warp shuffles below never see a lane that has left the loop.
  for (int wbase = k_begin + warp * KPW * NB; wbase < k_end; wbase += step) {
    const int base = wbase + grp * NB;
    uint4 kr[NB], vr[NB];
    bool valid[NB];
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int j = base + i;
      valid[i] = j < k_end;
      if (valid[i]) {
        kr[i] = *reinterpret_cast<const uint4 *>(sK + (j - k_begin) * HD + sub * 8);
        vr[i] = *reinterpret_cast<const uint4 *>(sV + (j - k_begin) * HD + sub * 8);
      } else {
        kr[i] = make_uint4(0, 0, 0, 0);
        vr[i] = make_uint4(0, 0, 0, 0);
      }
    }
    // scores of the NB keys for every head of the group (K converted once per key)
    float sc[GM][NB];
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const uint32_t kw[4] = {kr[i].x, kr[i].y, kr[i].z, kr[i].w};
      float kf[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 a = unpack_bf16x2(kw[e]);
        kf[2 * e] = a.x;
        kf[2 * e + 1] = a.y;
      }
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        float t = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) t = fmaf(qv[g][e], kf[e], t);
#pragma unroll
        for (int off = LPK / 2; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        sc[g][i] = valid[i] ? t : -INFINITY;
      }
    }
    // online-softmax update: one rescale per head per NB keys
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      float mx = m[g];
#pragma unroll
      for (int i = 0; i < NB; ++i) mx = fmaxf(mx, sc[g][i]);
      const float mu = (mx == -INFINITY) ? 0.f : mx;
      const float alpha = exp2f(m[g] - mu);
      m[g] = mx;
      float lsum = l[g] * alpha;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[g][e] *= alpha;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        sc[g][i] = exp2f(sc[g][i] - mu);
        lsum += sc[g][i];
      }
      l[g] = lsum;
    }
    // accumulate P V (V converted once per key)
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const uint32_t vw[4] = {vr[i].x, vr[i].y, vr[i].z, vr[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 c = unpack_bf16x2(vw[e]);
#pragma unroll
        for (int g = 0; g < GM; ++g) {
          acc[g][2 * e] = fmaf(sc[g][i], c.x, acc[g][2 * e]);
          acc[g][2 * e + 1] = fmaf(sc[g][i], c.y, acc[g][2 * e + 1]);
        }
      }
    }
  }

  // merge the KPW lane groups of the warp (lanes with equal `sub`)
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    if (g < G) {
#pragma unroll
      for (int off = LPK; off < 32; off <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[g], off);
        const float lo = __shfl_xor_sync(0xffffffffu, l[g], off);
        const float mx = fmaxf(m[g], mo);
        const float mu = (mx == -INFINITY) ? 0.f : mx;
        const float a0 = exp2f(m[g] - mu), a1 = exp2f(mo - mu);
        l[g] = l[g] * a0 + lo * a1;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float ao = __shfl_xor_sync(0xffffffffu, acc[g][e], off);
          acc[g][e] = acc[g][e] * a0 + ao * a1;
        }
        m[g] = mx;
      }
    }
  }

  __shared__ float red_m[kDecWarps * GM], red_l[kDecWarps * GM];
  __shared__ float red_o[kDecWarps * GM * HD];
  __shared__ int s_last;
  if (grp == 0) {
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      if (g < G) {
        if (sub == 0) {
          red_m[warp * GM + g] = m[g];
          red_l[warp * GM + g] = l[g];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) red_o[(warp * GM + g) * HD + sub * 8 + e] = acc[g][e];
      }
    }
  }
  __syncthreads();
  chunk_partial_and_combine<HD, GM, kDecWarps>(p, b, kvh, split, nsplit, red_m, red_l, red_o, &s_last);
}

template <int HD, int GM>
static cudaError_t launch_decode_attn_g(const DecAttnParams &ap, dim3 grid, cudaStream_t st) {
  const int smem = 2 * kChunk * HD * 2 + 16;
  constexpr auto kern = decode_attn_kernel<HD, GM>;
  cudaError_t e = ensure_smem_attr<kern>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, dim3(kDecWarps * 32), smem, st, ap);
}

template <int HD>
static cudaError_t launch_decode_attn_hd(const DecAttnParams &ap, dim3 grid, cudaStream_t st) {
  const int G = ap.H / ap.KV;
  if (G == 1) return launch_decode_attn_g<HD, 1>(ap, grid, st);
  if (G == 2) return launch_decode_attn_g<HD, 2>(ap, grid, st);
  if (G == 3) return launch_decode_attn_g<HD, 3>(ap, grid, st);
  if (G == 4) return launch_decode_attn_g<HD, 4>(ap, grid, st);
  return launch_decode_attn_g<HD, 8>(ap, grid, st);
}

template <int GM>
static cudaError_t launch_decode_attn_mma_g(const CUtensorMap &tk, const CUtensorMap &tv,
                                            const DecAttnParams &ap, dim3 grid, cudaStream_t st) {
  constexpr int NW = 4, HD = 64;
  const int smem = 1024 + 2 * kChunk * 128 + 16 + (2 * NW * GM + NW * GM * HD) * 4;
  constexpr auto kern = decode_attn_mma_kernel<GM>;
  cudaError_t e = ensure_smem_attr<kern>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, dim3(NW * 32), smem, st, tk, tv, ap);
}

// head_dim 64 runs on tensor cores (the cache seen as one 2-D tensor of
// L*B*KV*S_max rows of 64 values); other head sizes on the CUDA-core kernel.
static cudaError_t launch_decode_attn(const DecAttnParams &ap, int hd, dim3 grid, cudaStream_t st,
                                      const bf16 *k_all, const bf16 *v_all, int L) {
  if (hd == 64) {
    CUtensorMap tk, tv;
    const uint64_t rows = (uint64_t)L * ap.B * ap.KV * ap.S_max;
    if (!get_tmap_f16(&tk, k_all, rows, 64, 64, kChunk)) return cudaErrorInvalidValue;
    if (!get_tmap_f16(&tv, v_all, rows, 64, 64, kChunk)) return cudaErrorInvalidValue;
    const int G = ap.H / ap.KV;
    if (G == 1) return launch_decode_attn_mma_g<1>(tk, tv, ap, grid, st);
    if (G == 2) return launch_decode_attn_mma_g<2>(tk, tv, ap, grid, st);
    if (G == 3) return launch_decode_attn_mma_g<3>(tk, tv, ap, grid, st);
    if (G == 4) return launch_decode_attn_mma_g<4>(tk, tv, ap, grid, st);
    return launch_decode_attn_mma_g<8>(tk, tv, ap, grid, st);
  }
  return launch_decode_attn_hd<128>(ap, grid, st);
}

__global__ void zero_ints_kernel(int *p, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = 0;
}

static cudaError_t launch_zero_ints(int *p, int n, cudaStream_t st) {
  zero_ints_kernel<<<(unsigned)cdiv(n, 256), 256, 0, st>>>(p, n);
  return cudaGetLastError();
}

cudaError_t run_decode(const DecodeArgs &a, void *ws, int sms, cudaStream_t st, int *launches) {
  const smol_config &c = a.cfg;
  const DecWs W = dec_ws(&c, a.B);
  uint8_t *wb = static_cast<uint8_t *>(ws);
  const int B = a.B, d = c.hidden, H = c.n_heads, KV = c.n_kv_heads, hd = c.head_dim,
            I = c.intermediate, L = c.n_layers, V = c.vocab;
  int *status = reinterpret_cast<int *>(wb + W.status);
  f16 *x = reinterpret_cast<f16 *>(wb + W.x);
  f16 *h = reinterpret_cast<f16 *>(wb + W.h);
  f16 *q = reinterpret_cast<f16 *>(wb + W.q);
  f16 *o = reinterpret_cast<f16 *>(wb + W.o);
  f16 *act = reinterpret_cast<f16 *>(wb + W.a);
  float *ssq_a = reinterpret_cast<float *>(wb + W.ssq_a);
  float *ssq_b = reinterpret_cast<float *>(wb + W.ssq_b);
  int *counters = reinterpret_cast<int *>(wb + W.counters);
  int n = 0;
  cudaError_t e;
#define DEC_LAUNCH_K(kind, expr)     \
  do {                               \
    prof_before((kind), st);         \
    e = (expr);                      \
    prof_after((kind), st);          \
    if (e != cudaSuccess) return e;  \
    ++n;                             \
  } while (0)
#define DEC_LAUNCH(expr) DEC_LAUNCH_K(SMOL_K_OTHER, expr)

  DEC_LAUNCH(launch_zero_ints(counters, B * KV, st));
  DEC_LAUNCH_K(SMOL_K_EMBED, launch_embed_rows(a.ids, a.embed, V, d, B, x, nullptr, ssq_a, st));

  const float sl2 = 1.4426950408889634f / sqrtf((float)hd);
  for (int l = 0; l < L; ++l) {
    const uint8_t *lb = a.layer0 + (size_t)l * a.layer_bytes;
    const size_t kv_layer = (size_t)B * KV * hd;
    bf16 *kn = a.k_new + (size_t)l * kv_layer;
    bf16 *vn = a.v_new + (size_t)l * kv_layer;

    GemmParams p{};
    p.M = B; p.N = (H + 2 * KV) * hd; p.K = d;
    p.ssq_in = ssq_a; p.inv_dim = 1.0f / d; p.eps = c.rms_eps; p.ssq_zero = ssq_b;
    p.q = q; p.k_bf = kn; p.v_bf = vn; p.T = 1; p.H = H; p.KV = KV; p.hd = hd;
    p.rope = a.rope; p.valid_start = nullptr; p.pos_add = a.cache_len; p.pos_limit = min(a.S_max, c.max_pos - 1);
    p.max_pos = c.max_pos; p.status = status; p.pdl = 1;
    DEC_LAUNCH_K(SMOL_K_QKV, launch_gemm(kEpiQkvRope, hd, x, lb + a.off_qkv, p, sms, st));

    DecAttnParams ap{};
    ap.q = q;
    ap.k_cache = a.k_cache + (size_t)l * B * KV * a.S_max * hd;
    ap.v_cache = a.v_cache + (size_t)l * B * KV * a.S_max * hd;
    ap.k_new = kn; ap.v_new = vn; ap.cache_len = a.cache_len; ap.o = o;
    ap.part_m = reinterpret_cast<float *>(wb + W.part_m);
    ap.part_l = reinterpret_cast<float *>(wb + W.part_l);
    ap.part_o = reinterpret_cast<float *>(wb + W.part_o);
    ap.counters = counters;
    ap.B = B; ap.H = H; ap.KV = KV; ap.S_max = a.S_max; ap.max_pos = c.max_pos;
    ap.max_splits = W.max_splits; ap.scale_log2 = sl2; ap.status = status;
    const int lmax = min(a.S_max, c.max_pos - 1);
    dim3 grid((unsigned)cdiv(lmax + 1, kChunk), (unsigned)KV, (unsigned)B);
    ap.layer = l;
    DEC_LAUNCH_K(SMOL_K_DEC_ATTN, launch_decode_attn(ap, hd, grid, st, a.k_cache, a.v_cache, L));

    GemmParams po{};
    po.M = B; po.N = d; po.K = H * hd; po.out = h; po.out_is_f16 = 1; po.ldo = d; po.resid_f16 = x;
    po.ssq_out = ssq_b;
    po.status = status; po.pdl = 1;
    DEC_LAUNCH_K(SMOL_K_OPROJ, launch_gemm(kEpiResidual, 64, o, lb + a.off_o, po, sms, st));

    GemmParams pg{};
    pg.M = B; pg.N = 2 * I; pg.K = d; pg.out = act; pg.out_is_f16 = 1; pg.ldo = I; pg.ssq_in = ssq_b;
    pg.inv_dim = 1.0f / d; pg.eps = c.rms_eps; pg.ssq_zero = ssq_a; pg.status = status; pg.pdl = 1;
    DEC_LAUNCH_K(SMOL_K_GATEUP, launch_gemm(kEpiSwiglu, 128, h, lb + a.off_gu, pg, sms, st));

    GemmParams pd{};
    pd.M = B; pd.N = d; pd.K = I; pd.out = x; pd.out_is_f16 = 1; pd.ldo = d; pd.resid_f16 = h;
    pd.ssq_out = ssq_a;
    pd.status = status; pd.pdl = 1;
    DEC_LAUNCH_K(SMOL_K_DOWN, launch_gemm(kEpiResidual, 64, act, lb + a.off_down, pd, sms, st));
  }
  GemmParams ph{};
  ph.M = B; ph.N = V; ph.K = d; ph.out = a.logits; ph.out_is_f16 = 0; ph.ldo = V; ph.ssq_in = ssq_a;
  ph.inv_dim = 1.0f / d; ph.eps = c.rms_eps; ph.status = status; ph.pdl = 1;
  DEC_LAUNCH_K(SMOL_K_HEAD, launch_gemm(kEpiScale, gemm_pick_bn(kEpiScale, V, hd), x, a.head, ph, sms, st));
#undef DEC_LAUNCH
  *launches = n;
  return cudaSuccess;
}

}  // namespace smol
