// decode.cu - one KV-cache decode step on B sequences ("model.py"
// (SmolLM2-135M) section 4, the past_key_value branch: the new token's q and
// k are rotated at position past_len, k and v are concatenated after the
// cached ones, and with a single new token no causal mask applies; section 7
// generate slices the RoPE rows at past_len).
//
// Per layer: QKV projection (rstd, RoPE at cache_len[b], k/v written to
// k_new/v_new) -> decode attention over cache_len[b] cached keys plus the new
// key -> O projection + residual -> gate/up + SwiGLU -> down + residual.  Then
// the tied head.  The SmolLM3 per-block variants ("SmolLM3" page: "Every
// fourth block has no rotary", "A sliding window the 3B checkpoints leave
// off"): a NoPE block skips the rotation; a block with window w attends over
// the cache slots [cache_len[b] - w + 1, cache_len[b]) and the new key, each
// kernel shifting its slice of the cache by the first visible slot.  For batches of at most 64 rows the projections run on the
// narrow-unit kernel of decode_gemm.cu, otherwise on the tcgen05 GEMM of
// gemm.cu with M = B; every launch is a programmatic dependent of the one
// before (weights and cache chunks are requested before the wait).
//
// Decode attention is bound by HBM bandwidth (it streams the cache) and reads
// each cached key/value once for all g query heads of its kv head.  For head
// dim 64 and up to kDecMaxB sequences it is a persistent kernel (one CTA per
// SM streaming a contiguous range of (sequence, kv head, 256-key chunk)
// items through a TMA ring, tensor cores for the dot products, merge warps for
// the softmax states; see decode_attn_persist_kernel).  The per-chunk kernels
// below it serve larger batches (decode_attn_mma_kernel, one CTA per chunk)
// and head dim 128 (decode_attn_kernel on CUDA cores: lane groups of hd/8
// lanes take 8 dims each, 16-byte reads, shuffle-reduced dot products and an
// online softmax in the exp2 domain); their chunks' (max, sum, output)
// triples are merged by the last CTA of each (sequence, kv head) (an atomic
// arrival counter, no waiting).
#include <math.h>

#include "decode.cuh"
#include "profile.cuh"
#include "prims.cuh"

namespace smol {

constexpr int kChunk = 256;        // keys per CTA
constexpr int kDecWarps = 4;       // warps per CTA

struct DecWs {
  size_t status, x, h, q, o, a, ssq_a, ssq_b, part_m, part_l, part_o, counters, argmax, total;
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
  // B x KV arrival counters, then B packed row maxima of the logits (one
  // contiguous range, cleared by one kernel at the start of the step)
  W.counters = o; o += (size_t)B * KV * 4;
  o = align_up(o, 8);
  W.argmax = o; o = align_up(o + (size_t)B * 8, 1024);
  W.total = o;
  return W;
}

size_t decode_ws_bytes(const smol_config *cfg, int B) { return dec_ws(cfg, B).total; }

// The cache slots a new token at position Lb (already clamped) attends over:
// [first, Lb), plus its own key.  A window w keeps the w - 1 slots before it.
__device__ __forceinline__ int dec_first_slot(int Lb, int window) {
  return window > 0 ? max(0, Lb - window + 1) : 0;
}

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
  int window;               // > 0: only cache slots j >= cache_len - window + 1 are read
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
  const int first = dec_first_slot(Lb, p.window);   // keys below are outside the window
  Lb -= first;                                      // from here on: visible cached keys
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
    const int y = static_cast<int>(((long long)p.layer * p.B + b) * p.KV + kvh) * p.S_max + first + k_begin;
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


// Persistent decode attention on tensor cores (hd = 64).  The work items are
// (sequence, kv head, 256-key chunk), numbered sequence-major; CTA c takes the
// contiguous range [c*per, (c+1)*per) (per = ceil(items / CTAs)), so every CTA
// streams about the same number of K/V bytes.  Three kinds of warps:
//  - a producer warp keeps a ring of NS chunks in flight (two 2-D TMA boxes
//    each, 128-byte swizzle);
//  - eight compute warps take 32 keys each of every chunk with the same bf16
//    hi/lo mma.sync scheme as decode_attn_mma_kernel and carry a running
//    (max, sum, output) per warp across the chunks of one (sequence, kv head).
//    They never wait for one another: each releases a ring slot on its own;
//  - two merge warps: when a CTA's run of chunks of a pair ends, the compute
//    warps hand their states over through one of two shared-memory buffers
//    (runs alternate between them) and go on with the next pair, while the
//    buffer's merge warp combines the eight states.  A pair covered by one CTA is written directly; otherwise each
//    CTA writes a partial and the last to finish (atomic counter, no waiting)
//    merges them.
constexpr int kDecMaxB = 2048;                    // per-sequence tables in shared memory
constexpr int kPersistWarps = 8;                  // compute warps: 32 keys of every chunk each

template <int GM>
__host__ __device__ constexpr int persist_stages() { return GM <= 4 ? 3 : 2; }

// Shared memory of the persistent kernel: ring, barriers, two merge buffers,
// the clamped cache lengths and the chunk prefix sums.
template <int GM>
constexpr int persist_smem_fixed() {
  return 1024 + persist_stages<GM>() * 2 * kChunk * 128 + (2 * persist_stages<GM>() + 4) * 8 + 16 +
         2 * kPersistWarps * GM * (2 + 64) * 4;
}

template <int GM>
__global__ void __launch_bounds__((kPersistWarps + 3) * 32, 1) decode_attn_persist_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                     const __grid_constant__ CUtensorMap tmV,
                                                                     const DecAttnParams p) {
  constexpr int HD = 64, NW = kPersistWarps, NS = persist_stages<GM>();
  constexpr int KPW = kChunk / NW;                // keys per warp
  constexpr int N16 = KPW / 16;                   // 16-key groups per warp
  constexpr int STAGE = 2 * kChunk * 128;         // K and V rows of one chunk
  constexpr int RED = NW * GM * (2 + HD);         // floats of one merge buffer
  extern __shared__ uint8_t dsm_raw[];
  uint8_t *dsm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(dsm + NS * STAGE);   // [NS]
  uint64_t *empty = full + NS;                                        // [NS], NW arrivals
  uint64_t *mfull = empty + NS;                                       // [2], NW * 32 arrivals
  uint64_t *mempty = mfull + 2;                                       // [2], 32 arrivals (merge warp m owns buffer m)
  volatile int *abort_flag = reinterpret_cast<int *>(mempty + 2);
  float *red = reinterpret_cast<float *>(mempty + 2) + 4;             // [2][RED]
  int *lens = reinterpret_cast<int *>(red + 2 * RED);                 // [B] clamped cache lengths
  int *prefix = lens + p.B;                                           // [B + 1] chunks before sequence b

  const int G = p.H / p.KV;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lmax = min(p.S_max, p.max_pos - 1);

  // clamped lengths, chunk counts and their prefix sums (cache_len is an input of the step)
  if (warp == 0) {
    int run = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int bb = b0 + lane;
      int Lb = bb < p.B ? p.cache_len[bb] : 0;
      Lb = Lb < 0 ? 0 : (Lb > lmax ? lmax : Lb);
      Lb -= dec_first_slot(Lb, p.window);          // visible cached keys
      const int n = bb < p.B ? (Lb + 1 + kChunk - 1) / kChunk : 0;
      int v = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (bb < p.B) {
        lens[bb] = Lb;
        prefix[bb + 1] = run + v;
      }
      run += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) prefix[0] = 0;
  }
  if (threadIdx.x == 32) {
    for (int s2 = 0; s2 < NS; ++s2) {
      mbar_init(&full[s2], 1);
      mbar_init(&empty[s2], NW);
    }
    for (int s2 = 0; s2 < 2; ++s2) {
      mbar_init(&mfull[s2], NW * 32);
      mbar_init(&mempty[s2], 32);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int total = p.KV * prefix[p.B];
  const int per = (total + gridDim.x - 1) / gridDim.x;
  const int i0 = blockIdx.x * per, i1 = min(total, i0 + per);
  if (i0 >= i1) return;                            // uniform: nothing for this CTA
  // item -> (sequence, kv head, chunk, chunks of the sequence): a search for
  // the first item, then one step per item
  auto seek = [&](int i, int &b, int &kvh, int &ch, int &nsp) {
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.KV * prefix[mid] <= i) lo = mid;
      else hi = mid - 1;
    }
    b = lo;
    nsp = prefix[b + 1] - prefix[b];
    const int r = i - p.KV * prefix[b];
    kvh = r / nsp;
    ch = r - kvh * nsp;
  };
  auto step = [&](int &b, int &kvh, int &ch, int &nsp) {
    if (++ch < nsp) return;
    ch = 0;
    if (++kvh < p.KV) return;
    kvh = 0;
    ++b;
    nsp = b < p.B ? prefix[b + 1] - prefix[b] : 0;
  };

  if (warp == NW) {
    // ------------------------------------------------ producer (the cache is
    // an input of the step: requested before waiting on the preceding kernel)
    if (lane == 0) {
      griddep_launch_dependents();
      int stage = 0, phase = 0;
      long long issued = 0;
      bool ok = true;
      int b, kvh, ch, nsp;
      seek(i0, b, kvh, ch, nsp);
      for (int i = i0; i < i1; ++i, step(b, kvh, ch, nsp)) {
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        int first = 0;                              // first slot inside the window
        if (p.window > 0) {
          int Lf = p.cache_len[b];
          Lf = Lf < 0 ? 0 : (Lf > lmax ? lmax : Lf);
          first = Lf - lens[b];
        }
        const int y = static_cast<int>(((long long)p.layer * p.B + b) * p.KV + kvh) * p.S_max + first +
                      ch * kChunk;
        mbar_arrive_expect_tx(&full[stage], STAGE);
        tma_load_2d(dsm + stage * STAGE, &tmK, &full[stage], 0, y);
        tma_load_2d(dsm + stage * STAGE + kChunk * 128, &tmV, &full[stage], 0, y);
        ++issued;
        if (++stage == NS) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        atomicCAS(p.status, 0, kDevTimeoutProducer);
        *abort_flag = 1;
      }
      // every copy issued has landed before the CTA may exit
      int dummy = 0;
      const long long first = issued > NS ? issued - NS : 0;
      for (long long j = first; j < issued; ++j)
        if (!mbar_wait_bounded(&full[j % NS], (uint32_t)((j / NS) & 1), reinterpret_cast<volatile int *>(&dummy)))
          atomicCAS(p.status, 0, kDevTimeoutDrain);
    }
    return;
  }

  if (warp > NW) {
    // ------------------------------------------------ merge warps: warp NW + 1 + m
    // takes the runs with index % 2 == m through merge buffer m
    const int mwarp = warp - (NW + 1);
    griddep_wait();                                // o, partials and counters
    int b, kvh, ch, nsp;
    seek(i0, b, kvh, ch, nsp);
    int run = 0, mph = 0;
    for (int i = i0; i < i1; ++i, step(b, kvh, ch, nsp)) {
      if (i + 1 < i1 && ch + 1 < nsp) continue;    // the CTA's run of this pair goes on
      if ((run++ & 1) != mwarp) continue;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&mfull[mwarp], mph, abort_flag))) {
        if (lane == 0) atomicCAS(p.status, 0, kDevTimeoutEpilogue);
        *abort_flag = 1;
        break;
      }
      mph ^= 1;
      const float *rm = red + mwarp * RED, *rl = rm + NW * GM, *ro = rl + NW * GM;
      float Ms[GM], Ls[GM], O0[GM], O1[GM];
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        Ms[g] = -INFINITY;
        Ls[g] = O0[g] = O1[g] = 0.f;
        if (g < G) {
#pragma unroll
          for (int w = 0; w < NW; ++w) Ms[g] = fmaxf(Ms[g], rm[w * GM + g]);
          const float Mu = (Ms[g] == -INFINITY) ? 0.f : Ms[g];
#pragma unroll
          for (int w = 0; w < NW; ++w) {
            const float fw = exp2f(rm[w * GM + g] - Mu);
            Ls[g] += rl[w * GM + g] * fw;
            O0[g] += ro[(w * GM + g) * HD + lane] * fw;
            O1[g] += ro[(w * GM + g) * HD + lane + 32] * fw;
          }
        }
      }
      mbar_arrive(&mempty[mwarp]);                 // the buffer goes back to the compute warps
      const int pair = b * p.KV + kvh;
      const int pair_first = p.KV * prefix[b] + kvh * nsp;   // the pair's first item
      const int c_first = pair_first / per;
      const int nseg = (pair_first + nsp - 1) / per - c_first + 1;
      const int seg = blockIdx.x - c_first;
      const long long pbase = (long long)b * p.H + kvh * G;   // first query head of the group
      if (nseg > 1) {
#pragma unroll
        for (int g = 0; g < GM; ++g)
          if (g < G) {
            const long long ps = (pbase + g) * p.max_splits + seg;
            if (lane == 0) {
              p.part_m[ps] = Ms[g];
              p.part_l[ps] = Ls[g];
            }
            p.part_o[ps * HD + lane] = O0[g];
            p.part_o[ps * HD + lane + 32] = O1[g];
          }
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          __threadfence();                         // the warp's partials before the arrival
          const int prev = atomicAdd(p.counters + pair, 1);
          last = (prev == nseg - 1);
          if (last) {
            p.counters[pair] = 0;                  // ready for the next layer
            __threadfence();
          }
        }
        if (!__shfl_sync(0xffffffffu, last, 0)) continue;
        // the last segment to finish merges the others into its own state
        // (still in registers), U segments' loads in flight at a time
        constexpr int U = GM <= 4 ? 4 : 2;
        for (int s0 = 0; s0 < nseg; s0 += U) {
          float vm[U][GM], vl[U][GM], v0[U][GM], v1[U][GM];
#pragma unroll
          for (int u = 0; u < U; ++u)
#pragma unroll
            for (int g = 0; g < GM; ++g) {
              const int s2 = s0 + u;
              const bool ok = g < G && s2 < nseg && s2 != seg;
              const long long ps = (pbase + g) * p.max_splits + s2;
              vm[u][g] = ok ? __ldcg(p.part_m + ps) : -INFINITY;
              vl[u][g] = ok ? __ldcg(p.part_l + ps) : 0.f;
              v0[u][g] = ok ? __ldcg(p.part_o + ps * HD + lane) : 0.f;
              v1[u][g] = ok ? __ldcg(p.part_o + ps * HD + lane + 32) : 0.f;
            }
#pragma unroll
          for (int u = 0; u < U; ++u)
#pragma unroll
            for (int g = 0; g < GM; ++g) {
              const float mn = fmaxf(Ms[g], vm[u][g]);
              const float mu = (mn == -INFINITY) ? 0.f : mn;
              const float fa = exp2f(Ms[g] - mu), fb = exp2f(vm[u][g] - mu);
              Ls[g] = Ls[g] * fa + vl[u][g] * fb;
              O0[g] = O0[g] * fa + v0[u][g] * fb;
              O1[g] = O1[g] * fa + v1[u][g] * fb;
              Ms[g] = mn;
            }
        }
      }
#pragma unroll
      for (int g = 0; g < GM; ++g)
        if (g < G) {
          const float inv = Ls[g] > 0.f ? 1.f / Ls[g] : 0.f;
          p.o[(pbase + g) * HD + lane] = __float2half_rn(O0[g] * inv);
          p.o[(pbase + g) * HD + lane + 32] = __float2half_rn(O1[g] * inv);
        }
    }
    return;
  }

  // -------------------------------------------------- compute warps 0..NW-1
  griddep_wait();                                  // q, k_new, v_new
  const int r = lane >> 2, c2 = (lane & 3) * 2;    // fragment row (head) and column pair
  const int kw0 = warp * KPW;                      // this warp's keys within a chunk
  int b, kvh, ch, nsp;
  seek(i0, b, kvh, ch, nsp);
  // raw q words of head r of a pair (dims kk*16 + c2 + {0,1} and + 8 + {0,1})
  uint32_t qraw[8];
  auto load_q = [&](int qb, int qkvh) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if (r < G && qb < p.B) {
        const f16 *qr = p.q + ((long long)qb * p.H + qkvh * G + r) * HD + kk * 16 + c2;
        qraw[2 * kk] = *reinterpret_cast<const uint32_t *>(qr);
        qraw[2 * kk + 1] = *reinterpret_cast<const uint32_t *>(qr + 8);
      } else {
        qraw[2 * kk] = qraw[2 * kk + 1] = 0u;
      }
    }
  };
  load_q(b, kvh);
  int stage = 0, phase = 0, mb = 0, mph = 0;
  int cur_pair = -1;
  uint32_t qa[4][4];
  float mw = -INFINITY, lw = 0.f;                  // running max / sum of head r (this warp)
  float o[8][4];
  for (int i = i0; i < i1; ++i, step(b, kvh, ch, nsp)) {
    const int pair = b * p.KV + kvh;
    if (pair != cur_pair) {
      cur_pair = pair;
      mw = -INFINITY;
      lw = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) o[q][0] = o[q][1] = o[q][2] = o[q][3] = 0.f;
      // q as A fragments (rows r < G: bf16 hi part; rows r + 8: the lo remainder)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float2 a2 = unpack_f16x2(qraw[2 * kk]);
        const float2 b2 = unpack_f16x2(qraw[2 * kk + 1]);
        float h0, l0, h1, l1, h2, l2, h3, l3;
        split_bf16(a2.x, h0, l0);
        split_bf16(a2.y, h1, l1);
        split_bf16(b2.x, h2, l2);
        split_bf16(b2.y, h3, l3);
        qa[kk][0] = pack_bf16x2(h0, h1);
        qa[kk][1] = pack_bf16x2(l0, l1);
        qa[kk][2] = pack_bf16x2(h2, h3);
        qa[kk][3] = pack_bf16x2(l2, l3);
      }
      // the next pair's q is read while this one's chunks stream
      load_q(kvh + 1 < p.KV ? b : b + 1, kvh + 1 < p.KV ? kvh + 1 : 0);
    }
    const int Lb = lens[b];
    const int k_begin = ch * kChunk;
    const int n_valid = min(kChunk, Lb + 1 - k_begin);
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[stage], phase, abort_flag))) {
      if (lane == 0) atomicCAS(p.status, 0, kDevTimeoutEpilogue);
      *abort_flag = 1;
      break;
    }
    uint8_t *sK = dsm + stage * STAGE, *sV = sK + kChunk * 128;
    // this warp's keys: the new token's key/value into its slot, V rows past
    // the valid keys zeroed (unused cache slots must not inject NaN)
    const int slot = Lb - k_begin;
    if (slot >= kw0 && slot < kw0 + KPW && lane < 8) {
      const long long row = (long long)b * p.KV + kvh;
      *reinterpret_cast<uint4 *>(sK + slot * 128 + ((lane ^ (slot & 7)) << 4)) =
          reinterpret_cast<const uint4 *>(p.k_new + row * HD)[lane];
      *reinterpret_cast<uint4 *>(sV + slot * 128 + ((lane ^ (slot & 7)) << 4)) =
          reinterpret_cast<const uint4 *>(p.v_new + row * HD)[lane];
    }
    for (int e = max(n_valid, kw0) * 8 + lane; e < (kw0 + KPW) * 8; e += 32)
      reinterpret_cast<uint4 *>(sV)[e] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    if (kw0 < n_valid) {                           // warp-uniform
      float s[2 * N16][4];
#pragma unroll
      for (int q = 0; q < 2 * N16; ++q) s[q][0] = s[q][1] = s[q][2] = s[q][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int j = 0; j < N16; ++j) {
          const int key = kw0 + j * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int chunk = kk * 2 + ((lane >> 3) & 1);
          uint32_t bk[4];
          ldsm_x4(bk, sK + key * 128 + ((chunk ^ (key & 7)) << 4));
          mma_bf16_16816(s[2 * j], qa[kk], bk[0], bk[1]);
          mma_bf16_16816(s[2 * j + 1], qa[kk], bk[2], bk[3]);
        }
      }
      // head r's score = hi row + lo row, in the exp2 domain; keys past the valid range masked
      float sc[2 * N16][2];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2 * N16; ++j) {
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
      const float m_new = fmaxf(mw, mx);
      const float mu = (m_new == -INFINITY) ? 0.f : m_new;
      const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - mu);    // rescale of the running state
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < 2 * N16; ++j) {
        sc[j][0] = exp2f(sc[j][0] - mu);
        sc[j][1] = exp2f(sc[j][1] - mu);
        sum += sc[j][0] + sc[j][1];
      }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      lw = lw * f + sum;
      mw = m_new;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        o[q][0] *= f; o[q][1] *= f; o[q][2] *= f; o[q][3] *= f;
      }
#pragma unroll
      for (int kk = 0; kk < N16; ++kk) {
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
    // the stage goes back to the producer (generic writes above precede the next TMA fill)
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == NS) {
      stage = 0;
      phase ^= 1;
    }
    if (i + 1 < i1 && ch + 1 < nsp) continue;      // this CTA's run of chunks of the pair goes on
    // ---- end of the run: this warp's state goes to the merge warp
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&mempty[mb], mph ^ 1, abort_flag))) {
      if (lane == 0) atomicCAS(p.status, 0, kDevTimeoutEpilogue);
      *abort_flag = 1;
      break;
    }
    float *rm = red + mb * RED, *rl = rm + NW * GM, *ro = rl + NW * GM;
    if (r < G) {
      if ((lane & 3) == 0) {
        rm[warp * GM + r] = mw;
        rl[warp * GM + r] = lw;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        ro[(warp * GM + r) * HD + 8 * q + c2] = o[q][0] + o[q][2];
        ro[(warp * GM + r) * HD + 8 * q + c2 + 1] = o[q][1] + o[q][3];
      }
    }
    mbar_arrive(&mfull[mb]);
    if (++mb == 2) {
      mb = 0;
      mph ^= 1;
    }
  }
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
  const int first = dec_first_slot(Lb, p.window);   // keys below are outside the window
  Lb -= first;                                      // from here on: visible cached keys
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
  const bf16 *kc = p.k_cache + (row * p.S_max + first) * HD;
  const bf16 *vc = p.v_cache + (row * p.S_max + first) * HD;
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

template <int GM>
static cudaError_t launch_decode_attn_persist_g(const CUtensorMap &tk, const CUtensorMap &tv,
                                                const DecAttnParams &ap, int sms, cudaStream_t st) {
  const int smem = persist_smem_fixed<GM>() + (2 * ap.B + 1) * 4;
  constexpr auto kern = decode_attn_persist_kernel<GM>;
  cudaError_t e = ensure_smem_attr<kern>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(sms), dim3((kPersistWarps + 3) * 32), smem, st, tk, tv, ap);
}

// head_dim 64 runs on tensor cores (the cache seen as one 2-D tensor of
// L*B*KV*S_max rows of 64 values); other head sizes on the CUDA-core kernel.
static cudaError_t launch_decode_attn(const DecAttnParams &ap, int hd, dim3 grid, cudaStream_t st,
                                      const bf16 *k_all, const bf16 *v_all, int L, int sms) {
  if (hd == 64) {
    CUtensorMap tk, tv;
    const uint64_t rows = (uint64_t)L * ap.B * ap.KV * ap.S_max;
    if (!get_tmap_f16(&tk, k_all, rows, 64, 64, kChunk)) return cudaErrorInvalidValue;
    if (!get_tmap_f16(&tv, v_all, rows, 64, 64, kChunk)) return cudaErrorInvalidValue;
    const int G = ap.H / ap.KV;
    if (ap.B <= kDecMaxB) {
      if (G == 1) return launch_decode_attn_persist_g<1>(tk, tv, ap, sms, st);
      if (G == 2) return launch_decode_attn_persist_g<2>(tk, tv, ap, sms, st);
      if (G == 3) return launch_decode_attn_persist_g<3>(tk, tv, ap, sms, st);
      if (G == 4) return launch_decode_attn_persist_g<4>(tk, tv, ap, sms, st);
      return launch_decode_attn_persist_g<8>(tk, tv, ap, sms, st);
    }
    if (G == 1) return launch_decode_attn_mma_g<1>(tk, tv, ap, grid, st);
    if (G == 2) return launch_decode_attn_mma_g<2>(tk, tv, ap, grid, st);
    if (G == 3) return launch_decode_attn_mma_g<3>(tk, tv, ap, grid, st);
    if (G == 4) return launch_decode_attn_mma_g<4>(tk, tv, ap, grid, st);
    return launch_decode_attn_mma_g<8>(tk, tv, ap, grid, st);
  }
  return launch_decode_attn_hd<128>(ap, grid, st);
}

// next[b] = the column of row b's packed maximum (argmax_pack).
__global__ void argmax_finish_kernel(const unsigned long long *argmax, int B, int *next) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) next[b] = argmax_index(argmax[b]);
}

__global__ void zero_ints_kernel(int *p, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = 0;
}

static cudaError_t launch_zero_ints(int *p, int n, cudaStream_t st) {
  zero_ints_kernel<<<(unsigned)cdiv(n, 256), 256, 0, st>>>(p, n);
  return cudaGetLastError();
}

// The narrow-unit kernel for batches of at most 64 rows, the tile GEMM otherwise.
static cudaError_t dec_gemm(int epi, int bn, const void *A, const void *W, const GemmParams &p, int sms,
                            cudaStream_t st) {
  if (skinny_gemm_supported(epi, p)) return launch_skinny_gemm(epi, A, W, p, st);
  return launch_gemm(epi, bn, A, W, p, sms, st);
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

  unsigned long long *argmax = reinterpret_cast<unsigned long long *>(wb + W.argmax);
  DEC_LAUNCH(launch_zero_ints(counters, static_cast<int>((W.argmax + (size_t)B * 8 - W.counters) / 4), st));
  DEC_LAUNCH_K(SMOL_K_EMBED, launch_embed_rows(a.ids, a.embed, V, d, B, x, nullptr, ssq_a, status,
                                                SeqCheck{a.cache_len, 1, min(a.S_max, c.max_pos - 1)}, st));

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
    p.rope = layer_rotary(&c, l) ? a.rope : nullptr; p.valid_start = nullptr; p.pos_add = a.cache_len; p.pos_limit = min(a.S_max, c.max_pos - 1);
    p.max_pos = c.max_pos; p.status = status; p.pdl = 1;
    DEC_LAUNCH_K(SMOL_K_QKV, dec_gemm(kEpiQkvRope, hd, x, lb + a.off_qkv, p, sms, st));

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
    ap.window = layer_window(&c, l);
    const int lmax = min(a.S_max, c.max_pos - 1);
    dim3 grid((unsigned)cdiv(lmax + 1, kChunk), (unsigned)KV, (unsigned)B);
    ap.layer = l;
    DEC_LAUNCH_K(SMOL_K_DEC_ATTN, launch_decode_attn(ap, hd, grid, st, a.k_cache, a.v_cache, L, sms));

    GemmParams po{};
    po.M = B; po.N = d; po.K = H * hd; po.out = h; po.out_is_f16 = 1; po.ldo = d; po.resid_f16 = x;
    po.ssq_out = ssq_b;
    po.status = status; po.pdl = 1;
    DEC_LAUNCH_K(SMOL_K_OPROJ, dec_gemm(kEpiResidual, 64, o, lb + a.off_o, po, sms, st));

    GemmParams pg{};
    pg.M = B; pg.N = 2 * I; pg.K = d; pg.out = act; pg.out_is_f16 = 1; pg.ldo = I; pg.ssq_in = ssq_b;
    pg.inv_dim = 1.0f / d; pg.eps = c.rms_eps; pg.ssq_zero = ssq_a; pg.status = status; pg.pdl = 1;
    DEC_LAUNCH_K(SMOL_K_GATEUP, dec_gemm(kEpiSwiglu, 128, h, lb + a.off_gu, pg, sms, st));

    GemmParams pd{};
    pd.M = B; pd.N = d; pd.K = I; pd.out = x; pd.out_is_f16 = 1; pd.ldo = d; pd.resid_f16 = h;
    pd.ssq_out = ssq_a;
    pd.status = status; pd.pdl = 1;
    DEC_LAUNCH_K(SMOL_K_DOWN, dec_gemm(kEpiResidual, 64, act, lb + a.off_down, pd, sms, st));
  }
  GemmParams ph{};
  ph.M = B; ph.N = V; ph.K = d; ph.out = a.logits; ph.out_is_f16 = 0; ph.ldo = V; ph.ssq_in = ssq_a;
  ph.inv_dim = 1.0f / d; ph.eps = c.rms_eps; ph.status = status; ph.pdl = 1;
  ph.argmax = a.next ? argmax : nullptr;         // the greedy choice, in the head's epilogue
  DEC_LAUNCH_K(SMOL_K_HEAD, launch_gemm(kEpiScale, gemm_pick_bn(kEpiScale, V, hd), x, a.head, ph, sms, st));
  if (a.next) {
    argmax_finish_kernel<<<(unsigned)cdiv(B, 128), 128, 0, st>>>(argmax, B, a.next);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ++n;
  }
#undef DEC_LAUNCH
  *launches = n;
  return cudaSuccess;
}

}  // namespace smol
