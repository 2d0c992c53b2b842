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
// Keys are spread over lane groups of hd/8 lanes (16-byte loads, 8 dims per
// lane); each lane group takes 4 keys per step (8 loads in flight per lane),
// reduces the q.k partial dots with shuffles and updates an online softmax in
// the exp2 domain.  Partial (max, sum, output) triples are merged inside the
// warp, then across warps in shared memory, then across chunks by the last
// CTA of the (b, kv head) pair (an atomic arrival counter, no waiting).
#include <math.h>

#include "decode.cuh"
#include "profile.cuh"
#include "prims.cuh"

namespace smol {

constexpr int kChunk = 512;        // keys per CTA
constexpr int kDecWarps = 8;       // warps per CTA

struct DecWs {
  size_t status, x, x32, h, h32, q, o, a, ssq_a, ssq_b, part_m, part_l, part_o, counters, total;
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
  W.x32 = o; o = align_up(o + B * d * 4, 1024);
  W.h = o; o = align_up(o + B * d * 2, 1024);
  W.h32 = o; o = align_up(o + B * d * 4, 1024);
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
};

__device__ __forceinline__ uint4 ld_stream(const bf16 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// GM: compile-time bound on the group size g = H / KV (arrays are sized GM).
template <int HD, int GM>
__global__ void __launch_bounds__(kDecWarps * 32, 2) decode_attn_kernel(const DecAttnParams p) {
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
      const bf16 *kp = (j < Lb) ? kc + (long long)j * HD : kn;
      const bf16 *vp = (j < Lb) ? vc + (long long)j * HD : vn;
      if (valid[i]) {
        kr[i] = ld_stream(kp + sub * 8);
        vr[i] = ld_stream(vp + sub * 8);
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

  __shared__ float red_m[kDecWarps][GM], red_l[kDecWarps][GM];
  __shared__ float red_o[kDecWarps][GM][HD];
  __shared__ int s_last;
  if (grp == 0) {
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      if (g < G) {
        if (sub == 0) {
          red_m[warp][g] = m[g];
          red_l[warp][g] = l[g];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) red_o[warp][g][sub * 8 + e] = acc[g][e];
      }
    }
  }
  __syncthreads();
  const long long pbase = (long long)b * p.H + kvh * G;   // first head of the group
  for (int t = threadIdx.x; t < G * HD; t += blockDim.x) {
    const int g = t / HD, dim = t - g * HD;
    float M = -INFINITY;
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, red_m[w][g]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float Ls = 0.f, Os = 0.f;
    for (int w = 0; w < kDecWarps; ++w) {
      const float f = exp2f(red_m[w][g] - Mu);
      Ls += red_l[w][g] * f;
      Os += red_o[w][g][dim] * f;
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
    s_last = (prev == nsplit - 1);
  }
  __syncthreads();
  if (!s_last) return;
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

template <int HD>
static cudaError_t launch_decode_attn_hd(const DecAttnParams &ap, dim3 grid, cudaStream_t st) {
  const int G = ap.H / ap.KV;
  if (G == 1) decode_attn_kernel<HD, 1><<<grid, kDecWarps * 32, 0, st>>>(ap);
  else if (G == 2) decode_attn_kernel<HD, 2><<<grid, kDecWarps * 32, 0, st>>>(ap);
  else if (G == 3) decode_attn_kernel<HD, 3><<<grid, kDecWarps * 32, 0, st>>>(ap);
  else if (G == 4) decode_attn_kernel<HD, 4><<<grid, kDecWarps * 32, 0, st>>>(ap);
  else decode_attn_kernel<HD, 8><<<grid, kDecWarps * 32, 0, st>>>(ap);
  return cudaGetLastError();
}

static cudaError_t launch_decode_attn(const DecAttnParams &ap, int hd, dim3 grid, cudaStream_t st) {
  return hd == 64 ? launch_decode_attn_hd<64>(ap, grid, st) : launch_decode_attn_hd<128>(ap, grid, st);
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
  float *x32 = reinterpret_cast<float *>(wb + W.x32);
  float *h32 = reinterpret_cast<float *>(wb + W.h32);
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
  DEC_LAUNCH_K(SMOL_K_EMBED, launch_embed_rows(a.ids, a.embed, V, d, B, x, x32, ssq_a, st));

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
    p.max_pos = c.max_pos; p.status = status;
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
    ap.max_splits = W.max_splits; ap.scale_log2 = sl2;
    const int lmax = min(a.S_max, c.max_pos - 1);
    dim3 grid((unsigned)cdiv(lmax + 1, kChunk), (unsigned)KV, (unsigned)B);
    DEC_LAUNCH_K(SMOL_K_DEC_ATTN, launch_decode_attn(ap, hd, grid, st));

    GemmParams po{};
    po.M = B; po.N = d; po.K = H * hd; po.out = h; po.out_is_f16 = 1; po.out_f32 = h32; po.ldo = d; po.resid_f32 = x32;
    po.ssq_out = ssq_b;
    po.status = status;
    DEC_LAUNCH_K(SMOL_K_OPROJ, launch_gemm(kEpiResidual, 64, o, lb + a.off_o, po, sms, st));

    GemmParams pg{};
    pg.M = B; pg.N = 2 * I; pg.K = d; pg.out = act; pg.out_is_f16 = 1; pg.ldo = I; pg.ssq_in = ssq_b;
    pg.inv_dim = 1.0f / d; pg.eps = c.rms_eps; pg.ssq_zero = ssq_a; pg.status = status;
    DEC_LAUNCH_K(SMOL_K_GATEUP, launch_gemm(kEpiSwiglu, 128, h, lb + a.off_gu, pg, sms, st));

    GemmParams pd{};
    pd.M = B; pd.N = d; pd.K = I; pd.out = x; pd.out_is_f16 = 1; pd.out_f32 = x32; pd.ldo = d; pd.resid_f32 = h32;
    pd.ssq_out = ssq_a;
    pd.status = status;
    DEC_LAUNCH_K(SMOL_K_DOWN, launch_gemm(kEpiResidual, 64, act, lb + a.off_down, pd, sms, st));
  }
  GemmParams ph{};
  ph.M = B; ph.N = V; ph.K = d; ph.out = a.logits; ph.out_is_f16 = 0; ph.ldo = V; ph.ssq_in = ssq_a;
  ph.inv_dim = 1.0f / d; ph.eps = c.rms_eps; ph.status = status;
  DEC_LAUNCH_K(SMOL_K_HEAD, launch_gemm(kEpiScale, gemm_pick_bn(kEpiScale, V, hd), x, a.head, ph, sms, st));
#undef DEC_LAUNCH
  *launches = n;
  return cudaSuccess;
}

}  // namespace smol
