// attention.cu - causal grouped-query flash attention for prefill (sm_103a).
//
// o[b,t,h,:] = sum_{j visible} softmax_j(q[b,h,t].k[b,h/g,j] / sqrt(hd)) v[b,h/g,j]
// with j visible iff valid_start[b] <= j <= t ("model.py" (SmolLM2-135M)
// section 4: scores / sqrt(head_dim), triu(1) causal mask plus the additive
// padding mask, softmax, probs @ v; GQA through repeat_interleave, i.e. query
// head h reads key/value head h // g, as in the "SmolLM3" page's
// "Grouped-query attention").  Rows with no visible key produce 0.  With a
// sliding window w (the "SmolLM3" page, "A sliding window the 3B checkpoints
// leave off") keys j <= t - w are hidden too, and so are the keys an optional
// key mask (the additive attention_mask of section 4, as bytes) marks 0.
//
// One CTA owns (sequence b, kv head, a block of BQ query tokens) and all g
// query heads of that kv head: each K/V tile is loaded once into shared memory
// and used by the g*BQ/16 warps of the group, so K/V are never expanded per
// query head.  Online softmax (running max and sum, exp2 domain) keeps S and P
// in registers; S = Q K^T and O += P V run on mma.sync m16n8k16 (f16 -> fp32).
// K/V tiles are double-buffered with cp.async; shared tiles are XOR-swizzled
// in 16-byte chunks so ldmatrix reads are conflict-free.
#include <math.h>

#include "common.cuh"
#include "prims.cuh"

namespace smol {

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// element offset of (row, col) in a [rows][HD] tile with 16-byte chunk swizzle
template <int HD>
__device__ __forceinline__ int swz(int row, int col) {
  return row * HD + ((((col >> 3) ^ (row & 7))) << 3) + (col & 7);
}

template <int HD, int BQ, int BK>
__global__ void __launch_bounds__(512, 1) flash_attn_kernel(const AttnParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int G = p.H / p.KV;
  f16 *sQ = reinterpret_cast<f16 *>(smem_raw);                   // [G*BQ][HD]
  f16 *sK = sQ + G * BQ * HD;                                     // [2][BK][HD]
  f16 *sV = sK + 2 * BK * HD;                                     // [2][BK][HD]

  // query block = slow launch index, descending: longest causal blocks first
  const int nqb = gridDim.y;
  const int qb = nqb - 1 - blockIdx.y;
  const int kvh = blockIdx.x % p.KV, b = blockIdx.x / p.KV;
  const int q0 = qb * BQ;
  const int T = p.T;
  const int vs = p.valid_start ? min(max(p.valid_start[b], 0), T) : 0;
  const int nthreads = blockDim.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- load Q rows (head hl, token q0+tl) -> sQ row hl*BQ + tl
  constexpr int CH = HD / 8;                                      // 16-byte chunks per row
  for (int idx = tid; idx < G * BQ * CH; idx += nthreads) {
    const int r = idx / CH, c = idx - r * CH;
    const int hl = r / BQ, tl = r - hl * BQ;
    const int t = q0 + tl;
    const bool ok = t < T;
    const f16 *src = p.q + ((((long long)b * p.H + kvh * G + hl) * T) + (ok ? t : 0)) * HD + c * 8;
    cp_async16(sQ + swz<HD>(r, c * 8), src, ok);
  }
  const f16 *kbase = p.k + ((long long)b * p.KV + kvh) * T * HD;
  const f16 *vbase = p.v + ((long long)b * p.KV + kvh) * T * HD;
  auto load_kv = [&](int kt, int st) {
    f16 *dk = sK + st * BK * HD, *dv = sV + st * BK * HD;
    for (int idx = tid; idx < BK * CH; idx += nthreads) {
      const int r = idx / CH, c = idx - r * CH;
      const int j = kt * BK + r;
      const bool ok = j < T;
      const long long off = (long long)(ok ? j : 0) * HD + c * 8;
      cp_async16(dk + swz<HD>(r, c * 8), kbase + off, ok);
      cp_async16(dv + swz<HD>(r, c * 8), vbase + off, ok);
    }
  };

  const int last_q = min(q0 + BQ, T) - 1;
  const int W = p.window;                                         // > 0: sliding window
  const uint8_t *kmask = p.key_mask ? p.key_mask + (long long)b * T : nullptr;   // 0 = key hidden
  const int kt_lo = (W > 0 ? max(vs, q0 - W + 1) : vs) / BK;      // first key any row of the block sees
  const int kt_hi = last_q / BK;
  load_kv(kt_lo, 0);
  cp_async_commit();

  const int slabs = BQ / 16;
  const int hl = warp / slabs, slab = warp - hl * slabs;
  const int h = kvh * G + hl;
  const int row0 = hl * BQ + slab * 16;                           // first sQ row of this warp
  const int t_a = q0 + slab * 16 + (lane >> 2), t_b = t_a + 8;
  const int tw_lo = q0 + slab * 16, tw_hi = tw_lo + 15;

  constexpr int NT = BK / 8;                                      // S n-tiles
  constexpr int OT = HD / 8;                                      // O n-tiles
  float o[OT][4];
#pragma unroll
  for (int i = 0; i < OT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  const float sl2 = p.scale_log2;

  for (int kt = kt_lo, it = 0; kt <= kt_hi; ++kt, ++it) {
    const int st = it & 1;
    if (kt + 1 <= kt_hi) {
      load_kv(kt + 1, st ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    const int k0 = kt * BK;
    // skip tiles whose keys are all in this warp's future or all before its
    // rows' windows, and warps made only of padding rows
    if (k0 <= tw_hi && tw_hi >= vs && (W == 0 || k0 + BK - 1 > tw_lo - W)) {
      const f16 *tK = sK + st * BK * HD;
      const f16 *tV = sV + st * BK * HD;
      float s[NT][4];
#pragma unroll
      for (int i = 0; i < NT; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        uint32_t a[4];
        ldsm_x4(a, sQ + swz<HD>(row0 + (lane & 15), kk * 16 + ((lane >> 4) << 3)));
#pragma unroll
        for (int j = 0; j < BK / 16; ++j) {
          uint32_t bk[4];
          ldsm_x4(bk, tK + swz<HD>(j * 16 + (lane & 7) + ((lane >> 4) << 3),
                                   kk * 16 + (((lane >> 3) & 1) << 3)));
          mma_f16_16816(s[2 * j], a, bk[0], bk[1]);
          mma_f16_16816(s[2 * j + 1], a, bk[2], bk[3]);
        }
      }
      // scale into the exp2 domain and mask
      const bool need_mask = (k0 + BK - 1 > tw_lo) || (k0 < vs) || (W > 0 && k0 <= tw_hi - W) || kmask != nullptr;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x = s[i][e] * sl2;
          if (need_mask) {
            const int j = k0 + i * 8 + ((lane & 3) << 1) + (e & 1);
            const int t = (e < 2) ? t_a : t_b;
            if (j > t || j < vs || (W > 0 && j <= t - W) || (kmask && (j >= T || !kmask[j]))) x = -INFINITY;
          }
          s[i][e] = x;
        }
      }
      float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        mx_a = fmaxf(mx_a, fmaxf(s[i][0], s[i][1]));
        mx_b = fmaxf(mx_b, fmaxf(s[i][2], s[i][3]));
      }
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      const float mu_a = (mn_a == -INFINITY) ? 0.f : mn_a;
      const float mu_b = (mn_b == -INFINITY) ? 0.f : mn_b;
      const float al_a = exp2f(m_a - mu_a), al_b = exp2f(m_b - mu_b);
      m_a = mn_a;
      m_b = mn_b;
      float rs_a = 0.f, rs_b = 0.f;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        s[i][0] = exp2f(s[i][0] - mu_a);
        s[i][1] = exp2f(s[i][1] - mu_a);
        s[i][2] = exp2f(s[i][2] - mu_b);
        s[i][3] = exp2f(s[i][3] - mu_b);
        rs_a += s[i][0] + s[i][1];
        rs_b += s[i][2] + s[i][3];
      }
      l_a = l_a * al_a + rs_a;
      l_b = l_b * al_b + rs_b;
#pragma unroll
      for (int i = 0; i < OT; ++i) {
        o[i][0] *= al_a;
        o[i][1] *= al_a;
        o[i][2] *= al_b;
        o[i][3] *= al_b;
      }
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        uint32_t a[4];
        a[0] = pack_f16x2(s[2 * kk][0], s[2 * kk][1]);
        a[1] = pack_f16x2(s[2 * kk][2], s[2 * kk][3]);
        a[2] = pack_f16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        a[3] = pack_f16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int nd = 0; nd < HD / 16; ++nd) {
          uint32_t bv[4];
          ldsm_x4_t(bv, tV + swz<HD>(kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                     nd * 16 + ((lane >> 4) << 3)));
          mma_f16_16816(o[2 * nd], a, bv[0], bv[1]);
          mma_f16_16816(o[2 * nd + 1], a, bv[2], bv[3]);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();   // no copy may still be in flight when the CTA exits

  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f;
  const float inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
  const long long ldo = (long long)p.H * HD;
#pragma unroll
  for (int i = 0; i < OT; ++i) {
    const int col = h * HD + i * 8 + ((lane & 3) << 1);
    if (t_a < T)
      *reinterpret_cast<uint32_t *>(p.o + ((long long)b * T + t_a) * ldo + col) =
          pack_f16x2(o[i][0] * inv_a, o[i][1] * inv_a);
    if (t_b < T)
      *reinterpret_cast<uint32_t *>(p.o + ((long long)b * T + t_b) * ldo + col) =
          pack_f16x2(o[i][2] * inv_b, o[i][3] * inv_b);
  }
}

template <int HD, int BQ, int BK>
static cudaError_t launch_fa(const AttnParams &p, cudaStream_t stream) {
  const int G = p.H / p.KV;
  const int threads = G * (BQ / 16) * 32;
  if (threads > 512) return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)(G * BQ + 4 * BK) * HD * sizeof(f16);
  auto kern = flash_attn_kernel<HD, BQ, BK>;
  cudaError_t e = ensure_smem_attr<flash_attn_kernel<HD, BQ, BK>>((int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(p.B * p.KV), (unsigned)cdiv(p.T, BQ), 1u);
  kern<<<grid, threads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_flash_attention(const AttnParams &p, cudaStream_t stream) {
  const int G = p.H / p.KV;
  if (p.hd == 64) return G <= 4 ? launch_fa<64, 64, 64>(p, stream) : launch_fa<64, 32, 64>(p, stream);
  if (p.hd == 128) return launch_fa<128, 32, 32>(p, stream);
  return cudaErrorInvalidConfiguration;
}

}  // namespace smol
