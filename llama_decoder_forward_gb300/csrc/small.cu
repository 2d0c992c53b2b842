// small.cu - bandwidth-bound helper kernels: embedding gather with row
// sum-of-squares, row sum-of-squares, one-time weight packing, RoPE table.
#include <math.h>

#include "common.cuh"
#include "prims.cuh"

namespace smol {

__device__ __forceinline__ void seq_check(const SeqCheck &chk, long long r, int lane, int *status) {
  if (chk.vals && lane == 0 && r % chk.rows_per_seq == 0) {
    const int v = chk.vals[r / chk.rows_per_seq];
    if (v < 0 || v > chk.vmax) set_status(status, kDevBadInput);
  }
}

// x[r, :] = E[ids[r], :] as an f16 operand copy (x16) and in fp32 (x_f32,
// optional), and ssq[r] = sum_k x[r,k]^2 (feeds the first RMSNorm).
// "model.py" (SmolLM2-135M) section 7: embed_tokens(input_ids).  One warp per
// row, 16-byte loads.  d must be a multiple of 8.  An id outside [0, V) is
// clamped into range and recorded in the status word (kDevBadInput); a value
// beyond the f16 range is recorded too (kDevRange).
__global__ void embed_rows_kernel(const int *__restrict__ ids, const bf16 *__restrict__ E, int V,
                                  int d, long long rows, f16 *__restrict__ x16,
                                  float *__restrict__ x_f32, float *__restrict__ ssq, int *status,
                                  const SeqCheck chk) {
  const long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  seq_check(chk, r, lane, status);
  int id = ids[r];
  if (id < 0 || id >= V) {
    if (lane == 0) set_status(status, kDevBadInput);
    id = id < 0 ? 0 : V - 1;
  }
  bool in_range = true;
  const uint4 *src = reinterpret_cast<const uint4 *>(E + (long long)id * d);
  uint4 *dst = reinterpret_cast<uint4 *>(x16 + r * d);
  float acc = 0.f;
  for (int c = lane; c < d / 8; c += 32) {
    const uint4 v = src[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 t = unpack_bf16x2(w[e]);
      f[2 * e] = t.x;
      f[2 * e + 1] = t.y;
      acc += t.x * t.x + t.y * t.y;
      in_range &= fabsf(t.x) < kF16Overflow && fabsf(t.y) < kF16Overflow;
    }
    dst[c] = make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]),
                        pack_f16x2(f[6], f[7]));
    if (x_f32) {
      float4 *d4 = reinterpret_cast<float4 *>(x_f32 + r * d) + 2 * c;
      d4[0] = make_float4(f[0], f[1], f[2], f[3]);
      d4[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) ssq[r] = acc;
  if (!__all_sync(0xffffffffu, in_range) && lane == 0) set_status(status, kDevRange);
}

// ssq[r] = sum_k x[r,k]^2 for an fp32 row, plus its f16 copy (the tensor-core
// operand of the next projection); values beyond the f16 range (or not finite)
// are recorded in the status word (kDevRange).
__global__ void row_ssq_f32_kernel(const float *__restrict__ x, long long rows, int d,
                                   f16 *__restrict__ x16, float *__restrict__ ssq, int *status,
                                   const SeqCheck chk) {
  const long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  seq_check(chk, r, lane, status);
  const float4 *src = reinterpret_cast<const float4 *>(x + r * d);
  uint4 *dst = reinterpret_cast<uint4 *>(x16 + r * d);
  float acc = 0.f, amax = 0.f;
  for (int c = lane; c < d / 8; c += 32) {
    const float4 a = src[2 * c], b = src[2 * c + 1];
    acc += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z + b.w * b.w;
    amax = fmaxf(amax, fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                             fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w)))));
    dst[c] = make_uint4(pack_f16x2(a.x, a.y), pack_f16x2(a.z, a.w), pack_f16x2(b.x, b.y),
                        pack_f16x2(b.z, b.w));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) ssq[r] = acc;
  // fmaxf ignores NaN: a NaN row shows in the non-finite sum of squares
  if (!__all_sync(0xffffffffu, amax < kF16Overflow && isfinite(acc)) && lane == 0) set_status(status, kDevRange);
}

// The same for a bf16 row.
__global__ void row_ssq_kernel(const bf16 *__restrict__ x, long long rows, int d,
                               f16 *__restrict__ x16, float *__restrict__ ssq, int *status,
                               const SeqCheck chk) {
  const long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  seq_check(chk, r, lane, status);
  const uint4 *src = reinterpret_cast<const uint4 *>(x + r * d);
  uint4 *dst = reinterpret_cast<uint4 *>(x16 + r * d);
  float acc = 0.f;
  bool in_range = true;
  for (int c = lane; c < d / 8; c += 32) {
    const uint4 v = src[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = unpack_bf16x2(w[e]);
      acc += f.x * f.x + f.y * f.y;
      in_range &= fabsf(f.x) < kF16Overflow && fabsf(f.y) < kF16Overflow;
      o[e] = pack_f16x2(f.x, f.y);
    }
    dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) ssq[r] = acc;
  if (!__all_sync(0xffffffffu, in_range) && lane == 0) set_status(status, kDevRange);
}

// dst[r, c] = f16(src[r, c] * w[c]) (w == nullptr: plain conversion).  Folds
// an RMSNorm weight into the columns of the matrix that consumes its output.
__global__ void scale_cols_kernel(const bf16 *__restrict__ src, const bf16 *__restrict__ w,
                                  long long rows, int cols, f16 *__restrict__ dst) {
  const long long n = rows * cols;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = static_cast<int>(i % cols);
    float v = __bfloat162float(src[i]);
    if (w) v *= __bfloat162float(w[c]);
    dst[i] = __float2half_rn(v);
  }
}

// Packed gate/up matrix [2I, d]: rows 128j..128j+63 are gate rows 64j..64j+63,
// rows 128j+64..128j+127 are the matching up rows; both scaled by the MLP
// norm weight along d, stored as f16.
__global__ void interleave_gate_up_kernel(const bf16 *__restrict__ wg, const bf16 *__restrict__ wu,
                                          const bf16 *__restrict__ w, int I, int d,
                                          f16 *__restrict__ dst) {
  const long long n = 2LL * I * d;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / d;
    const int c = static_cast<int>(i - r * d);
    const long long grp = r / 128, within = r % 128;
    const bf16 *src = within < 64 ? wg : wu;
    const long long sr = grp * 64 + (within & 63);
    float v = __bfloat162float(src[sr * d + c]);
    if (w) v *= __bfloat162float(w[c]);
    dst[i] = __float2half_rn(v);
  }
}

// Two-level RoPE table ("model.py" (SmolLM2-135M) section 3 rope_freqs /
// build_rope_cache; "components.py" RotaryEmbedding), f_i = theta^(-2i/hd):
// fine entries hold (cos, sin)(b f_i) for b < 64, coarse entries
// (cos, sin)(64 a f_i); angles in double, stored as fp32, float4 entries of
// the pairs i = 2j, 2j + 1, laid out position-fastest (see rope_table_rows).
__global__ void rope_table_kernel(int max_pos, int hd, double theta, float4 *__restrict__ table) {
  const int quarter = hd / 4;
  const long long nc = cdiv(max_pos, 64);
  const long long n = (64 + nc) * quarter;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    long long j, pos;
    if (idx < 64LL * quarter) {
      j = idx / 64;
      pos = idx - j * 64;
    } else {
      const long long r = idx - 64LL * quarter;
      j = r / nc;
      pos = 64 * (r - j * nc);
    }
    const double a0 = static_cast<double>(pos) * pow(theta, -2.0 * (2 * j) / hd);
    const double a1 = static_cast<double>(pos) * pow(theta, -2.0 * (2 * j + 1) / hd);
    table[idx] = make_float4(static_cast<float>(cos(a0)), static_cast<float>(sin(a0)),
                             static_cast<float>(cos(a1)), static_cast<float>(sin(a1)));
  }
}

static int grid_for(long long n, int threads) {
  long long g = cdiv(n, threads);
  return static_cast<int>(g > 65535LL * 8 ? 65535LL * 8 : (g < 1 ? 1 : g));
}

cudaError_t launch_embed_rows(const int *ids, const bf16 *embed, int vocab, int d, long long rows,
                              f16 *x16, float *x_f32, float *ssq, int *status, SeqCheck chk,
                              cudaStream_t stream) {
  const int wpb = 8;
  embed_rows_kernel<<<(unsigned)cdiv(rows, wpb), wpb * 32, 0, stream>>>(ids, embed, vocab, d, rows,
                                                                          x16, x_f32, ssq, status, chk);
  return cudaGetLastError();
}

cudaError_t launch_row_ssq(const bf16 *x, long long rows, int d, f16 *x16, float *ssq, int *status,
                           SeqCheck chk, cudaStream_t stream) {
  const int wpb = 8;
  row_ssq_kernel<<<(unsigned)cdiv(rows, wpb), wpb * 32, 0, stream>>>(x, rows, d, x16, ssq, status, chk);
  return cudaGetLastError();
}

cudaError_t launch_row_ssq_f32(const float *x, long long rows, int d, f16 *x16, float *ssq, int *status,
                               SeqCheck chk, cudaStream_t stream) {
  const int wpb = 8;
  row_ssq_f32_kernel<<<(unsigned)cdiv(rows, wpb), wpb * 32, 0, stream>>>(x, rows, d, x16, ssq, status, chk);
  return cudaGetLastError();
}

cudaError_t launch_scale_cols_copy(const bf16 *src, const bf16 *norm_w, long long rows, int cols,
                                   f16 *dst, cudaStream_t stream) {
  scale_cols_kernel<<<grid_for(rows * cols, 256), 256, 0, stream>>>(src, norm_w, rows, cols, dst);
  return cudaGetLastError();
}

cudaError_t launch_interleave_gate_up(const bf16 *wg, const bf16 *wu, const bf16 *norm_w, int I,
                                      int d, f16 *dst, cudaStream_t stream) {
  interleave_gate_up_kernel<<<grid_for(2LL * I * d, 256), 256, 0, stream>>>(wg, wu, norm_w, I, d, dst);
  return cudaGetLastError();
}

// Keys and values of one layer for attention over a KV cache plus T new
// tokens, laid out as one left-padded sequence of Tk keys per (sequence b,
// kv head): slots [Tk - T - L_b, Tk - T) hold the L_b cached rows (bf16 ->
// f16, exact for values in f16 range), slots [Tk - T, Tk) the new rows, the
// slots before are zero.  K: [B, KV, Tk, hd]; V^T: [B, KV, hd, Tk_pad].
// vs[b] = Tk - T - L_b is the first visible slot (the padding start), and
// order[] lists the sequences by descending L_b (ties by index): the attention
// takes them in that order, the longest first, so that the short ones fill the
// tail of its launch.
// One CTA per (b, kv head) and 64 slots: K rows are converted 16 bytes per
// thread; V goes through shared memory and leaves as 64-key rows of V^T, so
// every global access is a contiguous run.  Slots in 128-key tiles wholly
// before the padding start are never read by the attention and are skipped.
constexpr int kGatherSlots = 64;

__global__ void __launch_bounds__(256) gather_cache_kv_kernel(
    const bf16 *__restrict__ kc, const bf16 *__restrict__ vc, int S_max, const int *__restrict__ cache_len,
    int lmax, const f16 *__restrict__ kn, const f16 *__restrict__ vtn, int T_pad, int KV, int T, int Tk, int Tk_pad,
    int hd, f16 *__restrict__ Kc, f16 *__restrict__ Vtc, int *__restrict__ vs, int *__restrict__ order) {
  extern __shared__ uint4 gather_smem[];
  // [64 slots][hd + 2]: the odd word stride keeps the column reads below at
  // two lanes per bank
  uint32_t *sV = reinterpret_cast<uint32_t *>(gather_smem);
  const int ldw = hd / 2 + 1;
  const long long bk = blockIdx.y;                   // b * KV + kv head
  const int b = static_cast<int>(bk / KV);
  const int r0 = blockIdx.x * kGatherSlots;
  int L = cache_len[b];
  L = L < 0 ? 0 : (L > lmax ? lmax : L);
  const int start = Tk - T - L;
  if (blockIdx.x == 0 && bk % KV == 0) {
    // this sequence's place in the order: the longer sequences, and the equal
    // ones of lower index, come before it
    __shared__ int s_rank;
    if (threadIdx.x == 0) s_rank = 0;
    __syncthreads();
    const int B = static_cast<int>(gridDim.y) / KV;
    int n = 0;
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
      int Li = cache_len[i];
      Li = Li < 0 ? 0 : (Li > lmax ? lmax : Li);
      n += (Li > L || (Li == L && i < b)) ? 1 : 0;
    }
    if (n) atomicAdd(&s_rank, n);
    __syncthreads();
    if (threadIdx.x == 0) {
      vs[b] = start;
      order[s_rank] = b;
    }
  }
  if (r0 + kGatherSlots <= start / 128 * 128) return;   // before the first key tile the attention reads
  const int cpr = hd / 8;                             // 16-byte chunks per row
  for (int i = threadIdx.x; i < kGatherSlots * cpr; i += blockDim.x) {
    const int sl = i / cpr, c = i - sl * cpr, r = r0 + sl;
    uint4 kw = make_uint4(0u, 0u, 0u, 0u), vw = make_uint4(0u, 0u, 0u, 0u);
    if (r >= start && r < Tk - T) {                   // cached row: bf16 -> f16
      const long long src = (bk * S_max + (r - start)) * hd + c * 8;
      const uint4 ku = *reinterpret_cast<const uint4 *>(kc + src);
      const uint4 vu = *reinterpret_cast<const uint4 *>(vc + src);
      const uint32_t *kp = reinterpret_cast<const uint32_t *>(&ku), *vp = reinterpret_cast<const uint32_t *>(&vu);
      uint32_t *ko = reinterpret_cast<uint32_t *>(&kw), *vo = reinterpret_cast<uint32_t *>(&vw);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 kf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kp[q]));
        const float2 vf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&vp[q]));
        const __half2 kh = __floats2half2_rn(kf.x, kf.y), vh = __floats2half2_rn(vf.x, vf.y);
        ko[q] = *reinterpret_cast<const uint32_t *>(&kh);
        vo[q] = *reinterpret_cast<const uint32_t *>(&vh);
      }
    } else if (r >= Tk - T && r < Tk) {              // new row: k as is, v from its transposed copy
      const int n = r - (Tk - T);
      kw = *reinterpret_cast<const uint4 *>(kn + (bk * T + n) * hd + c * 8);
      f16 *vh = reinterpret_cast<f16 *>(&vw);
#pragma unroll
      for (int e = 0; e < 8; ++e) vh[e] = vtn[(bk * hd + c * 8 + e) * T_pad + n];
    }
    if (r < Tk) *reinterpret_cast<uint4 *>(Kc + (bk * Tk + r) * hd + c * 8) = kw;
    const uint32_t *vq = reinterpret_cast<const uint32_t *>(&vw);   // zeros past Tk as well
#pragma unroll
    for (int q = 0; q < 4; ++q) sV[sl * ldw + c * 4 + q] = vq[q];
  }
  __syncthreads();
  // V^T rows: dimension d, eight keys per thread and step
  for (int i = threadIdx.x; i < hd * (kGatherSlots / 8); i += blockDim.x) {
    const int d = i / (kGatherSlots / 8), k8 = i - d * (kGatherSlots / 8);
    const int r = r0 + k8 * 8;
    if (r >= Tk_pad) continue;
    uint4 w;
    f16 *wh = reinterpret_cast<f16 *>(&w);
#pragma unroll
    for (int e = 0; e < 8; ++e) wh[e] = reinterpret_cast<const f16 *>(sV + (k8 * 8 + e) * ldw)[d];
    *reinterpret_cast<uint4 *>(Vtc + (bk * hd + d) * Tk_pad + r) = w;
  }
}

cudaError_t launch_gather_cache_kv(const bf16 *kc, const bf16 *vc, int S_max, const int *cache_len, int lmax,
                                   const f16 *kn, const f16 *vtn, int T_pad, int B, int KV, int T, int Tk,
                                   int Tk_pad, int hd, f16 *Kc, f16 *Vtc, int *vs, int *order,
                                   cudaStream_t stream) {
  if (hd % 8 || Tk_pad % 8 || B * KV > 65535) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>((Tk + kGatherSlots - 1) / kGatherSlots), static_cast<unsigned>(B * KV));
  const int smem = kGatherSlots * (hd + 2) * 2;
  gather_cache_kv_kernel<<<grid, 256, smem, stream>>>(kc, vc, S_max, cache_len, lmax, kn, vtn, T_pad, KV, T, Tk,
                                                      Tk_pad, hd, Kc, Vtc, vs, order);
  return cudaGetLastError();
}

// Appends one decode step's new keys and values ("model.py" (SmolLM2-135M)
// section 4: the cache grows by the new token's post-RoPE key and its value);
// one thread per 16 bytes of a row, K and V alike.
__global__ void append_kv_kernel(const bf16 *__restrict__ k_new, const bf16 *__restrict__ v_new,
                                 bf16 *__restrict__ k_cache, bf16 *__restrict__ v_cache,
                                 const int *__restrict__ cache_len, int L, int B, int KV, int S_max, int hd) {
  const int cpr = hd / 8;                                   // 16-byte chunks per row
  const long long items = 2LL * L * B * KV * cpr;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < items;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int ch = static_cast<int>(i % cpr);
    long long r = i / cpr;                                  // ((which * L + l) * B + b) * KV + kv
    const int kv = static_cast<int>(r % KV);
    r /= KV;
    const int b = static_cast<int>(r % B);
    r /= B;
    const int l = static_cast<int>(r % L);
    const int which = static_cast<int>(r / L);
    const int pos = cache_len[b];
    if (pos < 0 || pos >= S_max) continue;
    const long long src = (((long long)l * B + b) * KV + kv) * hd + ch * 8;
    const long long dst = ((((long long)l * B + b) * KV + kv) * S_max + pos) * hd + ch * 8;
    const bf16 *s = which ? v_new : k_new;
    bf16 *d = which ? v_cache : k_cache;
    *reinterpret_cast<uint4 *>(d + dst) = *reinterpret_cast<const uint4 *>(s + src);
  }
}

__global__ void bump_lengths_kernel(int *cache_len, int B, int S_max) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B && cache_len[b] >= 0 && cache_len[b] < S_max) cache_len[b] += 1;
}

cudaError_t launch_append_kv(const bf16 *k_new, const bf16 *v_new, bf16 *k_cache, bf16 *v_cache, int *cache_len,
                             int L, int B, int KV, int S_max, int hd, cudaStream_t stream) {
  const long long items = 2LL * L * B * KV * (hd / 8);
  append_kv_kernel<<<grid_for(items, 256), 256, 0, stream>>>(k_new, v_new, k_cache, v_cache, cache_len, L, B, KV,
                                                             S_max, hd);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bump_lengths_kernel<<<static_cast<unsigned>(cdiv(B, 128)), 128, 0, stream>>>(cache_len, B, S_max);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(int max_pos, int hd, float theta, float2 *table, cudaStream_t stream) {
  rope_table_kernel<<<grid_for(rope_table_rows(max_pos) * (hd / 4), 256), 256, 0, stream>>>(
      max_pos, hd, static_cast<double>(theta), reinterpret_cast<float4 *>(table));
  return cudaGetLastError();
}

}  // namespace smol
