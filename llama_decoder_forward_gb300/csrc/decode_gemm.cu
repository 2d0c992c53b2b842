// decode_gemm.cu - the four projections of a decode step when M = B <= 64.
//
// Same arithmetic as the tcgen05 GEMM of gemm.cu with the same epilogues
// ("model.py" (SmolLM2-135M) sections 3-6: RMSNorm folded into the weights
// with the row scale rstd = rsqrt(mean(x^2) + eps) applied to the product,
// q/k rotated by rotate_half RoPE at the token's position, the residual adds,
// SiLU(gate) * up), shaped for a decode step: a few dozen rows against weight
// matrices of 0.7-3.5 MB.  There the tile GEMM leaves most SMs idle and each
// CTA walks all of K through one MMA chain; here every CTA owns a narrow unit
// of output columns (8 to 32 weight rows, all of K), so 36-96 CTAs stream the
// weights at once:
//   - one thread requests the unit's weight boxes before waiting on the
//     preceding kernel (weights are inputs of the step), the activation rows
//     (M x K, zero-filled past M) after it, with a barrier per 64-wide k block;
//   - eight warps take interleaved 16-wide k steps of the whole unit with
//     mma.sync m16n8k16 (f16 operands, fp32 accumulation; at M <= 64 the
//     tensor work is a few hundred cycles, the legacy path is not the limit);
//   - the warps' partial sums meet in shared memory and every thread finishes
//     four adjacent output columns of one row through the epilogue.
// All waits are bounded (status word, no hang on a lost copy).
#include <math.h>

#include "common.cuh"
#include "prims.cuh"
#include "skinny.cuh"

namespace smol {

namespace {

constexpr int kSkThreads = 256;
constexpr int kSkWarps = kSkThreads / 32;
constexpr int kSkMaxKb = 32;                   // k blocks of 64 (K <= 2048)

template <int EPI, int NT>
__global__ void __launch_bounds__(kSkThreads, 1)
    skinny_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                       const GemmParams p) {
  extern __shared__ uint8_t sk_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(sk_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int nkb = p.K / 64;
  uint8_t *sA = smem;                                  // [nkb][64 rows][128 B], swizzled
  uint8_t *sW = smem + nkb * 8192;                     // [nkb][NT][8 rows][128 B], swizzled
  uint64_t *bars = reinterpret_cast<uint64_t *>(sW + nkb * NT * 1024);   // [nkb]
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + kSkMaxKb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int kb = 0; kb < nkb; ++kb) mbar_init(&bars[kb], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // QKV: this thread's rotation factors (fine and coarse (cos, sin) entries of
  // its two pairs at its row's position) depend only on inputs of the step,
  // so they are read before the wait on the preceding kernel
  float c0 = 1.f, s0 = 0.f, c1 = 1.f, s1 = 0.f;
  if constexpr (EPI == kEpiQkvRope) {
    const int row = threadIdx.x >> 2, c = (threadIdx.x & 3) * 2;
    if (p.rope && row < p.M && (u >> 2) < p.H + p.KV) {   // no table: a NoPE block
      int pos = 0;
      if (p.pos_add) {
        const int pa = p.pos_add[row];                  // one token per sequence
        pos = pa < 0 ? 0 : (pa > p.pos_limit ? p.pos_limit : pa);
      }
      pos = pos < 0 ? 0 : (pos >= p.max_pos ? p.max_pos - 1 : pos);
      const int n_coarse = static_cast<int>(cdiv(p.max_pos, 64));
      const int jj = ((u & 3) * 8 + c) >> 1;            // pairs i0+c and i0+c+1
      const float4 f = reinterpret_cast<const float4 *>(p.rope)[jj * 64 + (pos & 63)];
      const float4 gq = reinterpret_cast<const float4 *>(p.rope)[16 * 64 + jj * n_coarse + (pos >> 6)];
      c0 = gq.x * f.x - gq.y * f.y;
      s0 = gq.y * f.x + gq.x * f.y;
      c1 = gq.z * f.z - gq.w * f.w;
      s1 = gq.w * f.z + gq.z * f.w;
    }
  }
  if (threadIdx.x == 0) {
    griddep_launch_dependents();
    // weights first (inputs of the step), then the rows the preceding kernel wrote
    for (int kb = 0; kb < nkb; ++kb) {
      mbar_arrive_expect_tx(&bars[kb], 8192 + NT * 1024);
#pragma unroll
      for (int g = 0; g < NT; ++g) {
        tma_load_2d(sW + (kb * NT + g) * 1024, &tmW, &bars[kb], kb * 64, unit_wrow<EPI, NT>(u, g));
      }
    }
    griddep_wait();
    for (int kb = 0; kb < nkb; ++kb) tma_load_2d(sA + kb * 8192, &tmA, &bars[kb], kb * 64, 0);
  } else {
    griddep_wait();                                   // the epilogue reads the preceding kernel's output
  }

  // ---- products: warp w takes the 16-wide k steps s = w, w + 8, ...
  float acc[4][NT][4];
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
  bool ok = true;
  int waited = -1;
  const uint32_t a_base = smem_u32(sA), w_base = smem_u32(sW);
  for (int s = warp; s < nkb * 4; s += kSkWarps) {
    const int kb = s >> 2, kk = s & 3;
    if (kb != waited) {
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[kb], 0, abort_flag));
      if (!ok) break;
      waited = kb;
    }
    uint32_t bw[NT][2];
    if constexpr (NT == 1) {
      // lanes 0-7: rows, k chunk 2kk; lanes 8-15: k chunk 2kk+1
      const int r = lane & 7, ch = kk * 2 + ((lane >> 3) & 1);
      ldsm2(bw[0], w_base + kb * NT * 1024 + r * 128 + ((ch ^ r) << 4));
    } else {
#pragma unroll
      for (int g = 0; g < NT; g += 2) {
        const int r = lane & 7, ch = kk * 2 + ((lane >> 3) & 1), gg = g + (lane >> 4);
        uint32_t t4[4];
        ldsm4(t4, w_base + (kb * NT + gg) * 1024 + r * 128 + ((ch ^ r) << 4));
        bw[g][0] = t4[0];
        bw[g][1] = t4[1];
        bw[g + 1][0] = t4[2];
        bw[g + 1][1] = t4[3];
      }
    }
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int row = mt * 16 + (lane & 15), ch = kk * 2 + (lane >> 4);
      uint32_t a4[4];
      ldsm4(a4, a_base + kb * 8192 + row * 128 + ((ch ^ (row & 7)) << 4));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_f16_16816(acc[mt][nt], a4, bw[nt][0], bw[nt][1]);
    }
  }
  if (!ok) {
    if (lane == 0) atomicCAS(p.status, 0, kDevTimeoutEpilogue);
    *abort_flag = 1;
  }
  // every copy has landed before shared memory is reused or the CTA exits
  if (threadIdx.x == 0) {
    int dummy = 0;
    for (int kb = 0; kb < nkb; ++kb)
      if (!mbar_wait_bounded(&bars[kb], 0, reinterpret_cast<volatile int *>(&dummy)))
        atomicCAS(p.status, 0, kDevTimeoutDrain);
  }
  __syncthreads();
  if (*abort_flag) return;                            // uniform: set before the barrier

  // ---- the warps' partial sums: red[w][row][NT*8] in the A area
  constexpr int NC = NT * 8;
  float *red = reinterpret_cast<float *>(sA);
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int r0 = mt * 16 + (lane >> 2), c = nt * 8 + (lane & 3) * 2;
      *reinterpret_cast<float2 *>(red + (warp * 64 + r0) * NC + c) = make_float2(acc[mt][nt][0], acc[mt][nt][1]);
      *reinterpret_cast<float2 *>(red + (warp * 64 + r0 + 8) * NC + c) = make_float2(acc[mt][nt][2], acc[mt][nt][3]);
    }
  __syncthreads();
  auto sum4 = [&](int row, int c) {
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kSkWarps; ++w) {
      const float4 v = *reinterpret_cast<const float4 *>(red + (w * 64 + row) * NC + c);
      t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
    }
    return t;
  };
  auto rstd = [&](int row) { return p.ssq_in ? rsqrtf(p.ssq_in[row] * p.inv_dim + p.eps) : 1.0f; };
  if (u == 0 && p.ssq_zero && threadIdx.x < p.M) p.ssq_zero[threadIdx.x] = 0.f;

  // ---- epilogues: thread -> (row, four adjacent output columns)
  if constexpr (EPI == kEpiResidual) {
    constexpr int GPR = NC / 4;                      // column groups per row (2 or 4 lanes)
    const int t = threadIdx.x;
    if (t >= 64 * GPR) return;
    const int row = t / GPR, c = (t % GPR) * 4;
    const bool row_ok = row < p.M;
    float part = 0.f;
    if (row_ok) {
      const float4 v = sum4(row, c);
      const long long off = (long long)row * p.ldo + u * NC + c;
      const uint2 rr = *reinterpret_cast<const uint2 *>(p.resid_f16 + off);
      const float2 r01 = unpack_f16x2(rr.x), r23 = unpack_f16x2(rr.y);
      const __half2 o01 = __floats2half2_rn(r01.x + v.x, r01.y + v.y);
      const __half2 o23 = __floats2half2_rn(r23.x + v.z, r23.y + v.w);
      uint2 ow;
      ow.x = *reinterpret_cast<const uint32_t *>(&o01);
      ow.y = *reinterpret_cast<const uint32_t *>(&o23);
      *reinterpret_cast<uint2 *>(static_cast<f16 *>(p.out) + off) = ow;
      const float2 f01 = __half22float2(o01), f23 = __half22float2(o23);
      part = f01.x * f01.x + f01.y * f01.y + f23.x * f23.x + f23.y * f23.y;   // sum of the rounded values
    }
#pragma unroll
    for (int o = 1; o < GPR; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (row_ok && (t % GPR) == 0 && p.ssq_out) atomicAdd(p.ssq_out + row, part);
    // the sum of squares of the rounded outputs is finite iff none overflowed
    if (row_ok && (t % GPR) == 0 && !isfinite(part)) set_status(p.status, kDevRange);
  } else if constexpr (EPI == kEpiSwiglu) {
    // columns 0..15 gate, 16..31 up of act columns 16u .. 16u+15
    const int row = threadIdx.x >> 2, c = (threadIdx.x & 3) * 4;
    if (row >= p.M) return;
    const float rs = rstd(row);
    const float4 g = sum4(row, c), up = sum4(row, 16 + c);
    const float gv[4] = {g.x * rs, g.y * rs, g.z * rs, g.w * rs};
    const float uv[4] = {up.x * rs, up.y * rs, up.z * rs, up.w * rs};
    float y[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) y[j] = __fdividef(gv[j], 1.0f + __expf(-gv[j])) * uv[j];   // SiLU(g) * u
    const __half2 y01 = __floats2half2_rn(y[0], y[1]), y23 = __floats2half2_rn(y[2], y[3]);
    uint2 ow;
    ow.x = *reinterpret_cast<const uint32_t *>(&y01);
    ow.y = *reinterpret_cast<const uint32_t *>(&y23);
    *reinterpret_cast<uint2 *>(static_cast<f16 *>(p.out) + (long long)row * p.ldo + u * 16 + c) = ow;
  } else {
    // columns 0..7: first elements of pairs i0..i0+7, 8..15: their partners
    // (+32); thread -> pairs i0 + c and i0 + c + 1 of one row (one token)
    const int row = threadIdx.x >> 2, c = (threadIdx.x & 3) * 2;
    if (row >= p.M || c >= 8) return;
    const int gh = u >> 2, i0 = (u & 3) * 8;
    const int n_heads = p.H + 2 * p.KV;
    if (gh >= n_heads) return;
    const float rs = rstd(row);
    float2 lo2 = make_float2(0.f, 0.f), hi2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kSkWarps; ++w) {
      const float2 v = *reinterpret_cast<const float2 *>(red + (w * 64 + row) * NC + c);
      const float2 x = *reinterpret_cast<const float2 *>(red + (w * 64 + row) * NC + 8 + c);
      lo2.x += v.x; lo2.y += v.y; hi2.x += x.x; hi2.y += x.y;
    }
    const float a[2] = {lo2.x * rs, lo2.y * rs}, bb[2] = {hi2.x * rs, hi2.y * rs};
    const bool is_q = gh < p.H, is_k = !is_q && gh < p.H + p.KV;
    float ylo[2], yhi[2];
    if (is_q || is_k) {
      ylo[0] = a[0] * c0 - bb[0] * s0;
      yhi[0] = a[0] * s0 + bb[0] * c0;
      ylo[1] = a[1] * c1 - bb[1] * s1;
      yhi[1] = a[1] * s1 + bb[1] * c1;
    } else {
      ylo[0] = a[0]; ylo[1] = a[1];
      yhi[0] = bb[0]; yhi[1] = bb[1];
    }
    const int hsub = is_q ? gh : (is_k ? gh - p.H : gh - p.H - p.KV);
    const long long base = ((long long)row * (is_q ? p.H : p.KV) + hsub) * 64;   // T = 1
    const int d_lo = i0 + c, d_hi = 32 + i0 + c;
    if (is_q) {
      *reinterpret_cast<__half2 *>(p.q + base + d_lo) = __floats2half2_rn(ylo[0], ylo[1]);
      *reinterpret_cast<__half2 *>(p.q + base + d_hi) = __floats2half2_rn(yhi[0], yhi[1]);
    } else {
      f16 *d16 = is_k ? p.k : p.v;
      bf16 *dbf = is_k ? p.k_bf : p.v_bf;
      if (d16) {
        *reinterpret_cast<__half2 *>(d16 + base + d_lo) = __floats2half2_rn(ylo[0], ylo[1]);
        *reinterpret_cast<__half2 *>(d16 + base + d_hi) = __floats2half2_rn(yhi[0], yhi[1]);
      }
      if (dbf) {
        *reinterpret_cast<__nv_bfloat162 *>(dbf + base + d_lo) = __floats2bfloat162_rn(ylo[0], ylo[1]);
        *reinterpret_cast<__nv_bfloat162 *>(dbf + base + d_hi) = __floats2bfloat162_rn(yhi[0], yhi[1]);
      }
    }
  }
}

template <int EPI, int NT>
cudaError_t launch_sk(const CUtensorMap &ta, const CUtensorMap &tw, const GemmParams &p, int units,
                      cudaStream_t st) {
  const int nkb = p.K / 64;
  const int smem = 1024 + nkb * 8192 + nkb * NT * 1024 + kSkMaxKb * 8 + 16;
  constexpr auto kern = skinny_gemm_kernel<EPI, NT>;
  cudaError_t e = ensure_smem_attr<kern>(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units));
  cfg.blockDim = dim3(kSkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, ta, tw, p);
}

// weight rows per unit (8-row groups) for an epilogue and K
int sk_nt(int epi, int K) {
  if (epi == kEpiQkvRope) return 2;
  if (epi == kEpiSwiglu) return 4;
  return K > 1024 ? 1 : 2;
}

}  // namespace

bool skinny_gemm_supported(int epi, const GemmParams &p) {
  if (p.M < 1 || p.M > 64 || p.K % 64 || p.K / 64 > kSkMaxKb || p.status == nullptr) return false;
  const int nt = sk_nt(epi, p.K);
  if (p.K / 64 < 2 * nt) return false;               // the partial sums reuse the A area
  const long long smem = 1024 + (long long)(p.K / 64) * (8192 + nt * 1024) + kSkMaxKb * 8 + 16;
  if (smem > 232448) return false;
  if (epi == kEpiResidual)
    return p.out && p.resid_f16 && !p.resid && !p.resid_f32 && !p.out_f32 && p.out_is_f16 &&
           p.N % (nt * 8) == 0 && p.ldo % 4 == 0;
  if (epi == kEpiSwiglu) return p.out && p.out_is_f16 && p.N % 128 == 0 && p.ldo % 4 == 0;
  if (epi == kEpiQkvRope)
    return p.hd == 64 && p.T == 1 && p.q && !p.v_t && !p.valid_start &&
           p.N == (p.H + 2 * p.KV) * 64;
  return false;
}

cudaError_t launch_skinny_gemm(int epi, const void *A, const void *W, const GemmParams &p,
                               cudaStream_t st) {
  if (!skinny_gemm_supported(epi, p)) return cudaErrorInvalidValue;
  const int nt = sk_nt(epi, p.K);
  CUtensorMap ta, tw;
  if (!get_tmap_2d(&ta, A, p.M, p.K, p.K, 64, 64, true)) return cudaErrorInvalidValue;
  if (!get_tmap_2d(&tw, W, p.N, p.K, p.K, 64, 8, true)) return cudaErrorInvalidValue;
  if (epi == kEpiQkvRope) return launch_sk<kEpiQkvRope, 2>(ta, tw, p, (p.H + 2 * p.KV) * 4, st);
  if (epi == kEpiSwiglu) return launch_sk<kEpiSwiglu, 4>(ta, tw, p, p.N / 2 / 16, st);
  if (nt == 1) return launch_sk<kEpiResidual, 1>(ta, tw, p, p.N / 8, st);
  return launch_sk<kEpiResidual, 2>(ta, tw, p, p.N / 16, st);
}

}  // namespace smol
