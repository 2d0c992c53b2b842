// gemm.cu - persistent tcgen05 GEMM with fused decoder epilogues (sm_103a).
//
// D[M, N] = A[M, K] * B[N, K]^T, f16 operands, fp32 accumulation in TMEM.
// One CTA per SM walks tiles of 128 x BN.  Warp roles:
//   warp 0      TMA producer: 128x64 A box and BNx64 B box per stage (128 B swizzle)
//   warp 1      TMEM owner; lane 0 issues tcgen05.mma (M=128, N=BN, K=16) and commits
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 16 columns per load, fused math,
//               16-byte global stores
// Two TMEM accumulators (2 x BN columns) let the epilogue of tile i overlap the
// main loop of tile i+1.  Every wait is bounded; a wait that gives up records a
// status code, raises a CTA-wide abort flag, drains in-flight copies and MMAs,
// frees TMEM and returns.
//
// The epilogues implement, per output row r (one token):
//   kEpiQkvRope  [q|k|v] = rstd_r * (x_r . W'^T); rotate-half RoPE on q and k heads
//                ("model.py" (SmolLM2-135M) section 3 apply_rope, section 4 projections;
//                "components.py" RotaryEmbedding) with W' the norm-folded weights;
//   kEpiResidual out = resid + D  (section 6 SmolBlock residual adds);
//   kEpiSwiglu   a = SiLU(rstd*g) * (rstd*u)  (section 5 SmolMLP; components.py SwiGLU_FFN);
//   kEpiScale    logits = rstd * D  (section 7 final norm + tied lm_head).
#include <stdio.h>

#include "common.cuh"
#include "prims.cuh"

namespace smol {

template <int BN>
struct GemmCfg {
  static constexpr int BM = 128;
  static constexpr int BK = 64;                       // 64 x 16-bit = 128 B = one swizzle row
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES_RAW = (200 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int TMEM_COLS = (2 * BN <= 128) ? 128 : (2 * BN <= 256 ? 256 : 512);
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + BAR_BYTES;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128");
  static_assert(B_BYTES % 1024 == 0, "B stage must keep 1024-byte alignment");
  static_assert((2 * STAGES + 5) * 8 + 8 <= BAR_BYTES, "barrier area");
};

__device__ __forceinline__ void record_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float row_rstd(const GemmParams &p, int row) {
  if (p.ssq_in == nullptr || row >= p.M) return 1.0f;
  return rsqrtf(p.ssq_in[row] * p.inv_dim + p.eps);
}

__device__ __forceinline__ void store16(void *dst, const float (&v)[16], bool as_f16) {
  uint4 w0, w1;
  if (as_f16) {
    w0 = make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]),
                    pack_f16x2(v[6], v[7]));
    w1 = make_uint4(pack_f16x2(v[8], v[9]), pack_f16x2(v[10], v[11]), pack_f16x2(v[12], v[13]),
                    pack_f16x2(v[14], v[15]));
  } else {
    w0 = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
    w1 = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
                    pack_bf16x2(v[14], v[15]));
  }
  uint4 *d = reinterpret_cast<uint4 *>(dst);
  d[0] = w0;
  d[1] = w1;
}

// element pointer into a 16-bit row-major buffer
__device__ __forceinline__ void *elem16(void *base, long long idx) {
  return static_cast<uint16_t *>(base) + idx;
}

// ---------------------------------------------------------------- epilogues
// All tcgen05.ld calls are executed by every lane of the warp (they are
// warp-collective); only the global stores depend on the row bound.

template <int BN>
__device__ __forceinline__ void epi_scale(const GemmParams &p, uint32_t taddr, int row, int n0) {
  const float rs = row_rstd(p, row);
  const bool row_ok = row < p.M;
#pragma unroll 1
  for (int c = 0; c < BN; c += 16) {
    uint32_t r[16];
    tmem_ld16(taddr + c, r);
    tmem_ld_wait();
    const int col = n0 + c;
    if (row_ok && col < p.N) {
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]) * rs;
      store16(elem16(p.out, (long long)row * p.ldo + col), v, p.out_is_f16);
    }
  }
}

// out = resid + D.  The residual comes in fp32 or bf16; the result is written
// in fp32 (out_f32) and/or 16 bits (out).  The row sum of squares feeding the
// next RMSNorm is taken over the values the next step reads: fp32 when out_f32
// is written, else the rounded 16-bit values.
template <int BN>
__device__ __forceinline__ void epi_residual(const GemmParams &p, uint32_t taddr, int row, int n0) {
  const bool row_ok = row < p.M;
  float part = 0.f;
#pragma unroll 1
  for (int c = 0; c < BN; c += 16) {
    uint32_t r[16];
    tmem_ld16(taddr + c, r);
    tmem_ld_wait();
    const int col = n0 + c;
    if (row_ok && col < p.N) {
      const long long off = (long long)row * p.ldo + col;
      float v[16];
      if (p.resid_f32) {
        const float4 *src = reinterpret_cast<const float4 *>(p.resid_f32 + off);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 h = src[q];
          v[4 * q] = h.x; v[4 * q + 1] = h.y; v[4 * q + 2] = h.z; v[4 * q + 3] = h.w;
        }
      } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.resid + off);
        const uint4 h0 = src[0], h1 = src[1];
        const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 h = unpack_bf16x2(hw[e]);
          v[2 * e] = h.x;
          v[2 * e + 1] = h.y;
        }
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] += __uint_as_float(r[e]);
      if (p.out_f32) {
        float4 *dst = reinterpret_cast<float4 *>(p.out_f32 + off);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
#pragma unroll
        for (int e = 0; e < 16; ++e) part = fmaf(v[e], v[e], part);
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float rv = p.out_is_f16 ? __half2float(__float2half_rn(v[e]))
                                        : __bfloat162float(__float2bfloat16_rn(v[e]));
          part = fmaf(rv, rv, part);
        }
      }
      if (p.out) store16(elem16(p.out, off), v, p.out_is_f16);
    }
  }
  if (row_ok && p.ssq_out) atomicAdd(p.ssq_out + row, part);
}

template <int BN>
__device__ __forceinline__ void epi_swiglu(const GemmParams &p, uint32_t taddr, int row, int n0,
                                           int n_blk) {
  const float rs = row_rstd(p, row);
  const bool row_ok = row < p.M;
  const int I = p.N / 2;
#pragma unroll 1
  for (int grp = 0; grp < BN / 128; ++grp) {
    const int out_col0 = (n0 / 128 + grp) * 64;
#pragma unroll 1
    for (int e0 = 0; e0 < 64; e0 += 16) {
      uint32_t g[16], u[16];
      tmem_ld16(taddr + grp * 128 + e0, g);
      tmem_ld16(taddr + grp * 128 + 64 + e0, u);
      tmem_ld_wait();
      if (row_ok && out_col0 + e0 < I) {
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float gv = __uint_as_float(g[e]) * rs;
          const float uv = __uint_as_float(u[e]) * rs;
          v[e] = gv / (1.0f + __expf(-gv)) * uv;
        }
        store16(elem16(p.out, (long long)row * p.ldo + out_col0 + e0), v, p.out_is_f16);
      }
    }
  }
  if (n_blk == 0 && row_ok && p.ssq_zero) p.ssq_zero[row] = 0.f;
}

template <int BN, int HD>
__device__ __forceinline__ void epi_qkv_rope(const GemmParams &p, uint32_t taddr, int row, int n0,
                                             int n_blk) {
  const float rs = row_rstd(p, row);
  const bool row_ok = row < p.M;
  const int rr = row_ok ? row : 0;
  const int b = rr / p.T, t = rr - b * p.T;
  int pos = t - (p.valid_start ? p.valid_start[b] : 0);
  if (p.pos_add) {
    const int pa = p.pos_add[b];
    pos += pa < 0 ? 0 : (pa > p.pos_limit ? p.pos_limit : pa);
  }
  pos = pos < 0 ? 0 : (pos >= p.max_pos ? p.max_pos - 1 : pos);
  const float2 *cs = p.rope + (long long)pos * (HD / 2);
  const int n_heads_total = p.H + 2 * p.KV;
#pragma unroll 1
  for (int hh = 0; hh < BN / HD; ++hh) {
    const int gh = n0 / HD + hh;                 // global head index in [q | k | v]
    if (gh >= n_heads_total) break;              // uniform across the warp
    const uint32_t tcol = taddr + hh * HD;
    const bool is_q = gh < p.H, is_k = !is_q && gh < p.H + p.KV;
    long long off;                               // element offset of (b, head, t, 0)
    f16 *dst;
    bf16 *dst_bf;
    if (is_q) {
      off = (((long long)b * p.H + gh) * p.T + t) * HD;
      dst = p.q;
      dst_bf = nullptr;
    } else {
      const int kvh = is_k ? gh - p.H : gh - p.H - p.KV;
      off = (((long long)b * p.KV + kvh) * p.T + t) * HD;
      dst = is_k ? p.k : p.v;
      dst_bf = is_k ? p.k_bf : p.v_bf;
    }
    if (!is_q && !is_k) {
#pragma unroll 1
      for (int i0 = 0; i0 < HD; i0 += 16) {
        uint32_t x[16];
        tmem_ld16(tcol + i0, x);
        tmem_ld_wait();
        if (row_ok) {
          float y[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) y[e] = __uint_as_float(x[e]) * rs;
          if (dst) store16(dst + off + i0, y, true);
          if (dst_bf) store16(dst_bf + off + i0, y, false);
        }
      }
      continue;
    }
#pragma unroll 1
    for (int i0 = 0; i0 < HD / 2; i0 += 16) {
      uint32_t x1[16], x2[16];
      tmem_ld16(tcol + i0, x1);
      tmem_ld16(tcol + HD / 2 + i0, x2);
      tmem_ld_wait();
      if (row_ok) {
        float y1[16], y2[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 c = cs[i0 + e];
          const float a = __uint_as_float(x1[e]) * rs;
          const float bb = __uint_as_float(x2[e]) * rs;
          y1[e] = a * c.x - bb * c.y;
          y2[e] = a * c.y + bb * c.x;
        }
        if (dst) {
          store16(dst + off + i0, y1, true);
          store16(dst + off + HD / 2 + i0, y2, true);
        }
        if (dst_bf) {
          store16(dst_bf + off + i0, y1, false);
          store16(dst_bf + off + HD / 2 + i0, y2, false);
        }
      }
    }
  }
  if (n_blk == 0 && row_ok && p.ssq_zero) p.ssq_zero[row] = 0.f;
}

// ---------------------------------------------------------------- kernel
template <int BN, int EPI, int HD>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
  using C = GemmCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + C::STAGES * C::A_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sB + C::STAGES * C::B_BYTES);
  uint64_t *full = bars;
  uint64_t *empty = bars + C::STAGES;
  uint64_t *tfull = bars + 2 * C::STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_n = static_cast<int>(cdiv(p.N, BN));
  const int num_tiles = static_cast<int>(cdiv(p.M, C::BM)) * num_n;
  const int num_kb = static_cast<int>(cdiv(p.K, C::BK));

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      uint32_t stage = 0, phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int m_blk = tile / num_n, n_blk = tile - m_blk * num_n;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          tma_load_2d(sA + stage * C::A_BYTES, &tmA, &full[stage], kb * C::BK, m_blk * C::BM);
          tma_load_2d(sB + stage * C::B_BYTES, &tmB, &full[stage], kb * C::BK, n_blk * BN);
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        record_status(p.status, kDevTimeoutProducer);
        *abort_flag = 1;
        // wait (bounded) for the copies still in flight before the CTA exits
        const long long first = issued > C::STAGES ? issued - C::STAGES : 0;
        int dummy = 0;
        for (long long j = first; j < issued; ++j) {
          if (!mbar_wait_bounded(&full[j % C::STAGES], (uint32_t)((j / C::STAGES) & 1),
                                 reinterpret_cast<volatile int *>(&dummy)))
            record_status(p.status, kDevTimeoutDrain);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t kIdesc = idesc_f16_f32(C::BM, BN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, any = false;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t a_desc = sdesc_kmajor_sw128(smem_u32(sA + stage * C::A_BYTES));
          const uint64_t b_desc = sdesc_kmajor_sw128(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
          for (int k = 0; k < C::BK / 16; ++k) {
            // +32 bytes per K step of 16 elements (encoded >> 4)
            umma_f16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, kIdesc, (kb | k) != 0);
          }
          any = true;
          umma_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok) {
        record_status(p.status, kDevTimeoutMma);
        *abort_flag = 1;
        if (any) {
          // wait (bounded) for the MMAs already issued before TMEM is freed
          umma_commit(drain);
          int dummy = 0;
          if (!mbar_wait_bounded(drain, 0, reinterpret_cast<volatile int *>(&dummy)))
            record_status(p.status, kDevTimeoutDrain);
        }
      }
    }
  } else {
    // -------------------------------------------------- epilogue (warps 2..5)
    const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const int m_blk = tile / num_n, n_blk = tile - m_blk * num_n;
      // every lane waits; the outcome is made warp-uniform because the TMEM
      // loads below are warp-collective
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag));
      if (!ok) {
        if (lane == 0) record_status(p.status, kDevTimeoutEpilogue);
        *abort_flag = 1;
        break;
      }
      tc_fence_after_sync();
      const int row = m_blk * C::BM + quarter * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
      const int n0 = n_blk * BN;
      if constexpr (EPI == kEpiScale) epi_scale<BN>(p, taddr, row, n0);
      else if constexpr (EPI == kEpiResidual) epi_residual<BN>(p, taddr, row, n0);
      else if constexpr (EPI == kEpiSwiglu) epi_swiglu<BN>(p, taddr, row, n0, n_blk);
      else epi_qkv_rope<BN, HD>(p, taddr, row, n0, n_blk);
      tc_fence_before_sync();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

bool make_tmap_f16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                    uint64_t row_pitch_elems, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_pitch_elems * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int gemm_pick_bn(int epi, int N, int hd) {
  if (N <= 0 || N % 16) return 0;
  if (epi == kEpiQkvRope) {
    if (N % hd) return 0;
    const int cands[3] = {256, 192, 128};
    for (int c : cands)
      if (c % hd == 0 && N % c == 0) return c;
    return hd == 64 ? 128 : 256;                  // ragged last tile (whole heads)
  }
  if (epi == kEpiSwiglu) {
    if (N % 128) return 0;
    return N % 256 == 0 ? 256 : 128;
  }
  const int cands[4] = {256, 192, 128, 64};
  for (int c : cands)
    if (N % c == 0) return c;
  return 128;
}

template <int BN, int EPI, int HD>
static cudaError_t launch_impl(const CUtensorMap &ta, const CUtensorMap &tb, const GemmParams &p,
                               int num_sms, cudaStream_t stream) {
  using C = GemmCfg<BN>;
  auto kern = gemm_tc_kernel<BN, EPI, HD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long tiles = cdiv(p.M, C::BM) * cdiv(p.N, BN);
  const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
  kern<<<grid, 192, C::SMEM_BYTES, stream>>>(ta, tb, p);
  return cudaGetLastError();
}

cudaError_t launch_gemm(int epi, int bn, const void *A, const void *B, const GemmParams &p,
                        int num_sms, cudaStream_t stream) {
  CUtensorMap ta, tb;
  if (!make_tmap_f16(&ta, A, p.M, p.K, p.K, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_f16(&tb, B, p.N, p.K, p.K, bn)) return cudaErrorInvalidValue;
  switch (epi) {
    case kEpiScale:
      if (bn == 256) return launch_impl<256, kEpiScale, 64>(ta, tb, p, num_sms, stream);
      if (bn == 192) return launch_impl<192, kEpiScale, 64>(ta, tb, p, num_sms, stream);
      if (bn == 128) return launch_impl<128, kEpiScale, 64>(ta, tb, p, num_sms, stream);
      if (bn == 64) return launch_impl<64, kEpiScale, 64>(ta, tb, p, num_sms, stream);
      break;
    case kEpiResidual:
      if (bn == 256) return launch_impl<256, kEpiResidual, 64>(ta, tb, p, num_sms, stream);
      if (bn == 192) return launch_impl<192, kEpiResidual, 64>(ta, tb, p, num_sms, stream);
      if (bn == 128) return launch_impl<128, kEpiResidual, 64>(ta, tb, p, num_sms, stream);
      if (bn == 64) return launch_impl<64, kEpiResidual, 64>(ta, tb, p, num_sms, stream);
      break;
    case kEpiSwiglu:
      if (bn == 256) return launch_impl<256, kEpiSwiglu, 64>(ta, tb, p, num_sms, stream);
      if (bn == 128) return launch_impl<128, kEpiSwiglu, 64>(ta, tb, p, num_sms, stream);
      break;
    case kEpiQkvRope:
      if (p.hd == 64) {
        if (bn == 256) return launch_impl<256, kEpiQkvRope, 64>(ta, tb, p, num_sms, stream);
        if (bn == 192) return launch_impl<192, kEpiQkvRope, 64>(ta, tb, p, num_sms, stream);
        if (bn == 128) return launch_impl<128, kEpiQkvRope, 64>(ta, tb, p, num_sms, stream);
        if (bn == 64) return launch_impl<64, kEpiQkvRope, 64>(ta, tb, p, num_sms, stream);
      } else if (p.hd == 128) {
        if (bn == 256) return launch_impl<256, kEpiQkvRope, 128>(ta, tb, p, num_sms, stream);
        if (bn == 128) return launch_impl<128, kEpiQkvRope, 128>(ta, tb, p, num_sms, stream);
      }
      break;
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace smol
