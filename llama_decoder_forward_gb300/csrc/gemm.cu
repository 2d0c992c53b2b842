// gemm.cu - persistent tcgen05 GEMM with fused decoder epilogues (sm_103a).
//
// D[M, N] = A[M, K] * B[N, K]^T, f16 operands, fp32 accumulation in TMEM.
// One CTA per SM walks tiles of 128 x BN.  With PAIR == 2 two CTAs (a
// cluster of 2 on one TPC) share each 256 x BN tile: the even CTA issues
// cta_group::2 MMAs (M = 256) that read each CTA's own 128-row A box and
// half of the B box from each CTA's shared memory and write each CTA's 128
// rows into its own TMEM.  Per SM that halves the B bytes written by TMA and
// read by the tensor pipe; with one CTA, shared-memory bandwidth (TMA fill
// plus MMA operand reads) rather than the tensor pipe bounds these
// narrow-K GEMMs.  Warp roles:
//   warp 0      TMA producer: 128x64 A box and BNx64 B box per stage (128 B swizzle)
//   warp 1      TMEM owner; lane 0 issues tcgen05.mma (M=128, N=BN, K=16) and commits
//   warps 2..9  epilogue: two warps per TMEM lane quarter split the tile's columns
// Two TMEM accumulators (2 x BN columns) let the epilogue of tile i overlap the
// main loop of tile i+1.  Every wait is bounded; a wait that gives up records a
// status code, raises a CTA-wide abort flag, drains in-flight copies and MMAs,
// frees TMEM and returns.
//
// Epilogue data movement: tcgen05.ld gives each thread one row of the tile, so
// a direct global access by a warp would touch 32 rows (32 cache lines) per
// instruction.  Instead every epilogue warp owns 32-row staging tiles in shared
// memory (128-byte rows, 16-byte chunks XOR-swizzled by row so both the
// row-per-thread and the row-per-lane-group accesses are conflict-free);
// global reads and writes go through them with consecutive lanes on
// consecutive 16-byte chunks of a row (4-8 full rows per instruction).
//
// The epilogues implement, per output row r (one token):
//   kEpiQkvRope  [q|k|v] = rstd_r * (x_r . W'^T); rotate-half RoPE on q and k heads
//                ("model.py" (SmolLM2-135M) section 3 apply_rope, section 4 projections;
//                "components.py" RotaryEmbedding) with W' the norm-folded weights;
//   kEpiResidual out = resid + D  (section 6 SmolBlock residual adds);
//   kEpiSwiglu   a = SiLU(rstd*g) * (rstd*u)  (section 5 SmolMLP; components.py SwiGLU_FFN);
//   kEpiScale    logits = rstd * D  (section 7 final norm + tied lm_head).
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "prims.cuh"

namespace smol {

constexpr int kEpiWarps = 8;                       // two per TMEM lane quarter
constexpr int kSplit = kEpiWarps / 4;              // warps sharing one quarter's columns
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;
constexpr int kStgBytes = 32 * 128;                // one staging tile: 32 rows x 128 B

// Tensor maps of the epilogues' TMA traffic; GemmParams::epi_tma says which
// are valid.  Boxes are one warp's staging tile: 32 rows x 64 16-bit columns
// (128-byte swizzle, the staging layout below), or for V^T 64 dims x 32 tokens.
struct EpiMaps {
  CUtensorMap out;     // 16-bit output rows [M, out columns] (pitch ldo)
  CUtensorMap resid;   // 16-bit residual rows [M, N] (pitch ldo)
  CUtensorMap q, k;    // [B*H*T, 64] and [B*KV*T, 64]
  CUtensorMap vt;      // [B*KV*64, T] with pitch T_pad, no swizzle
};
enum EpiTma : int { kTmaOut = 1, kTmaResid = 2, kTmaQkv = 4 };

// Staging tiles (4 KB each) per epilogue warp: two for the residual and QKV
// epilogues (residual units loaded ahead of the accumulator; alternating
// tiles let one TMA store drain while the next unit is staged), one for the
// others.
template <int EPI>
struct EpiStage {
  static constexpr int kTiles = (EPI == 1 /*kEpiResidual*/ || EPI == 0 /*kEpiQkvRope*/) ? 2 : 1;
  static constexpr int kPerWarp = kTiles * kStgBytes;
};

template <int BN, int EPI, int PAIR>
struct GemmCfg {
  static constexpr int BM = 128;                      // rows per CTA
  static constexpr int BK = 64;                       // 64 x 16-bit = 128 B = one swizzle row
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = (BN / PAIR) * BK * 2;  // this CTA's share of the B box
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_BYTES = kEpiWarps * EpiStage<EPI>::kPerWarp;
  // QKV (hd 64): the fine part of the RoPE table (64 positions x 16 float4)
  // is copied to shared memory once per CTA
  static constexpr int TAB_BYTES = EPI == 0 /*kEpiQkvRope*/ ? 64 * 16 * 16 : 0;
  static constexpr int STAGES_RAW = (232448 - 1024 - 256 - EPI_BYTES - TAB_BYTES) / STAGE_BYTES;
  // the QKV epilogue's RoPE table reads want L1, which the shared-memory
  // carve-out shrinks: that epilogue keeps at most four stages
  static constexpr int STAGES_CAP = EPI == 0 /*kEpiQkvRope*/ ? 4 : 8;
  static constexpr int STAGES = STAGES_RAW > STAGES_CAP ? STAGES_CAP : STAGES_RAW;
  static constexpr int TMEM_COLS = (2 * BN <= 128) ? 128 : (2 * BN <= 256 ? 256 : 512);
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + EPI_BYTES + TAB_BYTES + BAR_BYTES;
  static_assert(BN % 64 == 0 && BN <= 256, "UMMA N for M=128 and whole 64-column epilogue units");
  static_assert(B_BYTES % 1024 == 0, "B stage must keep 1024-byte alignment");
  static_assert(STAGES >= 3, "pipeline depth");
  static_assert((2 * STAGES + 5 + kEpiWarps) * 8 + 8 <= BAR_BYTES, "barrier area");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

__device__ __forceinline__ void record_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float row_rstd(const GemmParams &p, int row) {
  if (p.ssq_in == nullptr || row >= p.M) return 1.0f;
  return rsqrtf(p.ssq_in[row] * p.inv_dim + p.eps);
}

// ---------------------------------------------------------------- staging tile
// Byte offset of 16-byte chunk c (0..7) of row r (0..31): the 128-byte
// swizzle of TMA (tile base 1024-byte aligned), conflict-free both for one
// row per thread and for consecutive lanes on consecutive chunks of a row.
__device__ __forceinline__ int stg_off(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// Row-per-thread writes: 32 values as fp32 (chunks 0..7), or as 16-bit values
// into chunks c0..c0+3.
__device__ __forceinline__ void stg_put_f32(uint8_t *st, int r, const float (&v)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<float4 *>(st + stg_off(r, c)) =
        make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

__device__ __forceinline__ void stg_put_16(uint8_t *st, int r, int c0, const float (&v)[32],
                                           bool as_f16) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 w;
    if (as_f16)
      w = make_uint4(pack_f16x2(v[8 * c], v[8 * c + 1]), pack_f16x2(v[8 * c + 2], v[8 * c + 3]),
                     pack_f16x2(v[8 * c + 4], v[8 * c + 5]), pack_f16x2(v[8 * c + 6], v[8 * c + 7]));
    else
      w = make_uint4(pack_bf16x2(v[8 * c], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                     pack_bf16x2(v[8 * c + 4], v[8 * c + 5]), pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
    *reinterpret_cast<uint4 *>(st + stg_off(r, c0 + c)) = w;
  }
}

// Row-per-thread reads of 32 values (fp32 chunks 0..7, or 16-bit chunks c0..c0+3).
__device__ __forceinline__ void stg_get_f32(const uint8_t *st, int r, float (&v)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float4 f = *reinterpret_cast<const float4 *>(st + stg_off(r, c));
    v[4 * c] = f.x; v[4 * c + 1] = f.y; v[4 * c + 2] = f.z; v[4 * c + 3] = f.w;
  }
}

__device__ __forceinline__ void stg_get_16(const uint8_t *st, int r, int c0, float (&v)[32],
                                           bool is_f16) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 u = *reinterpret_cast<const uint4 *>(st + stg_off(r, c0 + c));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = is_f16 ? unpack_f16x2(w[e]) : unpack_bf16x2(w[e]);
      v[8 * c + 2 * e] = f.x;
      v[8 * c + 2 * e + 1] = f.y;
    }
  }
}

// Cooperative copies between the staging tile (chunks c0..c0+NC-1 of each row)
// and NC*16 contiguous bytes per row in global memory; row rr's address is
// g + row_off(rr) bytes.  Rows >= rows_valid are skipped.  NC is 4 or 8.
// (Used where a TMA box does not fit: rows of a warp crossing a sequence,
// decode-sized problems, fp32 data.)
template <int NC, typename RowOff>
__device__ __forceinline__ void stg_to_global(const uint8_t *st, int c0, uint8_t *g, RowOff row_off,
                                              int rows_valid, int lane) {
  constexpr int RPI = 32 / NC;                    // rows per iteration
#pragma unroll
  for (int k = 0; k < 32 / RPI; ++k) {
    const int rr = k * RPI + lane / NC, c = lane % NC;
    const long long off = row_off(rr);            // evaluated by every lane (may shuffle)
    if (rr < rows_valid)
      *reinterpret_cast<uint4 *>(g + off + c * 16) =
          *reinterpret_cast<const uint4 *>(st + stg_off(rr, c0 + c));
  }
}

// Asynchronous (cp.async) copy of NC*16 bytes per row from global memory into
// chunks 0..NC-1 of the staging tile; missing rows are zero-filled.  The
// caller commits and waits.
template <int NC>
__device__ __forceinline__ void global_to_stg_async(uint8_t *st, const uint8_t *g, long long ld_bytes,
                                                    int rows_valid, int lane) {
  constexpr int RPI = 32 / NC;
#pragma unroll
  for (int k = 0; k < 32 / RPI; ++k) {
    const int rr = k * RPI + lane / NC, c = lane % NC;
    const bool ok = rr < rows_valid;
    cp_async16(st + stg_off(rr, c), ok ? g + rr * ld_bytes + c * 16 : g, ok);
  }
}

// Before a staging tile is rewritten: lane 0 waits until at most N of its
// earlier bulk groups may still be reading shared memory, then the warp
// proceeds together (this also orders the lanes' earlier reads of the tile).
template <int N>
__device__ __forceinline__ void stg_reuse_wait(int lane) {
  if (lane == 0) bulk_wait_group_read<N>();
  __syncwarp();
}

// Every lane's writes of the staged box are made visible to the async proxy;
// lane 0 issues its TMA store (none for a warp without rows) and commits one
// bulk group.
__device__ __forceinline__ void stg_tma_store(const CUtensorMap *map, const uint8_t *tile, int x,
                                              int y, int lane, int rows_valid) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (rows_valid > 0) tma_store_2d(map, tile, x, y);
    bulk_commit_group();
  }
}

// An empty bulk group, so that every use of an alternating staging tile is
// one group whatever path wrote it out.
__device__ __forceinline__ void stg_empty_group(int lane) {
  if (lane == 0) bulk_commit_group();
}

// ---------------------------------------------------------------- epilogues
// Every tcgen05.ld is executed by all lanes (it is warp-collective); only
// global accesses depend on the row bound.
struct EpiCtx {
  uint32_t taddr;     // TMEM address of (row0, column 0 of the tile)
  int row0;           // the warp's first tile row
  int rows_valid;     // how many of its 32 rows exist
  int lane, n0, n_blk, split;
  uint8_t *st;        // the warp's staging tiles
  const EpiMaps *maps;
  uint64_t *rbar;     // the warp's residual-load barrier and its next parity
  uint32_t rphase;
  uint32_t seq;       // staging uses so far (selects the alternating tile)
  float rs;           // the lane's row scale rstd, read before the accumulator is waited for
  const float4 *tab;  // fine RoPE entries in shared memory (QKV, hd 64), else nullptr
};

// logits = rstd * D; units of 64 columns (one full 128-byte row segment).
template <int BN>
__device__ __forceinline__ void epi_scale(const GemmParams &p, EpiCtx &e) {
  const float rs = e.rs;
  const bool tma = p.epi_tma & kTmaOut;
  const long long ld = p.ldo * 2;
  uint8_t *gbase = p.out ? static_cast<uint8_t *>(p.out) + ((long long)e.row0 * p.ldo) * 2 : nullptr;
  unsigned long long best = 0;                    // this row's largest rounded output (argmax_pack)
#pragma unroll 1
  for (int c = e.split * 64; c < BN; c += 64 * kSplit) {
    if (e.n0 + c >= p.N) break;                   // uniform across the warp
    uint32_t r0[32], r1[32];
    tmem_ld32(e.taddr + c, r0);
    tmem_ld32(e.taddr + c + 32, r1);
    tmem_ld_wait();
    float v[32];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(h ? r1[k] : r0[k]) * rs;
      if (p.argmax) {
        // the same bf16 rounding as the stored logits
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const uint16_t bits = __bfloat16_as_ushort(__float2bfloat16_rn(v[k]));
          best = max(best, argmax_pack(bf16_order_key(bits), static_cast<uint32_t>(e.n0 + c + 32 * h + k)));
        }
      }
      if (p.out) {
        if (h == 0) stg_reuse_wait<0>(e.lane);
        stg_put_16(e.st, e.lane, 4 * h, v, p.out_is_f16);
      }
    }
    if (!p.out) continue;                         // uniform: only the row maxima are wanted
    if (tma) {
      stg_tma_store(&e.maps->out, e.st, e.n0 + c, e.row0, e.lane, e.rows_valid);
    } else {
      __syncwarp();
      stg_to_global<8>(e.st, 0, gbase + (long long)(e.n0 + c) * 2,
                       [&](int rr) { return rr * ld; }, e.rows_valid, e.lane);
    }
  }
  if (p.argmax && e.lane < e.rows_valid && best) atomicMax(p.argmax + e.row0 + e.lane, best);
}

// ---- residual: out = resid + D.
// Fast path (16-bit residual in, 16-bit result out): the warp's residual
// units of 64 columns are fetched by TMA into its staging tiles before the
// accumulator is ready, the sum is written back in place and stored by TMA.
// Row sums of squares (feeding the next RMSNorm) are taken over the rounded
// 16-bit values the next step reads.
template <int BN>
__device__ __forceinline__ int residual_units(const GemmParams &p, const EpiCtx &e) {
  int nu = 0;
  if (e.rows_valid <= 0) return 0;                // a CTA of a pair past the last row block
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int c = (e.split + kSplit * k) * 64;
    if (c < BN && e.n0 + c < p.N) ++nu;
  }
  return nu;
}

template <int BN>
__device__ __forceinline__ void residual_load_tma(const GemmParams &p, EpiCtx &e) {
  const int nu = residual_units<BN>(p, e);
  if (nu == 0) return;
  stg_reuse_wait<0>(e.lane);                      // earlier stores have read the tiles
  if (e.lane == 0) {
    mbar_arrive_expect_tx(e.rbar, nu * kStgBytes);
    for (int k = 0; k < nu; ++k)
      tma_load_2d(e.st + k * kStgBytes, &e.maps->resid, e.rbar, e.n0 + (e.split + kSplit * k) * 64,
                  e.row0);
  }
}

template <int BN>
__device__ __forceinline__ bool epi_residual_tma(const GemmParams &p, EpiCtx &e,
                                                 volatile int *abort_flag) {
  const int nu = residual_units<BN>(p, e);
  if (nu == 0) return true;
  const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(e.rbar, e.rphase, abort_flag));
  if (!ok) {
    mbar_wait_drain(e.rbar, e.rphase);            // the residual boxes land before the CTA exits
    e.rphase ^= 1u;
    return false;
  }
  e.rphase ^= 1u;
  const bool resid_f16 = p.resid_f16 != nullptr;
  float part = 0.f;
#pragma unroll 1
  for (int k = 0; k < nu; ++k) {
    const int c = (e.split + kSplit * k) * 64;
    uint8_t *tile = e.st + k * kStgBytes;
    uint32_t r[32];
    float v[32];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      tmem_ld32(e.taddr + c + 32 * h, r);
      tmem_ld_wait();
      stg_get_16(tile, e.lane, 4 * h, v, resid_f16);
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const float x = v[q] + __uint_as_float(r[q]);
        const float rx = p.out_is_f16 ? __half2float(__float2half_rn(x))
                                      : __bfloat162float(__float2bfloat16_rn(x));
        v[q] = rx;
        part = fmaf(rx, rx, part);
      }
      stg_put_16(tile, e.lane, 4 * h, v, p.out_is_f16);   // own row only: in place
    }
    stg_tma_store(&e.maps->out, tile, e.n0 + c, e.row0, e.lane, e.rows_valid);
  }
  if (e.lane < e.rows_valid && p.ssq_out) atomicAdd(p.ssq_out + e.row0 + e.lane, part);
  // the sum of squares of the rounded outputs is finite iff none overflowed
  if (e.lane < e.rows_valid && !isfinite(part)) set_status(p.status, kDevRange);
  return true;
}

// General path (fp32 residual and/or fp32 output; 32-column units; cp.async
// and per-lane stores): tile 0 holds the residual unit, tile 1 the 16-bit result.
template <int BN>
__device__ __forceinline__ void residual_prefetch_lane(const GemmParams &p, const EpiCtx &e, int c,
                                                       uint8_t *buf) {
  const long long off = (long long)e.row0 * p.ldo + e.n0 + c;
  if (p.resid_f32)
    global_to_stg_async<8>(buf, reinterpret_cast<const uint8_t *>(p.resid_f32 + off), p.ldo * 4,
                           e.rows_valid, e.lane);
  else
    global_to_stg_async<4>(buf,
                           p.resid_f16 ? reinterpret_cast<const uint8_t *>(p.resid_f16 + off)
                                       : reinterpret_cast<const uint8_t *>(p.resid + off),
                           p.ldo * 2, e.rows_valid, e.lane);
  cp_async_commit();
}

template <int BN>
__device__ __forceinline__ void epi_residual_lane(const GemmParams &p, EpiCtx &e) {
  const bool row_ok = e.lane < e.rows_valid;
  float part = 0.f;
  bool big = false;                               // an fp32 output whose f16 copy overflows
  uint8_t *buf = e.st, *st16 = e.st + kStgBytes;
  const long long row0_off = (long long)e.row0 * p.ldo;
  // unit 0's residual was prefetched by the caller into buf
#pragma unroll 1
  for (int c = e.split * 32; c < BN; c += 32 * kSplit) {
    const int col = e.n0 + c;
    if (col >= p.N) break;                        // uniform across the warp
    cp_async_wait<0>();
    uint32_t r[32];
    tmem_ld32(e.taddr + c, r);
    tmem_ld_wait();
    __syncwarp();                                 // every lane's copies into buf landed
    float v[32];
    if (p.resid_f32) stg_get_f32(buf, e.lane, v);
    else stg_get_16(buf, e.lane, 0, v, p.resid_f16 != nullptr);
#pragma unroll
    for (int q = 0; q < 32; ++q) v[q] += __uint_as_float(r[q]);
    if (p.out_f32) {
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        part = fmaf(v[q], v[q], part);
        big |= p.out && p.out_is_f16 && !(fabsf(v[q]) < kF16Overflow);
      }
      stg_put_f32(buf, e.lane, v);                // own row only: no hazard with other lanes
    } else {
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const float rv = p.out_is_f16 ? __half2float(__float2half_rn(v[q]))
                                      : __bfloat162float(__float2bfloat16_rn(v[q]));
        part = fmaf(rv, rv, part);
      }
    }
    if (p.out) stg_put_16(st16, e.lane, 0, v, p.out_is_f16);
    __syncwarp();
    if (p.out_f32)
      stg_to_global<8>(buf, 0, reinterpret_cast<uint8_t *>(p.out_f32 + row0_off + col),
                       [&](int rr) { return rr * p.ldo * 4; }, e.rows_valid, e.lane);
    if (p.out)
      stg_to_global<4>(st16, 0, static_cast<uint8_t *>(p.out) + (row0_off + col) * 2,
                       [&](int rr) { return rr * p.ldo * 2; }, e.rows_valid, e.lane);
    __syncwarp();                                 // copy-out has read buf and st16
    const int cn = c + 32 * kSplit;
    if (cn < BN && e.n0 + cn < p.N) residual_prefetch_lane<BN>(p, e, cn, buf);
  }
  cp_async_wait<0>();
  if (row_ok && p.ssq_out) atomicAdd(p.ssq_out + e.row0 + e.lane, part);
  if (row_ok && (big || !isfinite(part))) set_status(p.status, kDevRange);
}

// Gate and up columns come in groups of 64 + 64 per 128 accumulator columns;
// a unit is one group: 64 outputs written as one 128-byte row segment.
template <int BN>
__device__ __forceinline__ void epi_swiglu(const GemmParams &p, EpiCtx &e) {
  const float rs = e.rs;
  const int I = p.N / 2;
  const bool tma = p.epi_tma & kTmaOut;
  uint8_t *gbase = static_cast<uint8_t *>(p.out) + (long long)e.row0 * p.ldo * 2;
#pragma unroll 1
  for (int grp = e.split; grp < BN / 128; grp += kSplit) {
    const int out_col = (e.n0 / 128 + grp) * 64;
    if (out_col >= I) break;                      // uniform across the warp
    stg_reuse_wait<0>(e.lane);
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      uint32_t g[32], up[32];
      tmem_ld32(e.taddr + grp * 128 + h * 32, g);
      tmem_ld32(e.taddr + grp * 128 + 64 + h * 32, up);
      tmem_ld_wait();
      float v[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float gv = __uint_as_float(g[k]) * rs;
        const float uv = __uint_as_float(up[k]) * rs;
        v[k] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;   // SiLU(g) * u
      }
      stg_put_16(e.st, e.lane, 4 * h, v, p.out_is_f16);
    }
    if (tma) {
      stg_tma_store(&e.maps->out, e.st, out_col, e.row0, e.lane, e.rows_valid);
    } else {
      __syncwarp();
      stg_to_global<8>(e.st, 0, gbase + (long long)out_col * 2,
                       [&](int rr) { return rr * p.ldo * 2; }, e.rows_valid, e.lane);
    }
  }
  const bool row_ok = e.lane < e.rows_valid;
  if (e.n_blk == 0 && e.split == 0 && row_ok && p.ssq_zero) p.ssq_zero[e.row0 + e.lane] = 0.f;
}

// Units of 64 accumulator columns of one head: for a q or k head the 32
// rotation pairs (i, i + hd/2), i in [i0, i0 + 32); for a v head 64
// consecutive columns.  Output rows of [B, heads, T, hd] are addressed per
// row.  When the warp's 32 rows are 32 tokens of one sequence (and hd = 64) a
// head's 32 x 64 block is one TMA box: q and k rows go out through the
// swizzled staging tile, V^T through a [64 dims][32 tokens] tile.  Otherwise
// (a warp crossing a sequence, decode) each lane computes its own row's
// destination and the copying lanes fetch it with a shuffle.
// cos/sin come from a two-level table (fine: angle b*f_i; coarse: angle
// 64*a*f_i; pos = 64a + b) combined by the angle-sum identities: the fine
// part stays in L1, and consecutive rows (positions) read consecutive entries.
template <int BN, int HD>
__device__ __forceinline__ void epi_qkv_rope(const GemmParams &p, EpiCtx &e) {
  const int row = e.row0 + e.lane;
  const bool row_ok = e.lane < e.rows_valid;
  const float rs = e.rs;
  const int rr_ = row_ok ? row : min(e.row0, p.M - 1);   // rows past M: any valid index
  const int b = rr_ / p.T, t = rr_ - b * p.T;
  int pos = t - (p.valid_start ? p.valid_start[b] : 0);
  if (p.pos_add) {
    const int pa = p.pos_add[b];
    pos += pa < 0 ? 0 : (pa > p.pos_limit ? p.pos_limit : pa);
  }
  pos = pos < 0 ? 0 : (pos >= p.max_pos ? p.max_pos - 1 : pos);
  // entry (j, pos & 63) of the fine part and (j, pos >> 6) of the coarse part
  const int n_coarse = static_cast<int>(cdiv(p.max_pos, 64));
  const bool rotary = p.rope != nullptr;          // launch-uniform; false on a NoPE block
  const float4 *tab = rotary ? reinterpret_cast<const float4 *>(p.rope) : nullptr;
  const float4 *fine4 = rotary ? (HD == 64 && e.tab ? e.tab : tab) + (pos & 63) : nullptr;
  const float4 *coarse4 = rotary ? tab + (HD / 4) * 64 + (pos >> 6) : nullptr;
  // element offsets of (b, head 0, t, 0) in [B, H, T, hd] and [B, KV, T, hd]
  const long long q_row = ((long long)b * p.H * p.T + t) * HD;
  const long long kv_row = ((long long)b * p.KV * p.T + t) * HD;
  const long long head_stride = (long long)p.T * HD;
  const int n_heads_total = p.H + 2 * p.KV;
  constexpr int kUnitsPerHead = HD / 64;
  // whole-warp TMA boxes: 32 existing rows that are tokens t0..t0+31 of one sequence
  const int wb = min(e.row0, p.M - 1) / p.T, wt0 = min(e.row0, p.M - 1) - wb * p.T;
  const bool warp_box = HD == 64 && (p.epi_tma & kTmaQkv) && e.rows_valid == 32 && wt0 + 31 < p.T;
#pragma unroll 1
  for (int u = e.split; u < BN / 64; u += kSplit) {
    const int hh = u / kUnitsPerHead, j = u - hh * kUnitsPerHead;
    const int gh = e.n0 / HD + hh;                // global head index in [q | k | v]
    if (gh >= n_heads_total) break;               // uniform across the warp
    const uint32_t tcol = e.taddr + hh * HD;
    const bool is_q = gh < p.H, is_k = !is_q && gh < p.H + p.KV;
    const int hsub = is_q ? gh : (is_k ? gh - p.H : gh - p.H - p.KV);
    const long long my_row = (is_q ? q_row : kv_row) + hsub * head_stride;
    f16 *dst = is_q ? p.q : (is_k ? p.k : p.v);
    bf16 *dst_bf = is_q ? nullptr : (is_k ? p.k_bf : p.v_bf);
    auto row_off = [&](int rr) { return __shfl_sync(0xffffffffu, my_row, rr) * 2; };
    float y1[32], y2[32];
    int seg1, seg2;                               // element offsets of the two 32-wide segments
    if (is_q || is_k) {
      const int i0 = j * 32;
      uint32_t x1[32], x2[32];
      tmem_ld32(tcol + i0, x1);
      tmem_ld32(tcol + HD / 2 + i0, x2);
      tmem_ld_wait();
      if (rotary) {
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const int jj = (i0 + k) >> 1;           // pairs i0+k and i0+k+1
          const float4 f = fine4[jj * 64];        // (cos, sin) of b*f
          const float4 g = coarse4[jj * n_coarse];  // (cos, sin) of 64*a*f
          const float c0 = g.x * f.x - g.y * f.y, s0 = g.y * f.x + g.x * f.y;
          const float c1 = g.z * f.z - g.w * f.w, s1 = g.w * f.z + g.z * f.w;
          const float a0 = __uint_as_float(x1[k]) * rs, b0 = __uint_as_float(x2[k]) * rs;
          const float a1 = __uint_as_float(x1[k + 1]) * rs, b1 = __uint_as_float(x2[k + 1]) * rs;
          y1[k] = a0 * c0 - b0 * s0;
          y2[k] = a0 * s0 + b0 * c0;
          y1[k + 1] = a1 * c1 - b1 * s1;
          y2[k + 1] = a1 * s1 + b1 * c1;
        }
      } else {                                    // a NoPE block: the scaled projections
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          y1[k] = __uint_as_float(x1[k]) * rs;
          y2[k] = __uint_as_float(x2[k]) * rs;
        }
      }
      seg1 = i0;
      seg2 = HD / 2 + i0;
    } else {
      const int i0 = j * 64;
      uint32_t x1[32], x2[32];
      tmem_ld32(tcol + i0, x1);
      tmem_ld32(tcol + i0 + 32, x2);
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        y1[k] = __uint_as_float(x1[k]) * rs;
        y2[k] = __uint_as_float(x2[k]) * rs;
      }
      seg1 = i0;
      seg2 = i0 + 32;
    }
    if (!is_q && !is_k && p.v_t) {
      // V transposed ([B, KV, hd, T_pad]), keys contiguous
      uint8_t *tile = e.st + (e.seq++ & 1u) * kStgBytes;
      stg_reuse_wait<1>(e.lane);
      if (warp_box && (wt0 & 7) == 0) {
        // [64 dims][32 tokens] tile, one TMA box at (token t0, row (b, kv head, dim 0))
        __half *tt = reinterpret_cast<__half *>(tile);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          tt[k * 32 + e.lane] = __float2half_rn(y1[k]);
          tt[(32 + k) * 32 + e.lane] = __float2half_rn(y2[k]);
        }
        stg_tma_store(&e.maps->vt, tile, wt0, (wb * p.KV + hsub) * HD, e.lane, e.rows_valid);
      } else {
        // stage the 32 x 64 block, then each lane writes 8 consecutive tokens
        // of one dimension (16 bytes when the 8 rows are consecutive tokens of
        // one sequence starting at a multiple of 8, element by element otherwise)
        stg_put_16(tile, e.lane, 0, y1, true);
        stg_put_16(tile, e.lane, 4, y2, true);
        __syncwarp();
        const long long my_vt = ((long long)b * p.KV + hsub) * HD * p.T_pad + t;
        const int tg = e.lane & 3;
        long long vrow[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) vrow[i] = __shfl_sync(0xffffffffu, my_vt, 8 * tg + i);
        const bool fast = (8 * tg + 7 < e.rows_valid) && (vrow[7] == vrow[0] + 7) && ((vrow[0] & 7) == 0);
#pragma unroll 1
        for (int it = 0; it < 8; ++it) {
          const int dd = it * 8 + (e.lane >> 2);  // dimension within this 64-wide unit
          uint16_t val[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            val[i] = *reinterpret_cast<const uint16_t *>(tile + stg_off(8 * tg + i, dd >> 3) + (dd & 7) * 2);
          const long long dim_off = (long long)(seg1 + dd) * p.T_pad;
          uint16_t *vt = reinterpret_cast<uint16_t *>(p.v_t);
          if (fast) {
            uint4 w;
            w.x = val[0] | (uint32_t(val[1]) << 16);
            w.y = val[2] | (uint32_t(val[3]) << 16);
            w.z = val[4] | (uint32_t(val[5]) << 16);
            w.w = val[6] | (uint32_t(val[7]) << 16);
            *reinterpret_cast<uint4 *>(vt + vrow[0] + dim_off) = w;
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (8 * tg + i < e.rows_valid) vt[vrow[i] + dim_off] = val[i];
          }
        }
        stg_empty_group(e.lane);
      }
      dst = nullptr;                              // the row-layout f16 copy is not needed
    }
    const bool contiguous = seg2 == seg1 + 32;    // both segments form one 128-byte row piece
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      void *base = pass == 0 ? static_cast<void *>(dst) : static_cast<void *>(dst_bf);
      if (base == nullptr) continue;              // uniform across the warp
      uint8_t *tile = e.st + (e.seq++ & 1u) * kStgBytes;
      stg_reuse_wait<1>(e.lane);
      stg_put_16(tile, e.lane, 0, y1, pass == 0);
      stg_put_16(tile, e.lane, 4, y2, pass == 0);
      if (pass == 0 && warp_box && (is_q || is_k)) {
        const int y = ((wb * (is_q ? p.H : p.KV)) + hsub) * p.T + wt0;
        stg_tma_store(is_q ? &e.maps->q : &e.maps->k, tile, 0, y, e.lane, e.rows_valid);
        continue;
      }
      __syncwarp();
      uint8_t *g = static_cast<uint8_t *>(base);
      if (contiguous) {
        stg_to_global<8>(tile, 0, g + seg1 * 2, row_off, e.rows_valid, e.lane);
      } else {
        stg_to_global<4>(tile, 0, g + seg1 * 2, row_off, e.rows_valid, e.lane);
        stg_to_global<4>(tile, 4, g + seg2 * 2, row_off, e.rows_valid, e.lane);
      }
      stg_empty_group(e.lane);
    }
  }
  if (e.n_blk == 0 && e.split == 0 && row_ok && p.ssq_zero) p.ssq_zero[row] = 0.f;
}

// ---------------------------------------------------------------- kernel
template <int BN, int EPI, int HD, int PAIR>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ EpiMaps maps, const GemmParams p) {
  using C = GemmCfg<BN, EPI, PAIR>;
  static_assert(PAIR == 1 || PAIR == 2, "one CTA or a CTA pair");
  static_assert((BN / PAIR) % 8 == 0, "B share must be whole 8-row swizzle atoms");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + C::STAGES * C::A_BYTES;
  uint8_t *sEpi = sB + C::STAGES * C::B_BYTES;
  float4 *sTab = reinterpret_cast<float4 *>(sEpi + C::EPI_BYTES);   // [16][64] fine RoPE entries (QKV)
  uint64_t *bars = reinterpret_cast<uint64_t *>(sEpi + C::EPI_BYTES + C::TAB_BYTES);
  uint64_t *full = bars;
  uint64_t *empty = bars + C::STAGES;
  uint64_t *tfull = bars + 2 * C::STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint64_t *rbar = drain + 1;                       // one per epilogue warp (residual loads)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(rbar + kEpiWarps);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_n = static_cast<int>(cdiv(p.N, BN));
  // a "tile" below is PAIR vertically adjacent 128 x BN tiles, one per CTA
  const int num_mg = static_cast<int>(cdiv(cdiv(p.M, C::BM), PAIR));
  const int num_tiles = num_mg * num_n;
  // tile order: with raster_m, concurrently running CTAs share one B tile (and
  // walk all of A, which then stays in L2) - for B larger than A, e.g. the
  // vocabulary projection; otherwise they share A and walk B
  const int num_kb = static_cast<int>(cdiv(p.K, C::BK));
  const int rank = PAIR > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  // tile -> (row group, column block).  Without raster_m the column block is
  // rotated by the row group, so that a CTA striding through the tiles by the
  // grid size meets every column block even when the grid is a multiple of
  // their number (column blocks can differ in cost: the QKV epilogue rotates
  // q and k heads but not v heads).
  auto decode_tile = [&](int tile, int &m_grp, int &n_blk) {
    m_grp = p.raster_m ? tile % num_mg : tile / num_n;
    n_blk = p.raster_m ? tile / num_mg : (tile - m_grp * num_n + m_grp) % num_n;
  };
  const int first_tile = blockIdx.x / PAIR, tile_step = gridDim.x / PAIR;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], PAIR * kEpiWarps);   // one arrival per epilogue warp (of both CTAs)
    }
    mbar_init(drain, 1);
    for (int w = 0; w < kEpiWarps; ++w) mbar_init(&rbar[w], 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    if constexpr (PAIR == 1) {
      tmem_alloc(tmem_slot, C::TMEM_COLS);
      tmem_relinquish();
    } else {
      tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
      tmem_relinquish_pair();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if constexpr (PAIR > 1) cluster_sync_all();     // the peer's barriers exist before any use
  const uint32_t tmem_base = *tmem_slot;
  // cluster addresses of the even CTA's full[0] and tempty[0] (pairs only)
  const uint32_t full0_leader = PAIR > 1 ? mapa_shared(smem_u32(full), 0) : 0u;
  const uint32_t tempty0_leader = PAIR > 1 ? mapa_shared(smem_u32(tempty), 0) : 0u;

  if (threadIdx.x == 0) griddep_launch_dependents();
  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      uint32_t stage = 0, phase = 0;
      long long issued = 0;
      bool ok = true;
      auto load_b = [&](uint32_t st, int kb, int n_blk) {
        if constexpr (PAIR == 1)
          tma_load_2d(sB + st * C::B_BYTES, &tmB, &full[st], kb * C::BK, n_blk * BN);
        else
          tma_load_2d_pair(sB + st * C::B_BYTES, &tmB, full0_leader + 8u * st, kb * C::BK,
                           n_blk * BN + rank * (BN / PAIR));
      };
      auto arm = [&](uint32_t st) {
        // with a pair both CTAs' boxes are counted on the even CTA's barrier
        if constexpr (PAIR == 1) mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
        else if (rank == 0) mbar_arrive_expect_tx(&full[st], 2 * C::STAGE_BYTES);
      };
      // The weights (B) do not depend on the preceding kernel: the first
      // stages' B boxes are requested before waiting for it, A (activations)
      // after.
      int pre = 0;
      if (first_tile < num_tiles) {
        int m_grp, n_blk;
        decode_tile(first_tile, m_grp, n_blk);
        pre = num_kb < C::STAGES ? num_kb : C::STAGES;
        for (int kb = 0; kb < pre; ++kb) {
          arm(kb);
          load_b(kb, kb, n_blk);
        }
      }
      // with row-block flags only the rows a tile reads must be complete;
      // otherwise the whole preceding kernel
      if (!p.done_in) griddep_wait();
      for (int tile = first_tile; tile < num_tiles && ok; tile += tile_step) {
        int m_grp, n_blk;
        decode_tile(tile, m_grp, n_blk);
        const int m_blk = m_grp * PAIR + rank;
        // (a pair's second row block may lie past M: no rows, no flag)
        if (p.done_in && m_blk * C::BM < p.M) {
          if (!flag_wait_geq(p.done_in + m_blk, p.done_need, abort_flag, p.status)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();             // the A rows are read by TMA
        }
        for (int kb = 0; kb < num_kb; ++kb) {
          const bool preloaded = issued < pre;     // stage armed and its B requested above
          if (!preloaded && !mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          if (!preloaded) arm(stage);
          if constexpr (PAIR == 1)
            tma_load_2d(sA + stage * C::A_BYTES, &tmA, &full[stage], kb * C::BK, m_blk * C::BM);
          else
            tma_load_2d_pair(sA + stage * C::A_BYTES, &tmA, full0_leader + 8u * stage, kb * C::BK,
                             m_blk * C::BM);
          if (!preloaded) load_b(stage, kb, n_blk);
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
        for (long long j = first; j < issued; ++j) {
          if (!mbar_wait_drain(&full[j % C::STAGES], (uint32_t)((j / C::STAGES) & 1)))
            record_status(p.status, kDevTimeoutDrain);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------ MMA issuer (the even CTA of a pair)
      constexpr uint32_t kIdesc = idesc_f16_f32(C::BM * PAIR, BN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, any = false;
      for (int tile = first_tile; tile < num_tiles && ok; tile += tile_step) {
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
            if constexpr (PAIR == 1)
              umma_f16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, kIdesc, (kb | k) != 0);
            else
              umma_f16_pair(d_tmem, a_desc + 2 * k, b_desc + 2 * k, kIdesc, (kb | k) != 0);
          }
          any = true;
          if constexpr (PAIR == 1) umma_commit(&empty[stage]);
          else umma_commit_pair(&empty[stage], 0x3);     // frees the stage in both CTAs
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if constexpr (PAIR == 1) umma_commit(&tfull[acc]);
        else umma_commit_pair(&tfull[acc], 0x3);         // both CTAs' accumulators are ready
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok) {
        record_status(p.status, kDevTimeoutMma);
        *abort_flag = 1;
        if (any) {
          // wait (bounded) for the MMAs already issued before TMEM is freed
          if constexpr (PAIR == 1) umma_commit(drain);
          else umma_commit_pair(drain, 0x1);
          if (!mbar_wait_drain(drain, 0)) record_status(p.status, kDevTimeoutDrain);
        }
      }
    }
  } else {
    // -------------------------------------------------- epilogue (warps 2 .. 1+kEpiWarps)
    // reads and writes activations: with row-block flags each tile waits for
    // its own rows below (the buffers it writes are not read by the preceding
    // kernel); otherwise the whole preceding kernel
    if (!p.done_in) griddep_wait();
    const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
    EpiCtx e;
    e.lane = lane;
    e.split = (warp - 2) >> 2;                    // which share of the tile's columns
    e.st = sEpi + (warp - 2) * EpiStage<EPI>::kPerWarp;
    e.maps = &maps;
    e.rbar = &rbar[warp - 2];
    e.rphase = 0;
    e.seq = 0;
    e.tab = nullptr;
    if constexpr (EPI == kEpiQkvRope && HD == 64) {
      // the table is an input of the step; every epilogue warp takes a share
      // (no table on a NoPE block)
      if (p.rope) {
        const float4 *src = reinterpret_cast<const float4 *>(p.rope);
        for (int i = static_cast<int>(threadIdx.x) - 64; i < 16 * 64; i += kEpiWarps * 32) sTab[i] = src[i];
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");   // the epilogue warps only
        e.tab = sTab;
      }
    }
    const bool resid_tma = EPI == kEpiResidual && (p.epi_tma & kTmaResid);
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = first_tile; tile < num_tiles; tile += tile_step) {
      int m_grp, n_blk;
      decode_tile(tile, m_grp, n_blk);
      const int m_blk = m_grp * PAIR + rank;
      e.row0 = m_blk * C::BM + quarter * 32;
      e.rows_valid = min(32, max(0, p.M - e.row0));
      e.n0 = n_blk * BN;
      e.n_blk = n_blk;
      if (p.done_in && m_blk * C::BM < p.M) {
        // the row statistics and the residual rows come from the preceding kernel
        if (!__all_sync(0xffffffffu, flag_wait_geq(p.done_in + m_blk, p.done_need, abort_flag, p.status))) {
          if (lane == 0) record_status(p.status, kDevTimeoutEpilogue);
          *abort_flag = 1;
          break;
        }
        fence_proxy_async_global();
      }
      if constexpr (EPI != kEpiResidual) e.rs = row_rstd(p, e.row0 + lane);
      if constexpr (EPI == kEpiResidual) {
        // start fetching this warp's residual while the MMAs run
        if (resid_tma) {
          residual_load_tma<BN>(p, e);
        } else {
          __syncwarp();
          if (e.n0 + e.split * 32 < p.N) residual_prefetch_lane<BN>(p, e, e.split * 32, e.st);
        }
      }
      // every lane waits; the outcome is made warp-uniform because the TMEM
      // loads below are warp-collective
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag));
      if (!ok) {
        if (lane == 0) record_status(p.status, kDevTimeoutEpilogue);
        *abort_flag = 1;
        cp_async_wait<0>();                       // no copy in flight when the CTA exits
        if (resid_tma && residual_units<BN>(p, e) > 0) mbar_wait_drain(e.rbar, e.rphase);
        break;
      }
      tc_fence_after_sync();
      e.taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
      if constexpr (EPI == kEpiScale) {
        epi_scale<BN>(p, e);
      } else if constexpr (EPI == kEpiResidual) {
        if (resid_tma) {
          if (!epi_residual_tma<BN>(p, e, abort_flag)) {
            if (lane == 0) record_status(p.status, kDevTimeoutEpilogue);
            *abort_flag = 1;
            break;
          }
        } else {
          epi_residual_lane<BN>(p, e);
        }
      } else if constexpr (EPI == kEpiSwiglu) {
        epi_swiglu<BN>(p, e);
      } else {
        epi_qkv_rope<BN, HD>(p, e);
      }
      tc_fence_before_sync();
      __syncwarp();
      // the accumulator may be overwritten once every warp's tcgen05.ld has
      // completed (its stores need not be visible): a relaxed arrival, on the
      // even CTA's barrier for a pair
      if (lane == 0)
        mbar_arrive_relaxed_cluster((PAIR == 1 ? smem_u32(tempty) : tempty0_leader) + 8u * acc);
      if (p.done_out && m_blk * C::BM < p.M) {
        // this warp's part of the tile is written (its TMA stores complete,
        // its lanes' stores and row-sum atomics fenced): one arrival on the
        // row block's flag
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          bulk_wait_group<0>();
          fence_proxy_async_global();
          flag_add_release(p.done_out + m_blk, 1);
        }
        __syncwarp();
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (lane == 0) bulk_wait_group<0>();          // this warp's TMA stores are complete
  }

  tc_fence_before_sync();
  __syncthreads();
  // neither CTA of a pair frees TMEM or leaves while the other may still use it
  if constexpr (PAIR > 1) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    if constexpr (PAIR == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
    else tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
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

bool make_tmap_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                  uint64_t row_pitch_elems, uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_pitch_elems * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_f16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                   uint64_t row_pitch_elems, uint32_t box_rows) {
  return make_tmap_2d(map, base, rows, cols, row_pitch_elems, 64, box_rows, true);
}

namespace {
struct TmapKey {
  const void *base;
  uint64_t rows, cols, pitch;
  uint32_t box_cols, box_rows;
  int swz, dev;
  bool operator==(const TmapKey &o) const {
    return base == o.base && rows == o.rows && cols == o.cols && pitch == o.pitch &&
           box_cols == o.box_cols && box_rows == o.box_rows && swz == o.swz && dev == o.dev;
  }
};
struct TmapKeyHash {
  size_t operator()(const TmapKey &k) const {
    size_t h = reinterpret_cast<uintptr_t>(k.base);
    for (uint64_t v : {k.rows, k.cols, k.pitch, (uint64_t)k.box_cols, (uint64_t)k.box_rows,
                       (uint64_t)k.swz, (uint64_t)k.dev})
      h = h * 1000003u ^ static_cast<size_t>(v);
    return h;
  }
};
std::mutex g_tmap_mu;
std::unordered_map<TmapKey, CUtensorMap, TmapKeyHash> g_tmap_cache;
constexpr size_t kTmapCacheMax = 4096;
}  // namespace

bool get_tmap_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                 uint64_t row_pitch_elems, uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  int dev = 0;
  cudaGetDevice(&dev);
  const TmapKey key{base, rows, cols, row_pitch_elems, box_cols, box_rows, swizzle128 ? 1 : 0, dev};
  {
    std::lock_guard<std::mutex> lock(g_tmap_mu);
    auto it = g_tmap_cache.find(key);
    if (it != g_tmap_cache.end()) {
      *map = it->second;
      return true;
    }
  }
  if (!make_tmap_2d(map, base, rows, cols, row_pitch_elems, box_cols, box_rows, swizzle128)) return false;
  std::lock_guard<std::mutex> lock(g_tmap_mu);
  if (g_tmap_cache.size() >= kTmapCacheMax) g_tmap_cache.clear();
  g_tmap_cache.emplace(key, *map);
  return true;
}

bool get_tmap_f16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                  uint64_t row_pitch_elems, uint32_t box_rows) {
  return get_tmap_2d(map, base, rows, cols, row_pitch_elems, 64, box_rows, true);
}

int gemm_pick_bn(int epi, int N, int hd) {
  if (N <= 0 || N % 64) return 0;
  if (epi == kEpiQkvRope) {
    if (N % hd) return 0;
    // 256 columns (four 64-wide head units, two per epilogue warp) even when
    // the last tile is ragged: the RoPE units cost about twice the MMAs of a
    // tile, so an even split between the warps matters more than the columns
    // the last tile computes in vain (for N = 960, five 192-column tiles ran
    // the SmolLM2 forward in 5.50 ms against 5.40 with four of 256)
    if (N >= 256) return 256;
    const int cands[2] = {192, 128};
    for (int c : cands)
      if (c % hd == 0 && N % c == 0) return c;
    return hd == 64 ? 128 : 256;                  // ragged last tile (whole heads)
  }
  if (epi == kEpiSwiglu) {
    if (N % 128) return 0;
    return N % 256 == 0 ? 256 : 128;
  }
  if (epi == kEpiResidual) {
    // 256 columns where they divide N and N is wide (fewer A re-reads and MMA
    // issues per flop); for N = 576 (SmolLM2) 192 divides it
    if (N >= 1024 && N % 256 == 0) return 256;
    const int cands[3] = {192, 128, 64};
    for (int c : cands)
      if (N % c == 0) return c;
    return 64;
  }
  const int cands[4] = {256, 192, 128, 64};
  for (int c : cands)
    if (N % c == 0) return c;
  return 64;
}

// CTA pairs for problems with at least kPairMinMBlocks row blocks of 128;
// single CTAs otherwise (decode-sized M).
constexpr int kPairMinMBlocks = 8;

// How many clusters of the kernel can be resident at once (cached per device).
template <auto Kern>
static int max_active_clusters(cudaLaunchConfig_t cfg, int fallback) {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fallback;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaOccupancyMaxActiveClusters(&n, Kern, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    return fallback;
  }
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <int BN, int EPI, int HD, int PAIR>
static cudaError_t launch_pair(const CUtensorMap &ta, const CUtensorMap &tb, const EpiMaps &maps,
                               const GemmParams &p, int num_sms, cudaStream_t stream) {
  using C = GemmCfg<BN, EPI, PAIR>;
  constexpr auto kern = gemm_tc_kernel<BN, EPI, HD, PAIR>;
  cudaError_t e = ensure_smem_attr<kern>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long groups = cdiv(cdiv(p.M, C::BM), PAIR) * cdiv(p.N, BN);
  cudaLaunchAttribute attr[2];
  int nattr = 0;
  if (p.pdl) {
    attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[nattr].val.programmaticStreamSerializationAllowed = 1;
    ++nattr;
  }
  if constexpr (PAIR == 1) {
    const int grid = static_cast<int>(groups < num_sms ? groups : num_sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, maps, p);
  } else {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = PAIR;
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms / PAIR * PAIR));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    const long long pairs_max = max_active_clusters<kern>(cfg, num_sms / PAIR);
    const long long pairs = groups < pairs_max ? groups : pairs_max;
    cfg.gridDim = dim3(static_cast<unsigned>(pairs * PAIR));
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, maps, p);
  }
}

static int gemm_pair(const GemmParams &p) { return cdiv(p.M, 128) >= kPairMinMBlocks ? 2 : 1; }

template <int BN, int EPI, int HD>
static cudaError_t launch_impl(const CUtensorMap &ta, const CUtensorMap &tb, const EpiMaps &maps,
                               const GemmParams &p, int num_sms, cudaStream_t stream) {
  if (gemm_pair(p) == 1) return launch_pair<BN, EPI, HD, 1>(ta, tb, maps, p, num_sms, stream);
  return launch_pair<BN, EPI, HD, 2>(ta, tb, maps, p, num_sms, stream);
}

cudaError_t launch_gemm(int epi, int bn, const void *A, const void *B, const GemmParams &p_in,
                        int num_sms, cudaStream_t stream) {
  GemmParams p = p_in;
  p.raster_m = (long long)p.N > (long long)p.M ? 1 : 0;   // keep the larger operand's tiles hot
  CUtensorMap ta, tb;
  if (!get_tmap_f16(&ta, A, p.M, p.K, p.K, 128)) return cudaErrorInvalidValue;
  // each CTA of a pair loads half of the B box
  if (!get_tmap_f16(&tb, B, p.N, p.K, p.K, bn / gemm_pair(p))) return cudaErrorInvalidValue;
  // epilogue tensor maps (a map that cannot be encoded leaves its per-lane path in use)
  EpiMaps maps;
  memset(&maps, 0, sizeof(maps));
  p.epi_tma = 0;
  if ((epi == kEpiScale || epi == kEpiSwiglu) && p.out) {
    const uint64_t cols = epi == kEpiSwiglu ? p.N / 2 : p.N;
    if (get_tmap_2d(&maps.out, p.out, p.M, cols, p.ldo, 64, 32, true)) p.epi_tma |= kTmaOut;
  }
  if (epi == kEpiResidual && p.out && !p.out_f32 && !p.resid_f32) {
    const void *r16 = p.resid_f16 ? static_cast<const void *>(p.resid_f16) : static_cast<const void *>(p.resid);
    if (r16 && get_tmap_2d(&maps.out, p.out, p.M, p.N, p.ldo, 64, 32, true) &&
        get_tmap_2d(&maps.resid, r16, p.M, p.N, p.ldo, 64, 32, true))
      p.epi_tma |= kTmaOut | kTmaResid;
  }
  if (epi == kEpiQkvRope && p.hd == 64 && p.T >= 32 && p.q && p.k && p.v_t && p.M % p.T == 0) {
    const uint64_t Bq = (uint64_t)(p.M / p.T);
    if (get_tmap_2d(&maps.q, p.q, Bq * p.H * p.T, 64, 64, 64, 32, true) &&
        get_tmap_2d(&maps.k, p.k, Bq * p.KV * p.T, 64, 64, 64, 32, true) &&
        get_tmap_2d(&maps.vt, p.v_t, Bq * p.KV * 64, p.T, p.T_pad, 32, 64, false))
      p.epi_tma |= kTmaQkv;
  }
  switch (epi) {
    case kEpiScale:
      if (bn == 256) return launch_impl<256, kEpiScale, 64>(ta, tb, maps, p, num_sms, stream);
      if (bn == 192) return launch_impl<192, kEpiScale, 64>(ta, tb, maps, p, num_sms, stream);
      if (bn == 128) return launch_impl<128, kEpiScale, 64>(ta, tb, maps, p, num_sms, stream);
      if (bn == 64) return launch_impl<64, kEpiScale, 64>(ta, tb, maps, p, num_sms, stream);
      break;
    case kEpiResidual:
      if (bn == 256) return launch_impl<256, kEpiResidual, 64>(ta, tb, maps, p, num_sms, stream);
      if (bn == 192) return launch_impl<192, kEpiResidual, 64>(ta, tb, maps, p, num_sms, stream);
      if (bn == 128) return launch_impl<128, kEpiResidual, 64>(ta, tb, maps, p, num_sms, stream);
      if (bn == 64) return launch_impl<64, kEpiResidual, 64>(ta, tb, maps, p, num_sms, stream);
      break;
    case kEpiSwiglu:
      if (bn == 256) return launch_impl<256, kEpiSwiglu, 64>(ta, tb, maps, p, num_sms, stream);
      if (bn == 128) return launch_impl<128, kEpiSwiglu, 64>(ta, tb, maps, p, num_sms, stream);
      break;
    case kEpiQkvRope:
      if (p.hd == 64) {
        if (bn == 256) return launch_impl<256, kEpiQkvRope, 64>(ta, tb, maps, p, num_sms, stream);
        if (bn == 192) return launch_impl<192, kEpiQkvRope, 64>(ta, tb, maps, p, num_sms, stream);
        if (bn == 128) return launch_impl<128, kEpiQkvRope, 64>(ta, tb, maps, p, num_sms, stream);
        if (bn == 64) return launch_impl<64, kEpiQkvRope, 64>(ta, tb, maps, p, num_sms, stream);
      } else if (p.hd == 128) {
        if (bn == 256) return launch_impl<256, kEpiQkvRope, 128>(ta, tb, maps, p, num_sms, stream);
        if (bn == 128) return launch_impl<128, kEpiQkvRope, 128>(ta, tb, maps, p, num_sms, stream);
      }
      break;
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace smol
