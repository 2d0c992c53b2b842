// common.cuh - declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "smol.h"

namespace smol {

typedef __nv_bfloat16 bf16;
typedef __half f16;

__host__ __device__ constexpr long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

// RoPE table, two levels: a position pos = 64a + b is recovered from
// (cos, sin)(b f_i) and (cos, sin)(64 a f_i) by the angle-sum identities.
// Stored as float4 entries holding pairs i = 2j and 2j + 1:
//   fine   entry (j, b), b < 64:          index j * 64 + b
//   coarse entry (j, a), a < cdiv(max_pos, 64): index (hd/4) * 64 + j * cdiv(max_pos, 64) + a
// so that consecutive positions are consecutive entries (coalesced loads).
// rope_table_rows counts float2 rows of hd/2 entries each.
__host__ __device__ constexpr long long rope_table_rows(int max_pos) { return 64 + cdiv(max_pos, 64); }

// Per-block variants (SmolLM3): does block `layer` rotate q and k, and its
// attention window (0 = full causal).  The arrays are host arrays of the config.
inline bool layer_rotary(const smol_config *c, int layer) {
  return c->no_rope_layers == nullptr || c->no_rope_layers[layer] != 0;
}
inline int layer_window(const smol_config *c, int layer) {
  return c->sliding_window ? c->sliding_window[layer] : 0;
}

// ------------------------------------------------------------------ GEMM
// D[M, N] = A[M, K] * B[N, K]^T on tcgen05 with one of these epilogues.
enum Epilogue : int {
  kEpiQkvRope = 0,   // rstd row scale, RoPE on q/k heads, scatter to [B, heads, T, hd]
  kEpiResidual = 1,  // out = resid + D (fp32 and/or bf16), accumulates row sum(out^2)
  kEpiSwiglu = 2,    // rstd row scale, silu(gate) * up over 64-column gate/up groups
  kEpiScale = 3,     // out = rstd * D (bf16); rstd = 1 without ssq_in
};

// Operands A and B are f16 (activations are kept as f16 tensor-core operands,
// weights are converted to f16 when packed); accumulation is fp32.
struct GemmParams {
  int M, N, K;
  void *out;              // 16-bit output rows, leading dimension ldo (elements); optional
                          // for kEpiResidual when out_f32 is given
  int out_is_f16;         // element type of `out`: 1 = f16, 0 = bf16
  long long ldo;
  const bf16 *resid;      // kEpiResidual: bf16 residual rows (leading dimension ldo), or
  const f16 *resid_f16;   //   f16 residual rows, or
  const float *resid_f32; //   fp32 residual rows (exactly one of the three is set)
  float *out_f32;         // kEpiResidual: optional fp32 copy of the output rows
  const float *ssq_in;    // per-row sum of squares feeding rstd (nullptr: scale 1)
  float inv_dim;          // 1 / d for the mean of squares
  float eps;
  float *ssq_out;         // kEpiResidual: atomically accumulates sum(out^2) per row
  float *ssq_zero;        // rows of this buffer are cleared by the n-block-0 tiles
  // kEpiQkvRope
  f16 *q, *k, *v;         // f16 [B, H, T, hd], [B, KV, T, hd], [B, KV, T, hd]; k, v optional
  f16 *v_t;               // optional f16 V transposed: [B, KV, hd, T_pad] (keys contiguous)
  int T_pad;              // row pitch of v_t in elements (T rounded up to a multiple of 8)
  bf16 *k_bf, *v_bf;      // optional bf16 copies of k and v (cache entries), same layout
  int T, H, KV, hd;
  const float2 *rope;     // [rope_table_rows(max_pos)][hd/2] (cos, sin), two-level;
                          // nullptr: q and k are not rotated (a NoPE block)
  const int *valid_start; // [B] or nullptr: position t - valid_start[b]
  const int *pos_add;     // [B] or nullptr: adds clamp(pos_add[b], 0, pos_limit) (decode)
  int pos_limit;
  int max_pos;
  int *status;            // device status word
  // kEpiScale with bf16 output: per-row maximum of the rounded outputs and its
  // first column (argmax_pack), combined by atomicMax; zero before the launch.
  // `out` may be nullptr then (only the maxima are wanted).
  unsigned long long *argmax;
  int raster_m;           // set by launch_gemm: 1 = consecutive tiles walk down M (B tile reused)
  int epi_tma;            // set by launch_gemm: which epilogue tensor maps are valid
  int pdl;                // launch as a programmatic dependent of the preceding kernel
  // Row-block completion flags (one int per 128 rows of M), or nullptr: the
  // producer waits for done_in[row block] >= done_need before loading A rows
  // (instead of waiting for the whole preceding kernel); every epilogue warp
  // adds 1 to done_out[row block] once a tile's outputs are written.
  int *done_out;
  const int *done_in;
  int done_need;
};

// Raises the dynamic shared-memory limit of kernel `Kern` to `bytes`, once per
// device (the host call is not repeated on every launch).
template <auto Kern>
cudaError_t ensure_smem_attr(int bytes) {
  static std::atomic<int> done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (done[dev].load(std::memory_order_relaxed) >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev].store(bytes, std::memory_order_relaxed);
  return e;
}

// Encodes a 2-D f16 tensor map (rows x cols, row pitch in elements) with a
// box of box_rows x 64 columns and 128-byte swizzle.  Returns false on error.
bool make_tmap_f16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                    uint64_t row_pitch_elems, uint32_t box_rows);
// General 2-D map of 16-bit elements: box of box_rows x box_cols, 128-byte
// swizzle or none.
bool make_tmap_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                  uint64_t row_pitch_elems, uint32_t box_cols, uint32_t box_rows, bool swizzle128);
// The same through a small per-process cache keyed by (device, arguments):
// encoding is a host call of a few microseconds, and the same buffers recur on
// every forward.
bool get_tmap_f16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                  uint64_t row_pitch_elems, uint32_t box_rows);
bool get_tmap_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                 uint64_t row_pitch_elems, uint32_t box_cols, uint32_t box_rows, bool swizzle128);

// Chooses the N tile for an epilogue and problem; 0 if unsupported.
int gemm_pick_bn(int epi, int N, int hd);

// Launches the persistent GEMM (A: M x K, B: N x K, both K-contiguous).
cudaError_t launch_gemm(int epi, int bn, const void *A, const void *B, const GemmParams &p,
                        int num_sms, cudaStream_t stream);

// Decode-sized projections (M <= 64 rows) on narrow column units: the
// residual, SwiGLU and QKV/RoPE epilogues of launch_gemm with f16 operands
// (A: M x K, W: N x K, K-contiguous); see decode_gemm.cu for what is covered.
bool skinny_gemm_supported(int epi, const GemmParams &p);
cudaError_t launch_skinny_gemm(int epi, const void *A, const void *W, const GemmParams &p,
                               cudaStream_t stream);

// ------------------------------------------------------------------ attention
struct AttnParams {
  const f16 *q;           // [B, H, T, hd]
  const f16 *k, *v;       // k: [B, KV, Tk, hd]; v unused (nullptr)
  const f16 *v_t;         // [B, KV, hd, T_pad], required
  int T_pad;
  int *status;            // device status word (bounded waits)
  int num_sms;
  f16 *o;                 // [B, T, H * hd]
  const int *valid_start; // [B] or nullptr
  const int *seq_order;   // [B] or nullptr: the CTAs take the sequences in this order (a permutation)
  int B, T, H, KV, hd;
  float scale_log2;       // log2(e) / sqrt(hd)
  int window;             // > 0: query t sees keys j > t - window only (sliding window)
  const uint8_t *key_mask; // [B, T] or nullptr: key j of sequence b hidden where 0
  int Tk;                 // keys per sequence (k: [B, KV, Tk, hd], v_t pitch T_pad >= Tk); 0: T
  int q_off;              // key index of query 0 (queries are the last T of Tk keys); 0 with Tk = T
  int pdl;                // launch as a programmatic dependent of the preceding kernel
  unsigned long long wait_ns;   // bounded-wait limit, 0 = the default 1 s
  int *done_out;          // or nullptr: each CTA adds 1 to done_out[b * T / 128 + query tile]
                          // once its outputs are written (T a multiple of 128)
};
// tcgen05 attention: head_dim 64 or 128, any query group; needs v_t.
bool attention_tc_supported(int hd, int H, int KV);
// CTAs that write one (sequence, query tile): the kv heads times the CTAs per group.
int attention_tc_ctas_per_tile(int hd, int H, int KV);
cudaError_t launch_attention_tc(const AttnParams &p, cudaStream_t stream);

// ------------------------------------------------------------------ next-token choice
// One CTA per row of bf16 logits [B][ld]; see sample.cu.
cudaError_t launch_sample(const void *logits, long long ld, int B, int V, float temperature, int top_k,
                          float top_p, int do_sample, const float *uniform, int *next, cudaStream_t st);

// ------------------------------------------------------------------ small kernels
// A per-sequence input value (left-padding start, cache length) that the
// kernels clamp into [0, vmax]: the first kernel of a call checks it once per
// sequence (the row with index a multiple of rows_per_seq) and records a value
// outside the range in the status word.  vals == nullptr: nothing to check.
struct SeqCheck {
  const int *vals;
  int rows_per_seq;
  int vmax;
};
// The input conversions record out-of-range ids (embedding), values beyond
// the f16 range and the SeqCheck in the status word.
cudaError_t launch_embed_rows(const int *ids, const bf16 *embed, int vocab, int d, long long rows,
                              f16 *x16, float *x_f32, float *ssq, int *status, SeqCheck chk,
                              cudaStream_t stream);
cudaError_t launch_row_ssq(const bf16 *x, long long rows, int d, f16 *x16, float *ssq, int *status,
                           SeqCheck chk, cudaStream_t stream);
cudaError_t launch_row_ssq_f32(const float *x, long long rows, int d, f16 *x16, float *ssq, int *status,
                               SeqCheck chk, cudaStream_t stream);
cudaError_t launch_scale_cols_copy(const bf16 *src, const bf16 *norm_w, long long rows, int cols,
                                   f16 *dst, cudaStream_t stream);
cudaError_t launch_interleave_gate_up(const bf16 *wg, const bf16 *wu, const bf16 *norm_w, int I,
                                      int d, f16 *dst, cudaStream_t stream);
cudaError_t launch_rope_table(int max_pos, int hd, float theta, float2 *table, cudaStream_t stream);
// Appends one decode step's keys and values to the caches: cache[l, b, kv,
// cache_len[b], :] = new[l, b, kv, :], then cache_len[b] += 1; rows whose
// length is outside [0, S_max) are left as they are (two launches).
cudaError_t launch_append_kv(const bf16 *k_new, const bf16 *v_new, bf16 *k_cache, bf16 *v_cache, int *cache_len,
                             int L, int B, int KV, int S_max, int hd, cudaStream_t stream);
// One layer's cached keys/values plus the T new ones as left-padded f16 sequences of Tk
// keys (hd 64 or 128): K [B, KV, Tk, hd], V^T [B, KV, hd, Tk_pad]; vs[b] = first visible
// slot; order[] = the sequences by descending cache length (ties by index).
cudaError_t launch_gather_cache_kv(const bf16 *kc, const bf16 *vc, int S_max, const int *cache_len, int lmax,
                                   const f16 *kn, const f16 *vtn, int T_pad, int B, int KV, int T, int Tk,
                                   int Tk_pad, int hd, f16 *Kc, f16 *Vtc, int *vs, int *order,
                                   cudaStream_t stream);

}  // namespace smol
