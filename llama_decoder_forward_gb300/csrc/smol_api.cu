// smol_api.cu - C ABI entry points of libsmol: argument validation, packed
// weight and workspace layouts, and the launch sequences of the block, model
// and decode paths.  No entry point allocates, frees or synchronises (except
// smol_workspace_status, which is documented as a synchronising query).
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "decode.cuh"
#include "profile.cuh"

using namespace smol;

#define SMOL_API extern "C" __attribute__((visibility("default")))

namespace {

thread_local char g_cuda_err[256] = "";
// Bounded-wait limit passed to the attention kernel (0: its default of 1 s);
// see smol_set_wait_limit_ns.
std::atomic<unsigned long long> g_attn_wait_ns{0};
thread_local int g_launches = 0;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct PackLayout {
  size_t rope_off, rope_bytes;
  size_t layer0_off, layer_bytes;
  size_t off_qkv, off_o, off_gu, off_down;   // within one layer
  size_t embed_off, head_off;
  size_t total;
};

PackLayout pack_layout(const smol_config *c, int n_layers, int with_embed) {
  PackLayout L{};
  const size_t d = c->hidden, hd = c->head_dim, H = c->n_heads, KV = c->n_kv_heads, I = c->intermediate;
  L.rope_off = 0;
  L.rope_bytes = align_up((size_t)rope_table_rows(c->max_pos) * (hd / 2) * sizeof(float2), 1024);
  L.layer0_off = L.rope_bytes;
  size_t o = 0;
  L.off_qkv = o; o = align_up(o + (H + 2 * KV) * hd * d * 2, 1024);
  L.off_o = o;   o = align_up(o + d * H * hd * 2, 1024);
  L.off_gu = o;  o = align_up(o + 2 * I * d * 2, 1024);
  L.off_down = o; o = align_up(o + d * I * 2, 1024);
  L.layer_bytes = o;
  size_t end = L.layer0_off + (size_t)n_layers * L.layer_bytes;
  if (with_embed) {
    L.embed_off = end;
    end = align_up(end + (size_t)c->vocab * d * 2, 1024);
    L.head_off = end;
    end = align_up(end + (size_t)c->vocab * d * 2, 1024);
  }
  L.total = end;
  return L;
}

struct WsLayout {
  size_t status, x, h, q, k, v, o, a, ssq_a, ssq_b;
  size_t kc, vtc, vs;        // prefill on top of a cache only
  size_t flags;              // the model forward only: row-block completion flags
  size_t total;
};

// V is stored transposed, [B, KV, hd, T_pad], when the tcgen05 attention
// kernel is used; T_pad = T rounded up to a multiple of 8.
long long t_pad(int T) { return (T + 7) / 8 * 8; }

// Row blocks of 128 rows of M = B*T (the tile GEMMs' row tiles).
long long row_blocks(int B, int T) { return ((long long)B * T + 127) / 128; }

// `chain`: the model forward, whose kernels hand some row blocks to one
// another through completion flags.
WsLayout ws_layout(const smol_config *c, int B, int T, bool chain = false) {
  WsLayout W{};
  const long long M = (long long)B * T;
  const size_t d = c->hidden, hd = c->head_dim, H = c->n_heads, KV = c->n_kv_heads, I = c->intermediate;
  const size_t v_elems = (size_t)B * KV * hd * t_pad(T);
  size_t o = 0;
  W.status = o; o += 1024;
  W.x = o; o = align_up(o + M * d * 2, 1024);
  W.h = o; o = align_up(o + M * d * 2, 1024);
  W.q = o; o = align_up(o + M * H * hd * 2, 1024);
  W.k = o; o = align_up(o + M * KV * hd * 2, 1024);
  W.v = o; o = align_up(o + v_elems * 2, 1024);
  W.o = o; o = align_up(o + M * H * hd * 2, 1024);
  W.a = o; o = align_up(o + M * I * 2, 1024);
  W.ssq_a = o; o = align_up(o + M * 4, 1024);
  W.ssq_b = o; o = align_up(o + M * 4, 1024);
  if (chain) {
    W.flags = o; o = align_up(o + (size_t)c->n_layers * 2 * row_blocks(B, T) * 4, 1024);
  }
  W.total = o;
  return W;
}

// Cache lengths accepted by prefill on top of a cache: positions L + t stay
// below max_pos and the cached rows fit the S_max slots.
int cache_lmax(const smol_config *c, int T, int S_max) { return min(S_max, c->max_pos - T); }

// The block workspace plus one layer's left-padded keys/values over Tk = lmax + T.
WsLayout ws_layout_cache(const smol_config *c, int B, int T, int S_max) {
  WsLayout W = ws_layout(c, B, T);
  const long long Tk = (long long)cache_lmax(c, T, S_max) + T;
  const size_t KV = c->n_kv_heads, hd = c->head_dim;
  size_t o = W.total;
  W.kc = o; o = align_up(o + (size_t)B * KV * Tk * hd * 2, 1024);
  W.vtc = o; o = align_up(o + (size_t)B * KV * hd * t_pad((int)Tk) * 2, 1024);
  W.vs = o; o = align_up(o + (size_t)B * 8, 1024);   // vs[B], then the sequence order[B]
  W.total = o;
  return W;
}

int check_cfg(const smol_config *c) {
  if (!c) return SMOL_ERR_INVALID_ARG;
  if (c->hidden <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
      c->intermediate <= 0 || c->n_layers <= 0 || c->max_pos <= 0 || c->vocab < 0)
    return SMOL_ERR_INVALID_ARG;
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return SMOL_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return SMOL_ERR_UNSUPPORTED_SHAPE;
  if (c->hidden != c->n_heads * c->head_dim) return SMOL_ERR_UNSUPPORTED_SHAPE;
  if (c->n_heads % c->n_kv_heads) return SMOL_ERR_UNSUPPORTED_SHAPE;
  if (c->n_heads / c->n_kv_heads > 8) return SMOL_ERR_UNSUPPORTED_SHAPE;
  if (c->hidden % 64 || c->intermediate % 64 || c->vocab % 64) return SMOL_ERR_UNSUPPORTED_SHAPE;
  for (int l = 0; l < c->n_layers; ++l) {
    if (c->no_rope_layers && c->no_rope_layers[l] != 0 && c->no_rope_layers[l] != 1) return SMOL_ERR_INVALID_ARG;
    if (c->sliding_window && c->sliding_window[l] < 0) return SMOL_ERR_INVALID_ARG;
  }
  return SMOL_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_fail(cudaError_t e) {
  snprintf(g_cuda_err, sizeof(g_cuda_err), "CUDA error %d: %s", (int)e, cudaGetErrorString(e));
  return SMOL_ERR_CUDA;
}

// Device check (compute capability 10.3) and SM count, cached per device.
int device_sms(int *sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  static int cache[64] = {0};
  if (dev < 0 || dev >= 64) return SMOL_ERR_DEVICE;
  if (cache[dev] == 0) {
    int major = 0, minor = 0, n = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    if (major != 10 || minor != 3) {
      cache[dev] = -1;
    } else {
      cache[dev] = n;
    }
  }
  if (cache[dev] < 0) return SMOL_ERR_DEVICE;
  *sms = cache[dev];
  return SMOL_OK;
}

#define LAUNCH_K(kind, st, expr)                       \
  do {                                                 \
    prof_before((kind), (st));                         \
    cudaError_t _e = (expr);                           \
    prof_after((kind), (st));                          \
    if (_e != cudaSuccess) return cuda_fail(_e);       \
    ++g_launches;                                      \
  } while (0)
#define LAUNCH(expr) LAUNCH_K(SMOL_K_OTHER, st, expr)

struct LayerPtrs {
  const f16 *qkv, *o, *gu, *down;
};

LayerPtrs layer_ptrs(const smol_config *c, const void *packed, int layer) {
  const PackLayout L = pack_layout(c, layer + 1, 0);
  const uint8_t *base = static_cast<const uint8_t *>(packed) + L.layer0_off + (size_t)layer * L.layer_bytes;
  return LayerPtrs{reinterpret_cast<const f16 *>(base + L.off_qkv),
                   reinterpret_cast<const f16 *>(base + L.off_o),
                   reinterpret_cast<const f16 *>(base + L.off_gu),
                   reinterpret_cast<const f16 *>(base + L.off_down)};
}

// Where one block reads its input and writes its output.
struct BlockIO {
  const f16 *x16;         // f16 copy of the input: the QKV GEMM operand
  const f16 *resid_f16;   // residual input in f16 (the model's residual stream), or
  const bf16 *resid_bf;   //   in bf16, or
  const float *resid_f32; //   in fp32
  void *out16;            // 16-bit output (may alias the input) or nullptr
  int out16_is_f16;
  float *out_f32;         // fp32 output or nullptr
  bf16 *k_bf, *v_bf;      // optional bf16 copies of post-RoPE k and of v
};

// One decoder block on M = B*T rows.  ssq_a holds the per-row sum of squares
// of the input; the output's sum of squares is accumulated into ssq_a (which
// is cleared in between).  The block-internal residual h is kept in f16.
// Prefill on top of a KV cache: this layer's cache slices and where the
// gathered keys go.
struct CacheCtx {
  const bf16 *k_cache, *v_cache;   // this layer: [B, KV, S_max, hd]
  const int32_t *cache_len;        // [B] device
  int S_max, lmax;
};

// Row-block completion flags of the model forward, zeroed before its first
// kernel: per layer two arrays of row_blocks ints, written by the attention
// (read by the O projection) and by the down projection (read by the next
// layer's QKV projection or the head).  These two hand-offs follow a kernel
// whose last CTAs run well after the others; between the other kernels the
// whole-kernel wait measured faster (the flag's stores-complete wait in every
// epilogue warp cost more than the overlap gained).
struct FlagCtx {
  int *flags;
  long long mblocks;
  int *at(int layer, int stage) const { return flags + ((long long)layer * 2 + stage) * mblocks; }
};

// Arrivals per row block from a tile GEMM of N columns and tile width bn: one
// per epilogue warp (eight per CTA) and column tile.
int gemm_arrivals(int N, int bn) { return 8 * static_cast<int>((N + bn - 1) / bn); }

int run_block(const smol_config *c, const void *packed, int layer, const BlockIO &io, int B, int T,
              const int32_t *valid_start, const uint8_t *key_mask, const WsLayout &W, uint8_t *ws, int sms,
              cudaStream_t st, const CacheCtx *cc = nullptr, const FlagCtx *fc = nullptr) {
  const long long M = (long long)B * T;
  const int d = c->hidden, H = c->n_heads, KV = c->n_kv_heads, hd = c->head_dim, I = c->intermediate;
  const LayerPtrs lp = layer_ptrs(c, packed, layer);
  const PackLayout PL = pack_layout(c, 1, 0);
  int *status = reinterpret_cast<int *>(ws + W.status);
  float *ssq_a = reinterpret_cast<float *>(ws + W.ssq_a);
  float *ssq_b = reinterpret_cast<float *>(ws + W.ssq_b);
  f16 *q = reinterpret_cast<f16 *>(ws + W.q);
  f16 *k = reinterpret_cast<f16 *>(ws + W.k);
  f16 *v = reinterpret_cast<f16 *>(ws + W.v);
  f16 *o = reinterpret_cast<f16 *>(ws + W.o);
  const int bn_qkv = gemm_pick_bn(kEpiQkvRope, (H + 2 * KV) * hd, hd);
  const int bn_o = gemm_pick_bn(kEpiResidual, d, hd);
  const int bn_gu = gemm_pick_bn(kEpiSwiglu, 2 * I, hd);
  const int bn_down = bn_o;
  // the attention's per-(sequence, query tile) flags coincide with row blocks
  // of 128 rows when T is a multiple of 128
  const bool attn_flags = fc && T % 128 == 0 && !cc;
  f16 *h = reinterpret_cast<f16 *>(ws + W.h);
  f16 *a = reinterpret_cast<f16 *>(ws + W.a);

  // 1. RMSNorm1 + QKV projection + RoPE (norm weight folded into W)
  GemmParams p{};
  p.M = (int)M; p.N = (H + 2 * KV) * hd; p.K = d;
  p.ssq_in = ssq_a; p.inv_dim = 1.0f / d; p.eps = c->rms_eps; p.ssq_zero = ssq_b;
  p.q = q; p.k = k; p.k_bf = io.k_bf; p.v_bf = io.v_bf;
  p.v_t = v;
  p.T_pad = (int)t_pad(T);
  p.T = T; p.H = H; p.KV = KV; p.hd = hd;
  // a NoPE block passes no table: the epilogue then leaves q and k unrotated
  p.rope = layer_rotary(c, layer)
               ? reinterpret_cast<const float2 *>(static_cast<const uint8_t *>(packed) + PL.rope_off)
               : nullptr;
  p.valid_start = valid_start; p.max_pos = c->max_pos; p.status = status;
  if (cc) {                        // new token t of sequence b sits at position cache_len[b] + t
    p.pos_add = cc->cache_len;
    p.pos_limit = cc->lmax;
  }
  // every kernel of the block is a programmatic dependent of the one before
  // (each waits for it with griddepcontrol.wait before touching its data, or,
  // in the model forward, for the flags of the row blocks it reads)
  p.pdl = 1;
  if (fc && layer > 0) {
    // the rows of x this tile reads, from the previous layer's down projection
    // (whose tiles complete only after the whole previous attention has, so
    // q, k and V^T are no longer read when they are overwritten here)
    p.done_in = fc->at(layer - 1, 1);
    p.done_need = gemm_arrivals(d, bn_down);
  }
  LAUNCH_K(SMOL_K_QKV, st, launch_gemm(kEpiQkvRope, bn_qkv, io.x16, lp.qkv, p, sms, st));

  // 2. causal GQA attention
  AttnParams ap{};
  ap.q = q; ap.k = k; ap.v = v; ap.o = o; ap.valid_start = valid_start;
  ap.B = B; ap.T = T; ap.H = H; ap.KV = KV; ap.hd = hd;
  ap.scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
  ap.window = layer_window(c, layer);
  ap.key_mask = key_mask;
  ap.status = status;
  ap.wait_ns = g_attn_wait_ns.load(std::memory_order_relaxed);
  ap.pdl = 1;
  if (attn_flags) ap.done_out = fc->at(layer, 0);
  if (cc) {
    // the cached slice and the new keys as one left-padded sequence of Tk keys;
    // the queries are its last T
    const int Tk = cc->lmax + T;
    f16 *kc = reinterpret_cast<f16 *>(ws + W.kc);
    f16 *vtc = reinterpret_cast<f16 *>(ws + W.vtc);
    int *vsb = reinterpret_cast<int *>(ws + W.vs);
    LAUNCH(launch_gather_cache_kv(cc->k_cache, cc->v_cache, cc->S_max, cc->cache_len, cc->lmax, k, v,
                                  (int)t_pad(T), B, KV, T, Tk, (int)t_pad(Tk), hd, kc, vtc, vsb, vsb + B, st));
    ap.k = kc;
    ap.v = nullptr;
    ap.v_t = vtc;
    ap.T_pad = (int)t_pad(Tk);
    ap.Tk = Tk;
    ap.q_off = Tk - T;
    ap.valid_start = vsb;
    ap.seq_order = vsb + B;        // longest caches first
    ap.pdl = 0;                    // the gather kernel in between is not a programmatic launch
    LAUNCH_K(SMOL_K_ATTN, st, launch_attention_tc(ap, st));
  } else {
    ap.v = nullptr;
    ap.v_t = v;
    ap.T_pad = (int)t_pad(T);
    LAUNCH_K(SMOL_K_ATTN, st, launch_attention_tc(ap, st));
  }

  // 3. O projection + residual: h = x + o Wo^T (f16), ssq_b += rowsum(h^2)
  GemmParams po{};
  po.M = (int)M; po.N = d; po.K = H * hd;
  po.out = h; po.out_is_f16 = 1; po.ldo = d; po.ssq_out = ssq_b; po.status = status;
  po.resid = io.resid_bf; po.resid_f16 = io.resid_f16; po.resid_f32 = io.resid_f32; po.pdl = 1;
  if (attn_flags) {
    po.done_in = fc->at(layer, 0);
    po.done_need = attention_tc_ctas_per_tile(hd, H, KV);
  }
  LAUNCH_K(SMOL_K_OPROJ, st, launch_gemm(kEpiResidual, bn_o, o, lp.o, po, sms, st));

  // 4. RMSNorm2 + gate/up + SwiGLU: a = silu(g) * u ; clears ssq_a for step 5
  GemmParams pg{};
  pg.M = (int)M; pg.N = 2 * I; pg.K = d;
  pg.out = a; pg.out_is_f16 = 1; pg.ldo = I; pg.ssq_in = ssq_b; pg.inv_dim = 1.0f / d;
  pg.eps = c->rms_eps; pg.ssq_zero = ssq_a; pg.status = status; pg.pdl = 1;
  LAUNCH_K(SMOL_K_GATEUP, st, launch_gemm(kEpiSwiglu, bn_gu, h, lp.gu, pg, sms, st));

  // 5. down projection + residual: out = h + a Wd^T, ssq_a += rowsum(out^2)
  GemmParams pd{};
  pd.M = (int)M; pd.N = d; pd.K = I;
  pd.out = io.out16; pd.out_is_f16 = io.out16_is_f16; pd.out_f32 = io.out_f32; pd.ldo = d;
  pd.resid_f16 = h; pd.ssq_out = ssq_a; pd.status = status; pd.pdl = 1;
  if (fc) pd.done_out = fc->at(layer, 1);
  LAUNCH_K(SMOL_K_DOWN, st, launch_gemm(kEpiResidual, bn_down, a, lp.down, pd, sms, st));
  return SMOL_OK;
}

}  // namespace

// ============================================================================
SMOL_API size_t smol_packed_bytes(const smol_config *cfg, int n_layers, int with_embed) {
  if (check_cfg(cfg) != SMOL_OK || n_layers < 0 || n_layers > cfg->n_layers) return 0;
  if (with_embed && cfg->vocab <= 0) return 0;
  return pack_layout(cfg, n_layers, with_embed).total;
}

SMOL_API int smol_prepare_weights(const smol_config *cfg, const smol_model_weights *w, int n_layers,
                                  void *packed, size_t packed_bytes, void *stream) {
  g_launches = 0;
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!w || !packed || n_layers < 0 || n_layers > cfg->n_layers) return SMOL_ERR_INVALID_ARG;
  if (n_layers > 0 && !w->layers) return SMOL_ERR_INVALID_ARG;
  const int with_embed = w->embed != nullptr;
  if (with_embed && (cfg->vocab <= 0 || !w->final_norm)) return SMOL_ERR_INVALID_ARG;
  const PackLayout L = pack_layout(cfg, n_layers, with_embed);
  if (packed_bytes < L.total) return SMOL_ERR_WORKSPACE;
  if (!aligned16(packed)) return SMOL_ERR_MISALIGNED;
  for (int l = 0; l < n_layers; ++l) {
    const smol_block_weights &b = w->layers[l];
    const void *ptrs[9] = {b.attn_norm, b.wq, b.wk, b.wv, b.wo, b.mlp_norm, b.wgate, b.wup, b.wdown};
    for (const void *p : ptrs) {
      if (!p) return SMOL_ERR_INVALID_ARG;
    }
  }
  int sms;
  if ((rc = device_sms(&sms))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t *base = static_cast<uint8_t *>(packed);
  const int d = cfg->hidden, hd = cfg->head_dim, H = cfg->n_heads, KV = cfg->n_kv_heads,
            I = cfg->intermediate;
  LAUNCH(launch_rope_table(cfg->max_pos, hd, cfg->rope_theta, reinterpret_cast<float2 *>(base + L.rope_off), st));
  for (int l = 0; l < n_layers; ++l) {
    const smol_block_weights &b = w->layers[l];
    uint8_t *lb = base + L.layer0_off + (size_t)l * L.layer_bytes;
    f16 *qkv = reinterpret_cast<f16 *>(lb + L.off_qkv);
    const bf16 *an = static_cast<const bf16 *>(b.attn_norm);
    const bf16 *mn = static_cast<const bf16 *>(b.mlp_norm);
    LAUNCH(launch_scale_cols_copy(static_cast<const bf16 *>(b.wq), an, (long long)H * hd, d, qkv, st));
    LAUNCH(launch_scale_cols_copy(static_cast<const bf16 *>(b.wk), an, (long long)KV * hd, d,
                                  qkv + (size_t)H * hd * d, st));
    LAUNCH(launch_scale_cols_copy(static_cast<const bf16 *>(b.wv), an, (long long)KV * hd, d,
                                  qkv + (size_t)(H + KV) * hd * d, st));
    LAUNCH(launch_scale_cols_copy(static_cast<const bf16 *>(b.wo), nullptr, d, H * hd,
                                  reinterpret_cast<f16 *>(lb + L.off_o), st));
    LAUNCH(launch_interleave_gate_up(static_cast<const bf16 *>(b.wgate), static_cast<const bf16 *>(b.wup),
                                     mn, I, d, reinterpret_cast<f16 *>(lb + L.off_gu), st));
    LAUNCH(launch_scale_cols_copy(static_cast<const bf16 *>(b.wdown), nullptr, d, I,
                                  reinterpret_cast<f16 *>(lb + L.off_down), st));
  }
  if (with_embed) {
    // bf16 copy of the table for the gather, f16 norm-folded copy for the tied head
    cudaError_t e = cudaMemcpyAsync(base + L.embed_off, w->embed, (size_t)cfg->vocab * d * 2,
                                    cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e);
    LAUNCH(launch_scale_cols_copy(static_cast<const bf16 *>(w->embed),
                                  static_cast<const bf16 *>(w->final_norm), cfg->vocab, d,
                                  reinterpret_cast<f16 *>(base + L.head_off), st));
  }
  return SMOL_OK;
}

SMOL_API size_t smol_workspace_bytes(const smol_config *cfg, int op, int B, int T) {
  if (check_cfg(cfg) != SMOL_OK || B <= 0) return 0;
  if (op == SMOL_OP_DECODE) return decode_ws_bytes(cfg, B);
  if (T <= 0) return 0;
  if (op != SMOL_OP_BLOCK && op != SMOL_OP_MODEL) return 0;
  return ws_layout(cfg, B, T, op == SMOL_OP_MODEL).total;
}

namespace {

int block_forward_impl(const smol_config *cfg, const void *packed, int layer, const void *x, void *out,
                       int act_dtype, int B, int T, const int32_t *valid_start, const uint8_t *key_mask,
                       void *k_out, void *v_out, void *ws, size_t ws_bytes, void *stream) {
  g_launches = 0;
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!packed || !x || !out || !ws || B <= 0 || T <= 0 || layer < 0 || layer >= cfg->n_layers ||
      (act_dtype != SMOL_ACT_BF16 && act_dtype != SMOL_ACT_F32))
    return SMOL_ERR_INVALID_ARG;
  if ((long long)B * T > 0x7fffffffLL) return SMOL_ERR_UNSUPPORTED_SHAPE;
  if (T > cfg->max_pos) return SMOL_ERR_TOO_LONG;
  if (!aligned16(packed) || !aligned16(x) || !aligned16(out) || !aligned16(ws) ||
      (k_out && !aligned16(k_out)) || (v_out && !aligned16(v_out)) ||
      (valid_start && (reinterpret_cast<uintptr_t>(valid_start) & 3u)))
    return SMOL_ERR_MISALIGNED;
  const WsLayout W = ws_layout(cfg, B, T);
  if (ws_bytes < W.total) return SMOL_ERR_WORKSPACE;
  int sms;
  if ((rc = device_sms(&sms))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  const long long M = (long long)B * T;
  float *ssq_a = reinterpret_cast<float *>(wsb + W.ssq_a);
  f16 *x16 = reinterpret_cast<f16 *>(wsb + W.x);
  BlockIO io{};
  io.x16 = x16;
  io.k_bf = static_cast<bf16 *>(k_out);
  io.v_bf = static_cast<bf16 *>(v_out);
  if (act_dtype == SMOL_ACT_F32) {
    LAUNCH_K(SMOL_K_ROWSTATS, st, launch_row_ssq_f32(static_cast<const float *>(x), M, cfg->hidden, x16, ssq_a,
                                                   reinterpret_cast<int *>(wsb + W.status), SeqCheck{valid_start, T, T}, st));
    io.resid_f32 = static_cast<const float *>(x);
    io.out_f32 = static_cast<float *>(out);
  } else {
    LAUNCH_K(SMOL_K_ROWSTATS, st, launch_row_ssq(static_cast<const bf16 *>(x), M, cfg->hidden, x16, ssq_a,
                                                   reinterpret_cast<int *>(wsb + W.status), SeqCheck{valid_start, T, T}, st));
    io.resid_bf = static_cast<const bf16 *>(x);
    io.out16 = out;
    io.out16_is_f16 = 0;
  }
  return run_block(cfg, packed, layer, io, B, T, valid_start, key_mask, W, wsb, sms, st);
}

int model_forward_impl(const smol_config *cfg, const void *packed, const int32_t *ids, int B, int T,
                       const int32_t *valid_start, const uint8_t *key_mask, void *logits, void *ws,
                       size_t ws_bytes, void *stream) {
  g_launches = 0;
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!packed || !ids || !logits || !ws || B <= 0 || T <= 0 || cfg->vocab <= 0)
    return SMOL_ERR_INVALID_ARG;
  if ((long long)B * T > 0x7fffffffLL) return SMOL_ERR_UNSUPPORTED_SHAPE;
  if (T > cfg->max_pos) return SMOL_ERR_TOO_LONG;
  if (!aligned16(packed) || !aligned16(logits) || !aligned16(ws) ||
      (reinterpret_cast<uintptr_t>(ids) & 3u) ||
      (valid_start && (reinterpret_cast<uintptr_t>(valid_start) & 3u)))
    return SMOL_ERR_MISALIGNED;
  const WsLayout W = ws_layout(cfg, B, T, true);
  if (ws_bytes < W.total) return SMOL_ERR_WORKSPACE;
  int sms;
  if ((rc = device_sms(&sms))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  const long long M = (long long)B * T;
  const PackLayout L = pack_layout(cfg, cfg->n_layers, 1);
  FlagCtx fc{reinterpret_cast<int *>(wsb + W.flags), row_blocks(B, T)};
  {
    const cudaError_t e = cudaMemsetAsync(fc.flags, 0, (size_t)cfg->n_layers * 2 * fc.mblocks * 4, st);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  const uint8_t *pk = static_cast<const uint8_t *>(packed);
  f16 *x = reinterpret_cast<f16 *>(wsb + W.x);
  float *ssq_a = reinterpret_cast<float *>(wsb + W.ssq_a);
  LAUNCH_K(SMOL_K_EMBED, st, launch_embed_rows(ids, reinterpret_cast<const bf16 *>(pk + L.embed_off), cfg->vocab,
                           cfg->hidden, M, x, nullptr, ssq_a, reinterpret_cast<int *>(wsb + W.status),
                           SeqCheck{valid_start, T, T}, st));
  // the residual stream is f16: each block reads x and writes its output over it
  BlockIO io{};
  io.x16 = x;
  io.resid_f16 = x;
  io.out16 = x;
  io.out16_is_f16 = 1;
  for (int l = 0; l < cfg->n_layers; ++l) {
    rc = run_block(cfg, packed, l, io, B, T, valid_start, key_mask, W, wsb, sms, st, nullptr, &fc);
    if (rc) return rc;
  }
  GemmParams p{};
  p.M = (int)M; p.N = cfg->vocab; p.K = cfg->hidden;
  p.done_in = fc.at(cfg->n_layers - 1, 1);
  p.done_need = gemm_arrivals(cfg->hidden, gemm_pick_bn(kEpiResidual, cfg->hidden, cfg->head_dim));
  p.out = logits; p.out_is_f16 = 0; p.ldo = cfg->vocab;
  p.ssq_in = ssq_a; p.inv_dim = 1.0f / cfg->hidden; p.eps = cfg->rms_eps;
  p.status = reinterpret_cast<int *>(wsb + W.status);
  p.pdl = 1;
  LAUNCH_K(SMOL_K_HEAD, st, launch_gemm(kEpiScale, gemm_pick_bn(kEpiScale, cfg->vocab, cfg->head_dim), x,
                     pk + L.head_off, p, sms, st));
  return SMOL_OK;
}

}  // namespace

SMOL_API int smol_block_forward(const smol_config *cfg, const void *packed, int layer, const void *x,
                                void *out, int act_dtype, int B, int T, const int32_t *valid_start,
                                void *k_out, void *v_out, void *ws, size_t ws_bytes, void *stream) {
  return block_forward_impl(cfg, packed, layer, x, out, act_dtype, B, T, valid_start, nullptr, k_out, v_out,
                            ws, ws_bytes, stream);
}

SMOL_API int smol_block_forward_masked(const smol_config *cfg, const void *packed, int layer, const void *x,
                                       void *out, int act_dtype, int B, int T, const uint8_t *key_mask,
                                       void *k_out, void *v_out, void *ws, size_t ws_bytes, void *stream) {
  if (!key_mask) {
    g_launches = 0;
    return SMOL_ERR_INVALID_ARG;
  }
  return block_forward_impl(cfg, packed, layer, x, out, act_dtype, B, T, nullptr, key_mask, k_out, v_out,
                            ws, ws_bytes, stream);
}

SMOL_API int smol_model_forward(const smol_config *cfg, const void *packed, const int32_t *ids, int B,
                                int T, const int32_t *valid_start, void *logits, void *ws,
                                size_t ws_bytes, void *stream) {
  return model_forward_impl(cfg, packed, ids, B, T, valid_start, nullptr, logits, ws, ws_bytes, stream);
}

SMOL_API int smol_model_forward_masked(const smol_config *cfg, const void *packed, const int32_t *ids, int B,
                                       int T, const uint8_t *key_mask, void *logits, void *ws,
                                       size_t ws_bytes, void *stream) {
  if (!key_mask) {
    g_launches = 0;
    return SMOL_ERR_INVALID_ARG;
  }
  return model_forward_impl(cfg, packed, ids, B, T, nullptr, key_mask, logits, ws, ws_bytes, stream);
}

namespace {

// The decode step; with `next` the greedy choice is taken in the head GEMM's
// epilogue (logits may then be nullptr).
int decode_impl(const smol_config *cfg, const void *packed, const int32_t *ids, const int32_t *cache_len, int B,
                const void *k_cache, const void *v_cache, int S_max, void *k_new, void *v_new, void *logits,
                int32_t *next, void *ws, size_t ws_bytes, void *stream) {
  g_launches = 0;
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!packed || !ids || !cache_len || !k_cache || !v_cache || !k_new || !v_new || (!logits && !next) || !ws ||
      B <= 0 || S_max <= 0 || cfg->vocab <= 0)
    return SMOL_ERR_INVALID_ARG;
  if (!aligned16(packed) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) ||
      !aligned16(v_new) || (logits && !aligned16(logits)) || !aligned16(ws) ||
      (reinterpret_cast<uintptr_t>(ids) & 3u) || (reinterpret_cast<uintptr_t>(cache_len) & 3u) ||
      (reinterpret_cast<uintptr_t>(next) & 3u))
    return SMOL_ERR_MISALIGNED;
  if (ws_bytes < decode_ws_bytes(cfg, B)) return SMOL_ERR_WORKSPACE;
  int sms;
  if ((rc = device_sms(&sms))) return rc;
  const PackLayout L = pack_layout(cfg, cfg->n_layers, 1);
  DecodeArgs a{};
  a.cfg = *cfg;
  a.B = B;
  a.S_max = S_max;
  a.ids = ids;
  a.cache_len = cache_len;
  a.k_cache = static_cast<const bf16 *>(k_cache);
  a.v_cache = static_cast<const bf16 *>(v_cache);
  a.k_new = static_cast<bf16 *>(k_new);
  a.v_new = static_cast<bf16 *>(v_new);
  a.logits = static_cast<bf16 *>(logits);
  a.next = next;
  const uint8_t *pk = static_cast<const uint8_t *>(packed);
  a.rope = reinterpret_cast<const float2 *>(pk + L.rope_off);
  a.embed = reinterpret_cast<const bf16 *>(pk + L.embed_off);
  a.head = reinterpret_cast<const f16 *>(pk + L.head_off);
  a.layer0 = pk + L.layer0_off;
  a.layer_bytes = L.layer_bytes;
  a.off_qkv = L.off_qkv;
  a.off_o = L.off_o;
  a.off_gu = L.off_gu;
  a.off_down = L.off_down;
  int n = 0;
  cudaError_t e = run_decode(a, ws, sms, static_cast<cudaStream_t>(stream), &n);
  g_launches = n;
  if (e != cudaSuccess) return cuda_fail(e);
  return SMOL_OK;
}

}  // namespace

SMOL_API int smol_decode_step(const smol_config *cfg, const void *packed, const int32_t *ids,
                              const int32_t *cache_len, int B, const void *k_cache,
                              const void *v_cache, int S_max, void *k_new, void *v_new,
                              void *logits, void *ws, size_t ws_bytes, void *stream) {
  if (!logits) {
    g_launches = 0;
    return SMOL_ERR_INVALID_ARG;
  }
  return decode_impl(cfg, packed, ids, cache_len, B, k_cache, v_cache, S_max, k_new, v_new, logits, nullptr,
                     ws, ws_bytes, stream);
}

SMOL_API int smol_decode_next(const smol_config *cfg, const void *packed, const int32_t *ids,
                              const int32_t *cache_len, int B, const void *k_cache, const void *v_cache,
                              int S_max, void *k_new, void *v_new, void *logits, float temperature,
                              int top_k, float top_p, int do_sample, const float *uniform, int32_t *next,
                              void *ws, size_t ws_bytes, void *stream) {
  g_launches = 0;
  if (!next || temperature != temperature || top_p != top_p) return SMOL_ERR_INVALID_ARG;
  const bool greedy = !do_sample || !(temperature > 0.f);
  if (greedy)
    return decode_impl(cfg, packed, ids, cache_len, B, k_cache, v_cache, S_max, k_new, v_new, logits, next,
                       ws, ws_bytes, stream);
  if (!logits || !uniform || (reinterpret_cast<uintptr_t>(uniform) & 3u)) return SMOL_ERR_INVALID_ARG;
  int rc = decode_impl(cfg, packed, ids, cache_len, B, k_cache, v_cache, S_max, k_new, v_new, logits, nullptr,
                       ws, ws_bytes, stream);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);   // g_launches holds the decode step's launches
  LAUNCH_K(SMOL_K_SAMPLE, st, launch_sample(logits, cfg->vocab, B, cfg->vocab, temperature, top_k, top_p, 1,
                                            uniform, next, st));
  return SMOL_OK;
}

SMOL_API int smol_append_kv(const smol_config *cfg, int B, const void *k_new, const void *v_new, void *k_cache,
                            void *v_cache, int S_max, int32_t *cache_len, void *stream) {
  g_launches = 0;
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!k_new || !v_new || !k_cache || !v_cache || !cache_len || B <= 0 || S_max <= 0) return SMOL_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(cache_len) & 3u))
    return SMOL_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LAUNCH(launch_append_kv(static_cast<const bf16 *>(k_new), static_cast<const bf16 *>(v_new),
                          static_cast<bf16 *>(k_cache), static_cast<bf16 *>(v_cache), cache_len, cfg->n_layers,
                          B, cfg->n_kv_heads, S_max, cfg->head_dim, st));
  ++g_launches;                                   // the copy and the length update
  return SMOL_OK;
}

SMOL_API size_t smol_prefill_cache_workspace_bytes(const smol_config *cfg, int B, int T, int S_max) {
  if (check_cfg(cfg) != SMOL_OK || B <= 0 || T <= 0 || S_max <= 0 || T >= cfg->max_pos) return 0;
  if (!attention_tc_supported(cfg->head_dim, cfg->n_heads, cfg->n_kv_heads)) return 0;
  return ws_layout_cache(cfg, B, T, S_max).total;
}

SMOL_API int smol_prefill_with_cache(const smol_config *cfg, const void *packed, const int32_t *ids, int B, int T,
                                     const int32_t *cache_len, const void *k_cache, const void *v_cache,
                                     int S_max, void *k_new, void *v_new, void *logits, void *ws,
                                     size_t ws_bytes, void *stream) {
  g_launches = 0;
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!packed || !ids || !cache_len || !k_cache || !v_cache || !k_new || !v_new || !logits || !ws || B <= 0 ||
      T <= 0 || S_max <= 0 || cfg->vocab <= 0)
    return SMOL_ERR_INVALID_ARG;
  if (!attention_tc_supported(cfg->head_dim, cfg->n_heads, cfg->n_kv_heads)) return SMOL_ERR_UNSUPPORTED_SHAPE;
  if ((long long)B * T > 0x7fffffffLL) return SMOL_ERR_UNSUPPORTED_SHAPE;
  if (T >= cfg->max_pos) return SMOL_ERR_TOO_LONG;
  if (!aligned16(packed) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) ||
      !aligned16(v_new) || !aligned16(logits) || !aligned16(ws) || (reinterpret_cast<uintptr_t>(ids) & 3u) ||
      (reinterpret_cast<uintptr_t>(cache_len) & 3u))
    return SMOL_ERR_MISALIGNED;
  const WsLayout W = ws_layout_cache(cfg, B, T, S_max);
  if (ws_bytes < W.total) return SMOL_ERR_WORKSPACE;
  int sms;
  if ((rc = device_sms(&sms))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  const long long M = (long long)B * T;
  const PackLayout L = pack_layout(cfg, cfg->n_layers, 1);
  const uint8_t *pk = static_cast<const uint8_t *>(packed);
  f16 *x = reinterpret_cast<f16 *>(wsb + W.x);
  float *ssq_a = reinterpret_cast<float *>(wsb + W.ssq_a);
  LAUNCH_K(SMOL_K_EMBED, st, launch_embed_rows(ids, reinterpret_cast<const bf16 *>(pk + L.embed_off), cfg->vocab,
                           cfg->hidden, M, x, nullptr, ssq_a, reinterpret_cast<int *>(wsb + W.status),
                           SeqCheck{cache_len, T, cache_lmax(cfg, T, S_max)}, st));
  const size_t layer_cache = (size_t)B * cfg->n_kv_heads * S_max * cfg->head_dim;
  const size_t layer_new = (size_t)B * cfg->n_kv_heads * T * cfg->head_dim;
  for (int l = 0; l < cfg->n_layers; ++l) {
    BlockIO io{};
    io.x16 = x;
    io.resid_f16 = x;
    io.out16 = x;
    io.out16_is_f16 = 1;
    io.k_bf = static_cast<bf16 *>(k_new) + l * layer_new;
    io.v_bf = static_cast<bf16 *>(v_new) + l * layer_new;
    CacheCtx cc{static_cast<const bf16 *>(k_cache) + l * layer_cache,
                static_cast<const bf16 *>(v_cache) + l * layer_cache, cache_len, S_max,
                cache_lmax(cfg, T, S_max)};
    rc = run_block(cfg, packed, l, io, B, T, nullptr, nullptr, W, wsb, sms, st, &cc);
    if (rc) return rc;
  }
  GemmParams p{};
  p.M = (int)M; p.N = cfg->vocab; p.K = cfg->hidden;
  p.out = logits; p.out_is_f16 = 0; p.ldo = cfg->vocab;
  p.ssq_in = ssq_a; p.inv_dim = 1.0f / cfg->hidden; p.eps = cfg->rms_eps;
  p.status = reinterpret_cast<int *>(wsb + W.status);
  p.pdl = 1;
  LAUNCH_K(SMOL_K_HEAD, st, launch_gemm(kEpiScale, gemm_pick_bn(kEpiScale, cfg->vocab, cfg->head_dim), x,
                     pk + L.head_off, p, sms, st));
  return SMOL_OK;
}

SMOL_API int smol_sample(const void *logits, int B, int V, long long ld, float temperature, int top_k,
                         float top_p, int do_sample, const float *uniform, int32_t *next, void *stream) {
  g_launches = 0;
  const bool greedy = !do_sample || !(temperature > 0.f);
  if (!logits || !next || (!greedy && !uniform)) return SMOL_ERR_INVALID_ARG;
  if (B < 1 || V < 1 || ld < V || temperature != temperature || top_p != top_p) return SMOL_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) & 1u) || (reinterpret_cast<uintptr_t>(next) & 3u) ||
      (reinterpret_cast<uintptr_t>(uniform) & 3u))
    return SMOL_ERR_MISALIGNED;
  int sms = 0;
  int rc = device_sms(&sms);
  if (rc != SMOL_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LAUNCH_K(SMOL_K_SAMPLE, st, launch_sample(logits, ld, B, V, temperature, top_k, top_p, do_sample, uniform,
                                            reinterpret_cast<int *>(next), st));
  return SMOL_OK;
}

// The host status of a device status word: the first code any kernel wrote
// (range 0x3xx: a value beyond f16; 0x4xx: a clamped input; the rest: a bounded
// wait that gave up).
int status_of_word(int h) {
  if (h == 0) return SMOL_OK;
  if ((h & 0xf00) == 0x300) return SMOL_ERR_RANGE;
  if ((h & 0xf00) == 0x400) return SMOL_ERR_INPUT;
  return SMOL_ERR_TIMEOUT;
}

SMOL_API int smol_workspace_status(void *ws, void *stream) {
  if (!ws) return SMOL_ERR_INVALID_ARG;
  int h = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&h, ws, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(int), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  return status_of_word(h);
}

SMOL_API int smol_last_launch_count(void) { return g_launches; }

SMOL_API void smol_set_wait_limit_ns(unsigned long long ns) {
  g_attn_wait_ns.store(ns, std::memory_order_relaxed);
}

SMOL_API const char *smol_status_string(int status) {
  switch (status) {
    case SMOL_OK: return "ok";
    case SMOL_ERR_INVALID_ARG: return "invalid argument";
    case SMOL_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case SMOL_ERR_MISALIGNED: return "device buffer not 16-byte aligned";
    case SMOL_ERR_TOO_LONG: return "positions exceed max_position_embeddings";
    case SMOL_ERR_WORKSPACE: return "workspace or packed buffer too small";
    case SMOL_ERR_CUDA: return g_cuda_err[0] ? g_cuda_err : "CUDA error";
    case SMOL_ERR_DEVICE: return "current device is not compute capability 10.3 (GB300)";
    case SMOL_ERR_TIMEOUT: return "a kernel's bounded wait gave up";
    case SMOL_ERR_RANGE: return "a value went beyond the f16 range of the residual stream or an operand";
    case SMOL_ERR_INPUT: return "an input value (token id, cache length, left-padding start) was out of range";
    default: return "unknown status";
  }
}
