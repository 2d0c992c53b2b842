// sample.cu - next-token choice from rows of logits ("model.py" (SmolLM2-135M)
// section 7 generate; the abi96062 "model.py" generate).
//
// Per row: greedy (do_sample off or temperature <= 0) is the first index of the
// row maximum.  Otherwise z = logits / temperature; top_k > 0 removes values
// below the k-th largest (values equal to it stay); top_p < 1 keeps, in
// descending z order with equal values in ascending index order, the shortest
// prefix whose cumulative softmax probability (over the top-k survivors)
// exceeds top_p; the token is the first index, in vocabulary order, at which
// the cumulative probability of the survivors exceeds the caller's uniform
// number u in [0, 1) (the inverse CDF).
//
// One CTA of 1024 threads per row; thread t owns the index range
// [t*seg, (t+1)*seg).  Values are ranked by a 16-bit key that orders bf16
// numbers (-0 counted as +0).  The k-th largest key and the top-p cut come from
// two-level radix histograms (high byte, then low byte inside the crossing bin)
// of counts and of softmax masses.  Masses are fixed point, e * 2^44 with
// e = exp(z - z_max) <= 1, accumulated as 64-bit integers: every sum is exact,
// so no decision depends on the order of the atomics.  Equal values have equal
// masses, so the cut inside the crossing value's group is arithmetic: its
// first t*+1 members in index order survive.  The draw is a block-wide
// exclusive scan of the surviving masses of each thread's range.
#include <math.h>

#include "common.cuh"
#include "prims.cuh"

namespace smol {
namespace {

constexpr int kSmpThreads = 1024;
constexpr float kMassScale = 17592186044416.f;   // 2^44

// 16-bit key ordering bf16 values numerically (larger value, larger key).
__device__ __forceinline__ uint32_t bf16_key(uint16_t bits) { return bf16_order_key(bits); }

__device__ __forceinline__ float key_value(uint32_t key) {
  const uint16_t bits = (key & 0x8000u) ? static_cast<uint16_t>(key & 0x7FFFu)
                                        : static_cast<uint16_t>(~key & 0xFFFFu);
  return __bfloat162float(__ushort_as_bfloat16(bits));
}

__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v, unsigned long long *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = sh[lane];
#pragma unroll
    for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) sh[32] = v;
  }
  __syncthreads();
  v = sh[32];
  __syncthreads();                               // sh may be reused at once
  return v;
}

// Exclusive prefix sum over the block (integers: exact); *total gets the sum.
__device__ __forceinline__ unsigned long long block_excl_scan_u64(unsigned long long v, unsigned long long *sh,
                                                                  unsigned long long *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long w = sh[lane];
    unsigned long long wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    sh[lane] = wi - w;                           // warp offsets
    if (lane == 31) sh[32] = wi;
  }
  __syncthreads();
  const unsigned long long r = sh[warp] + inc - v;
  *total = sh[32];
  __syncthreads();
  return r;
}

// Warp 0 only.  Visits bins 255 .. 0 from the top and returns the first bin h
// at which base + (bins above h) + bins[h] reaches thr (>= for counts, > for
// masses), with *above = the bins above h; -1 if no bin does.
template <typename Tb, bool kStrict>
__device__ __forceinline__ int find_desc(const Tb *bins, unsigned long long base, double thr,
                                         unsigned long long *above) {
  const int lane = threadIdx.x & 31;
  auto crosses = [&](unsigned long long c) {
    const double x = static_cast<double>(base + c);
    return kStrict ? (x > thr) : (x >= thr);
  };
  unsigned long long local = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) local += bins[255 - 8 * lane - j];
  unsigned long long inc = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  const unsigned m = __ballot_sync(0xffffffffu, crosses(inc));
  if (m == 0) return -1;
  const int L = __ffs(m) - 1;                    // the first lane whose running total crosses
  int h = -1;
  unsigned long long ab = 0;
  if (lane == L) {
    unsigned long long run = inc - local;        // exact: integers
    for (int j = 0; j < 8; ++j) {
      const int hb = 255 - 8 * lane - j;
      if (crosses(run + bins[hb])) {
        h = hb;
        ab = run;
        break;
      }
      run += bins[hb];
    }
  }
  h = __shfl_sync(0xffffffffu, h, L);
  ab = __shfl_sync(0xffffffffu, ab, L);
  *above = ab;
  return h;
}

struct SampleParams {
  const uint16_t *logits;   // bf16 [B][ld]
  long long ld;
  int V;
  float temperature;
  int top_k;
  float top_p;
  int do_sample;
  const float *uniform;     // [B]
  int *next;                // [B]
};

__global__ void __launch_bounds__(kSmpThreads, 1) sample_kernel(const SampleParams p) {
  __shared__ unsigned int cnt_hi[256], cnt_lo[256], cnt_p[256];
  __shared__ unsigned long long mass_hi[256], mass_lo[256];
  __shared__ unsigned long long red[33];
  __shared__ int s_h, s_l;
  __shared__ unsigned long long s_above, s_total;
  __shared__ int s_pick;

  const int tid = threadIdx.x;
  const int V = p.V;
  const uint16_t *row = p.logits + static_cast<long long>(blockIdx.x) * p.ld;
  const int seg = (V + kSmpThreads - 1) / kSmpThreads;
  const int i0 = min(V, tid * seg), i1 = min(V, i0 + seg);
  const bool greedy = !p.do_sample || !(p.temperature > 0.f);
  const bool use_k = !greedy && p.top_k > 0 && p.top_k < V;
  const bool use_p = !greedy && p.top_p < 1.f;
  auto key_at = [&](int i) -> uint32_t { return bf16_key(row[i]); };

  for (int i = tid; i < 256; i += kSmpThreads) {
    cnt_hi[i] = cnt_lo[i] = cnt_p[i] = 0u;
    mass_hi[i] = mass_lo[i] = 0ull;
  }
  if (tid == 0) s_pick = -1;
  __syncthreads();

  // ---- pass 1: row maximum (its first index) and high-byte counts for top-k
  unsigned long long best = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t k = key_at(i);
    best = max(best, argmax_pack(k, static_cast<uint32_t>(i)));
    if (use_k) atomicAdd(&cnt_hi[k >> 8], 1u);
  }
  best = block_max_u64(best, red);               // also orders the count atomics before their reads
  const uint32_t kmax = static_cast<uint32_t>(best >> 32);
  if (greedy) {
    if (tid == 0) p.next[blockIdx.x] = argmax_index(best);
    return;
  }
  const float T = p.temperature;
  const float zmax = key_value(kmax) / T;
  // fixed-point softmax mass of a value (the same integer for equal values)
  auto mass_of = [&](uint32_t k) -> unsigned long long {
    const float e = expf(key_value(k) / T - zmax);
    return __float2ull_rn(e * kMassScale);
  };

  // ---- top-k: the k-th largest key tau; survivors have key >= tau
  uint32_t tau = 0;
  if (use_k) {
    if (tid < 32) {
      unsigned long long above = 0;
      const int h = find_desc<unsigned int, false>(cnt_hi, 0ull, static_cast<double>(p.top_k), &above);
      if (tid == 0) {
        s_h = h;
        s_above = above;
      }
    }
    __syncthreads();
    const int h = s_h;                           // found: the V counts exceed top_k
    for (int i = i0; i < i1; ++i) {
      const uint32_t k = key_at(i);
      if (static_cast<int>(k >> 8) == h) atomicAdd(&cnt_lo[k & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      unsigned long long above = 0;
      const int l = find_desc<unsigned int, false>(cnt_lo, s_above, static_cast<double>(p.top_k), &above);
      if (tid == 0) s_l = l;
    }
    __syncthreads();
    tau = (static_cast<uint32_t>(h) << 8) | static_cast<uint32_t>(max(s_l, 0));
  }

  // ---- top-p: the value v at which the descending cumulative mass first
  // exceeds top_p * total, and how many of its members (index order) survive
  bool cut = false;
  uint32_t vcut = 0;
  unsigned long long tcut = 0;                   // members of v with rank <= tcut survive
  if (use_p) {
    for (int i = i0; i < i1; ++i) {
      const uint32_t k = key_at(i);
      if (k >= tau) atomicAdd(&mass_hi[k >> 8], mass_of(k));
    }
    __syncthreads();
    if (tid < 32) {
      unsigned long long tot = 0;
      for (int j = tid; j < 256; j += 32) tot += mass_hi[j];
#pragma unroll
      for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
      const double X = static_cast<double>(p.top_p) * static_cast<double>(tot);
      unsigned long long above = 0;
      const int h = find_desc<unsigned long long, true>(mass_hi, 0ull, X, &above);
      if (tid == 0) {
        s_h = h;
        s_above = above;
        s_total = tot;
      }
    }
    __syncthreads();
    const int h = s_h;
    if (h >= 0) {
      for (int i = i0; i < i1; ++i) {
        const uint32_t k = key_at(i);
        if (k >= tau && static_cast<int>(k >> 8) == h) {
          atomicAdd(&mass_lo[k & 255u], mass_of(k));
          atomicAdd(&cnt_p[k & 255u], 1u);
        }
      }
      __syncthreads();
      if (tid < 32) {
        const double X = static_cast<double>(p.top_p) * static_cast<double>(s_total);
        const unsigned long long base = s_above;
        __syncwarp();                            // every lane has read s_above before lane 0 rewrites it
        unsigned long long above = 0;
        const int l = find_desc<unsigned long long, true>(mass_lo, base, X, &above);
        if (tid == 0) {
          s_l = l;
          s_above = base + above;                // mass of the values above v
        }
      }
      __syncthreads();
      if (s_l >= 0) {                            // found whenever the high bin was
        cut = true;
        vcut = (static_cast<uint32_t>(h) << 8) | static_cast<uint32_t>(s_l);
        const double X = static_cast<double>(p.top_p) * static_cast<double>(s_total);
        const double mv = static_cast<double>(mass_of(vcut));   // > 0: a zero mass never crosses
        const double q = floor((X - static_cast<double>(s_above)) / mv);
        const unsigned long long nv = cnt_p[s_l];
        tcut = q < 0.0 ? 0ull : (q >= static_cast<double>(nv) ? nv - 1 : static_cast<unsigned long long>(q));
      }
    }
  }

  // ---- the draw: ranks of v's members in index order, surviving masses,
  // block scan, and the first index whose running mass exceeds u * total
  unsigned long long my_v = 0;
  if (cut)
    for (int i = i0; i < i1; ++i) my_v += key_at(i) == vcut ? 1ull : 0ull;
  unsigned long long nv_total = 0;
  const unsigned long long vbase = block_excl_scan_u64(my_v, red, &nv_total);
  auto survives = [&](uint32_t k, unsigned long long &r) {
    if (k < tau) return false;
    if (!cut || k > vcut) return true;
    if (k < vcut) return false;
    return r++ <= tcut;
  };
  unsigned long long my_mass = 0;
  int my_last = -1;
  {
    unsigned long long r = vbase;
    for (int i = i0; i < i1; ++i) {
      const uint32_t k = key_at(i);
      if (survives(k, r)) {
        const unsigned long long m = mass_of(k);
        if (m) {
          my_mass += m;
          my_last = i;
        }
      }
    }
  }
  unsigned long long total = 0;
  const unsigned long long pre = block_excl_scan_u64(my_mass, red, &total);
  const double target = static_cast<double>(p.uniform[blockIdx.x]) * static_cast<double>(total);
  auto crosses = [&](unsigned long long c) { return static_cast<double>(c) > target; };
  if (my_mass && !crosses(pre) && crosses(pre + my_mass)) {   // exactly one thread
    unsigned long long r = vbase, run = pre;
    for (int i = i0; i < i1; ++i) {
      const uint32_t k = key_at(i);
      if (survives(k, r)) {
        run += mass_of(k);
        if (crosses(run)) {
          s_pick = i;
          break;
        }
      }
    }
  }
  // u within rounding of 1: the last surviving index
  const unsigned long long lastp = block_max_u64(static_cast<unsigned long long>(my_last + 1), red);
  if (tid == 0) p.next[blockIdx.x] = s_pick >= 0 ? s_pick : static_cast<int>(lastp) - 1;
}

}  // namespace

cudaError_t launch_sample(const void *logits, long long ld, int B, int V, float temperature, int top_k,
                          float top_p, int do_sample, const float *uniform, int *next, cudaStream_t st) {
  SampleParams p{};
  p.logits = static_cast<const uint16_t *>(logits);
  p.ld = ld;
  p.V = V;
  p.temperature = temperature;
  p.top_k = top_k;
  p.top_p = top_p > 0.f ? top_p : 0.f;   // top_p <= 0 keeps the first token in descending order, as 0 does
  p.do_sample = do_sample;
  p.uniform = uniform;
  p.next = next;
  sample_kernel<<<static_cast<unsigned>(B), kSmpThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace smol
