// profile.cu - optional per-launch CUDA-event timing (measurement only).
#include <vector>

#include "profile.cuh"
#include "smol.h"

#define SMOL_API extern "C" __attribute__((visibility("default")))

namespace smol {
namespace {

struct ProfState {
  unsigned mask = 0;
  int capacity = 0;
  int count = 0;
  std::vector<cudaEvent_t> ev;   // 2 per launch
  std::vector<int> kinds;
  bool open = false;             // a launch is between prof_before and prof_after
};

thread_local ProfState g_prof;

}  // namespace

void prof_before(int kind, cudaStream_t st) {
  ProfState &s = g_prof;
  if (!(s.mask & (1u << kind)) || s.count >= s.capacity) return;
  cudaEventRecord(s.ev[2 * s.count], st);
  s.open = true;
}

void prof_after(int kind, cudaStream_t st) {
  ProfState &s = g_prof;
  if (!s.open) return;
  cudaEventRecord(s.ev[2 * s.count + 1], st);
  s.kinds[s.count] = kind;
  ++s.count;
  s.open = false;
}

}  // namespace smol

using smol::g_prof;

SMOL_API int smol_profile_begin(unsigned kind_mask, int capacity) {
  if (capacity < 0) return SMOL_ERR_INVALID_ARG;
  if ((int)g_prof.ev.size() < 2 * capacity) {
    const size_t old = g_prof.ev.size();
    g_prof.ev.resize(2 * capacity);
    for (size_t i = old; i < g_prof.ev.size(); ++i)
      if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) {
        g_prof.ev.resize(i);
        return SMOL_ERR_CUDA;
      }
  }
  g_prof.kinds.assign(capacity, -1);
  g_prof.mask = kind_mask;
  g_prof.capacity = capacity;
  g_prof.count = 0;
  g_prof.open = false;
  return SMOL_OK;
}

SMOL_API int smol_profile_end(int *kinds, float *ms, int cap) {
  const int n = g_prof.count < cap ? g_prof.count : cap;
  g_prof.mask = 0;
  for (int i = 0; i < n; ++i) {
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess) return SMOL_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess)
      return SMOL_ERR_CUDA;
    if (kinds) kinds[i] = g_prof.kinds[i];
    if (ms) ms[i] = t;
  }
  g_prof.count = 0;
  return n;
}
