// Combining the split-KV attention chunks of one (token row, query head):
//   out[d] = sum_c o_c[d] e^(m_c - M) / sum_c l_c e^(m_c - M),  M = max_c m_c,
// where chunk c of 64 cache slots left its running max m_c, its sum of
// exponentials l_c and its unnormalised output o_c. Any kernel that merges
// through this routine gets bit-identical results.
#pragma once

#include "sf_kernels.h"

namespace sf {

constexpr int kMaxKvChunks = 256;
constexpr int kMergeThreads = 256;
constexpr int kMergeLoads = 24;

struct MergeSmem {
  float wgt[kMaxKvChunks];
  float opart[kMergeThreads];
  float red[kMergeThreads / 32], red_l[kMergeThreads / 32];
  float l;
};

// All kMergeThreads threads of the CTA call this together. Thread (g, d)
// with g = tid / hd adds the chunks g, g + G, g + 2G, ... (G = 256 / hd) in
// order, up to kMergeLoads of them loaded at once, and the G partial sums
// are then added in order g = 0, 1, ...; every chunk's (max, sum) pair is
// loaded in the same round. The softmax denominator is a fixed tree (within
// warps, then warps in order). The result is valid in threads tid < hd
// (dimension d = tid); the scratch is free again when it returns.
__device__ __forceinline__ float merge_row_head(const float* part, int nq, int hd, int n_kv_chunks, int m, int h,
                                                int nch, MergeSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = kMergeThreads / hd;
  const int grp = tid / hd, d = tid - grp * hd;
  const int stride = hd + 2;
  const float* src = part + ((size_t)m * nq + h) * n_kv_chunks * stride;
  // Round one: every chunk's (max, sum) and this thread's first output terms.
  const float mc = tid < nch ? src[(size_t)tid * stride + hd] : -INFINITY;
  const float lc = tid < nch ? src[(size_t)tid * stride + hd + 1] : 0.f;
  float v[kMergeLoads];
#pragma unroll
  for (int q = 0; q < kMergeLoads; ++q) {
    const int c = grp + q * G;
    v[q] = c < nch ? src[(size_t)c * stride + d] : 0.f;
  }
  const float wm = warp_max(mc);
  if (lane == 0) sm.red[warp] = wm;
  __syncthreads();
  float mx = sm.red[0];
#pragma unroll
  for (int w = 1; w < kMergeThreads / 32; ++w) mx = fmaxf(mx, sm.red[w]);
  const float wc = tid < nch ? expf(mc - mx) : 0.f;
  if (tid < nch) sm.wgt[tid] = wc;
  const float lsum = warp_sum(lc * wc);
  if (lane == 0) sm.red_l[warp] = lsum;
  __syncthreads();
  if (tid == 0) {
    float l = sm.red_l[0];
    for (int w = 1; w < kMergeThreads / 32; ++w) l += sm.red_l[w];
    sm.l = l;
  }
  float o = 0.f;
#pragma unroll
  for (int q = 0; q < kMergeLoads; ++q) {
    const int c = grp + q * G;
    if (c < nch) o = fmaf(v[q], sm.wgt[c], o);
  }
  // Longer contexts: further rounds of kMergeLoads chunks per thread.
  for (int c0 = kMergeLoads * G; c0 < nch; c0 += kMergeLoads * G) {
#pragma unroll
    for (int q = 0; q < kMergeLoads; ++q) {
      const int c = c0 + grp + q * G;
      v[q] = c < nch ? src[(size_t)c * stride + d] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kMergeLoads; ++q) {
      const int c = c0 + grp + q * G;
      if (c < nch) o = fmaf(v[q], sm.wgt[c], o);
    }
  }
  sm.opart[tid] = o;
  __syncthreads();
  float t = 0.f;
  if (grp == 0) {
    t = sm.opart[d];
    for (int g2 = 1; g2 < G; ++g2) t += sm.opart[g2 * hd + d];
    t = t / sm.l;
  }
  __syncthreads();
  return t;
}

}  // namespace sf
