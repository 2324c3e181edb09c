// Epilogues of the weight-streaming GEMMs (mma.sync and tcgen05 kernels):
// they take a CTA's finished tile ys[m][128] (token row m of this launch's
// rows m0 .., output row 128 * rb + r) in shared memory and write the
// projection's result where the next kernel reads it.
#pragma once

#include "sf_kernels.h"

namespace sf {
namespace {

// Global operands of the epilogue, loaded right after the kernel waits on
// its producer so their latency overlaps the weight stream.
template <int T>
struct EpiPre {
  static constexpr int kE = (4 * T * kBlockRows + kGemmThreads - 1) / kGemmThreads;
  float v0[kE], v1[kE];
  float2 cs[kE];
};

// The epilogues' barrier: the first kGemmThreads threads of the CTA (all of
// them in the 256-thread kernels; the tcgen05 kernel's NF4 form has four more
// warps, which do not take part in the epilogue).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kGemmThreads) : "memory"); }

// Rows m < M of the CTA are token rows m0 + m of the forward; pos[m] is the
// cache slot of row m0 + m (its RoPE position differs for the rows of a
// multi-candidate verify).
// F32: the fp32-weight kernel (biases and gains in fp32); the others read bf16.
template <int T, int EPI, bool F32 = false>
__device__ __forceinline__ void epi_prefetch(const GemmArgs& a, int rb, int m0, int M, EpiPre<T>& pre,
                                             const int* pos) {
  constexpr int kE = EpiPre<T>::kE;
  if (EPI == EPI_RESID) {
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      const int i = threadIdx.x + e * kGemmThreads;
      const int m = i / kBlockRows, n = rb * kBlockRows + (i - m * kBlockRows);
      pre.v0[e] = (m < M && n < a.N) ? a.out[(size_t)(m0 + m) * a.out_ld + n] : 0.f;
      pre.v1[e] = (a.frag_gain && n < a.N) ? ldw(a.frag_gain, n, F32) : 0.f;
    }
  } else if (EPI == EPI_QKV) {
    const int half = a.hd >> 1;
    const int n0 = rb * kBlockRows;
    const int s = n0 < a.seg_end[0] ? 0 : (n0 < a.seg_end[1] ? 1 : 2);   // one segment per block
    const int seg0 = s ? a.seg_end[s - 1] : 0;
    const void* bias = a.bias[s];
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      const int i = threadIdx.x + e * kGemmThreads;
      const int m = i / kBlockRows, r = i - m * kBlockRows;
      const int local = n0 + r - seg0;
      const int d = local % a.hd;
      pre.v0[e] = pre.v1[e] = 0.f;
      pre.cs[e] = make_float2(1.f, 0.f);
      if (m < M && n0 + r < a.N) {
        if (bias) pre.v0[e] = ldw(bias, local, F32);
        if (s < 2 && d < half) {
          if (bias) pre.v1[e] = ldw(bias, local + half, F32);
          const int gap = a.rs.tree_g > 0 ? tree_gap(a.rs, (m0 + m) % a.rs.rps) : 0;
          pre.cs[e] = a.rope[(size_t)(pos[m] - gap) * half + d];
        }
      }
    }
  }
}

template <int T>
__device__ void epi_resid(const GemmArgs& a, float* ys, int rb, int m0, int M, int Tt, const EpiPre<T>& pre) {
  constexpr int kE = EpiPre<T>::kE;
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    const int i = threadIdx.x + e * kGemmThreads;
    if (i >= M * kBlockRows) continue;
    const int m = i / kBlockRows, n = rb * kBlockRows + (i - m * kBlockRows);
    float v = 0.f;
    if (n < a.N) {
      v = pre.v0[e] + ys[i];
      a.out[(size_t)(m0 + m) * a.out_ld + n] = v;
      if (a.frag_out) act_store(a.frag_out, m0 + m, n, Tt, v * pre.v1[e], a.frag_umma);
    }
    ys[i] = v;
  }
  epi_sync();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int m = warp; m < M; m += kGemmThreads / 32) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float v = ys[m * kBlockRows + lane + 32 * j];
      s = fmaf(v, v, s);
    }
    s = warp_sum(s);
    if (lane == 0) a.ssq_out[rb * kRows + m0 + m] = s;
  }
}

template <int T>
__device__ void epi_qkv(const GemmArgs& a, const float* ys, int rb, int m0, int M, const EpiPre<T>& pre,
                        const int* spos) {
  constexpr int kE = EpiPre<T>::kE;
  const int half = a.hd >> 1;
  const int n0 = rb * kBlockRows;
  const int s = n0 < a.seg_end[0] ? 0 : (n0 < a.seg_end[1] ? 1 : 2);
  const int seg0 = s ? a.seg_end[s - 1] : 0;
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    const int i = threadIdx.x + e * kGemmThreads;
    const int m = i / kBlockRows, r = i - m * kBlockRows;
    if (m >= M || n0 + r >= a.N) continue;
    const int local = n0 + r - seg0;
    const int d = local % a.hd;
    const int b = (m0 + m) / a.rs.rps;
    const int pos = spos[m];
    if (s == 2) {
      const int kvh = local / a.hd;
      a.vc[(((size_t)b * a.nkv + kvh) * a.s_max + pos) * a.hd + d] = __float2bfloat16_rn(ys[i] + pre.v0[e]);
      continue;
    }
    if (d >= half) continue;
    const float x1 = ys[i] + pre.v0[e];
    const float x2 = ys[i + half] + pre.v1[e];
    const float2 cs = pre.cs[e];
    const float y1 = x1 * cs.x - x2 * cs.y;
    const float y2 = x2 * cs.x + x1 * cs.y;
    if (s == 0) {
      float* q = a.out + (size_t)(m0 + m) * a.out_ld + local;
      q[0] = y1;
      q[half] = y2;
    } else {
      const int kvh = local / a.hd;
      bf16* kp = a.kc + (((size_t)b * a.nkv + kvh) * a.s_max + pos) * a.hd + d;
      kp[0] = __float2bfloat16_rn(y1);
      kp[half] = __float2bfloat16_rn(y2);
    }
  }
}

__device__ void epi_swiglu(const GemmArgs& a, const float* ys, int rb, int m0, int M, int Tt) {
  for (int i = threadIdx.x; i < M * 64; i += kGemmThreads) {
    const int m = i >> 6, j = i & 63;
    const int f = rb * 64 + j;
    if (f >= a.N) continue;
    const float gte = ys[m * kBlockRows + j];
    const float up = ys[m * kBlockRows + 64 + j];
    act_store(a.frag_out, m0 + m, f, Tt, gte / (1.0f + expf(-gte)) * up, a.frag_umma);
  }
}

__device__ void epi_store(const GemmArgs& a, const float* ys, int rb, int m0, int M) {
  for (int i = threadIdx.x; i < M * kBlockRows; i += kGemmThreads) {
    const int m = i / kBlockRows, r = i - m * kBlockRows;
    const int n = rb * kBlockRows + r;
    if (n < a.N) a.out[(size_t)(m0 + m) * a.out_ld + n] = ys[i];
  }
}

__device__ __forceinline__ unsigned long long shfl_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// `finishers`: CTAs that run this epilogue in the launch (row blocks x row
// groups); the last to arrive writes the tokens of all rows of the forward.
__device__ void epi_argmax(const GemmArgs& a, const float* ys, int rb, int m0, int M, int finishers, int* s_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int m = warp; m < M; m += kGemmThreads / 32) {
    unsigned long long best = 0ull;
    bool bad = false;
    const int mb = (m0 + m) / a.rs.rps, mj = (m0 + m) - mb * a.rs.rps;
    const int lg_row = mj >= a.tok_skip ? mb * a.lg_stride + a.lg_off + mj - a.tok_skip : -1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = lane + 32 * j;
      const int n = rb * kBlockRows + r;
      if (n < a.N) {
        const float v = ys[m * kBlockRows + r];
        if (a.logits && lg_row >= 0) a.logits[(size_t)lg_row * a.N + n] = v;
        bad |= !isfinite(v);
        const unsigned long long k = argmax_key(v, n);
        best = k > best ? k : best;
      }
    }
    best = shfl_max_u64(best);
    if (__any_sync(0xffffffffu, bad) && lane == 0) report_err(a.err, kErrNonfinite);
    if (lane == 0) atomicMax(a.keys + m0 + m, best);
  }
  __threadfence();
  epi_sync();
  if (threadIdx.x == 0) *s_flag = (atomicAdd(a.done, 1) == finishers - 1);
  epi_sync();
  if (!*s_flag) return;
  __threadfence();
  if (threadIdx.x < a.rs.M) {
    const int m = threadIdx.x;
    const unsigned long long k = atomicExch(a.keys + m, 0ull);
    const int b = m / a.rs.rps, j = m - b * a.rs.rps;
    if (j >= a.tok_skip) a.tok_out[b * a.tok_stride + a.tok_off + j - a.tok_skip] = key_index(k);
  }
  if (threadIdx.x == 0) *a.done = 0;
}

}  // namespace
}  // namespace sf
