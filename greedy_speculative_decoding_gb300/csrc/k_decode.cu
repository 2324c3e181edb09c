// A whole decoder forward of at most four token rows in one persistent
// kernel: the decode step of the draft model (one row per sequence, two in a
// round's first step) without a launch per projection.
//
// One CTA of 512 threads per SM, launched cooperatively so that every CTA is
// resident; the phases of a layer are separated by grid barriers:
//   A  every CTA: rms(x) of each row -> x * g (ln1) in shared memory;
//      q, k, v projections (+ bias, RoPE; keys and values appended to the
//      cache, queries to scratch)
//   B  attention partials: work item = (sequence, KV head, range of R
//      64-slot chunks), one CTA per item: scores, an online softmax over the
//      range, the unnormalised output with its running max and sum; the
//      last item of a (sequence, KV head) to finish (an arrival counter)
//      merges the ranges of its rows and heads in range order
//   C  O projection + residual
//   D  every CTA: rms(x) -> x * g (ln2); gate and up projections + SwiGLU
//   E  down projection + residual
// and after the last layer the final norm's input for the LM head (fragment
// order, x * g, and the per-128-feature sums of squares), which the LM-head
// kernel reads as it does after the per-projection kernels.
//
// Projections: a CTA owns a contiguous range of output rows (pairs of rows:
// a query or key dimension and its RoPE partner, two value rows, a gate row
// and its up row, or two rows of O / down). When it owns at least 16 pairs
// each warp takes whole pairs; otherwise 16 / pairs warps share a pair, each
// one contiguous slice of K, and the slices are added in order. Lane l of a
// warp reads 16 bytes of a weight row at k = 8l, 8l + 256, ... and multiplies
// them with every token row in fp32; the 32 lane sums are added by a fixed
// butterfly. The arithmetic of an output element therefore depends on the
// matrix shape and the SM count only, never on the other rows of the launch.
//
// The barrier is a counter and a generation word: the last CTA to arrive
// resets the counter and advances the generation; the others poll the
// generation with a bounded number of polls, after which they set the
// engine's error bit and end (the results are then unspecified; every other
// CTA ends at its next barrier the same way).
#include "sf_kernels.h"

namespace sf {

namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr uint32_t kDecBarrierPolls = 1u << 20;

// Weights are read-only for the kernel's lifetime: a non-volatile load the
// compiler may batch and hoist.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void st_relaxed_u32(unsigned* p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid barrier (see the file comment). `bar` = {arrival count, generation}.
// Returns false (in every thread of the CTA) when the wait gave up; the
// kernel then ends at once, so a failed barrier costs one poll limit.
__device__ bool grid_barrier(unsigned* bar, int* err, bool report_expiry = false) {
  __shared__ int s_fail;
  __syncthreads();
  if (threadIdx.x == 0) {
    s_fail = 0;
    // Test hook (as in the GEMM kernels): report an expired wait, then wait normally.
    if (report_expiry && blockIdx.x == 0) report_err(err, kErrWait);
    // Arrival releases this CTA's writes (ordered before it by the block
    // barrier); the last arriver acquires everyone's through the counter's
    // read-modify-write chain and releases them with the new generation.
    const unsigned g = ld_acquire_u32(bar + 1);
    const unsigned arrived = atom_add_acq_rel(bar, 1u);
    if (arrived == gridDim.x - 1) {
      st_relaxed_u32(bar, 0u);
      st_release_u32(bar + 1, g + 1);
    } else {
      uint32_t polls = 0;
      while (ld_acquire_u32(bar + 1) == g) {
        if (++polls > kDecBarrierPolls) {
          report_err(err, kErrWait);
          s_fail = 1;
          break;
        }
        __nanosleep(20);
      }
    }
  }
  __syncthreads();
  return s_fail == 0;
}

// L2 prefetch of `bytes` (a multiple of 16) from a 16-byte aligned address.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// This CTA's share [p0, p1) of npairs pairs.
__device__ __forceinline__ void cta_pairs(int npairs, int* p0, int* p1) {
  *p0 = (int)((long)npairs * blockIdx.x / gridDim.x);
  *p1 = (int)((long)npairs * (blockIdx.x + 1) / gridDim.x);
}

// Eight bf16 weights (one 16-byte load) times eight fp32 activations, added
// to acc in element order.
__device__ __forceinline__ float dot8(uint4 w, float4 a, float4 b, float acc) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
  const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc = fmaf(__uint_as_float(u[i] << 16), x[2 * i], acc);
    acc = fmaf(__uint_as_float(u[i] & 0xffff0000u), x[2 * i + 1], acc);
  }
  return acc;
}

// One warp: the dot products of two weight rows (w0, w1) with MR activation
// rows xs[m * xld + k] over k in [k0, k1) (multiples of 8), lane sums added by
// a butterfly; every lane ends with all 2 x MR sums.
template <int MR>
__device__ __forceinline__ void warp_dot2(const bf16* w0, const bf16* w1, const float* xs, int xld, int k0, int k1,
                                          float (&s0)[MR], float (&s1)[MR]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 0; m < MR; ++m) s0[m] = s1[m] = 0.f;
  int k = k0 + 8 * lane;
  // Four loads of each row in flight, then their products.
  for (; k + 768 < k1; k += 1024) {
    uint4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      a[u] = ldg_stream(w0 + k + 256 * u);
      b[u] = ldg_stream(w1 + k + 256 * u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        const float4 xa = *reinterpret_cast<const float4*>(xs + m * xld + k + 256 * u);
        const float4 xb = *reinterpret_cast<const float4*>(xs + m * xld + k + 256 * u + 4);
        s0[m] = dot8(a[u], xa, xb, s0[m]);
        s1[m] = dot8(b[u], xa, xb, s1[m]);
      }
  }
#pragma unroll 4
  for (; k < k1; k += 256) {
    const uint4 a = ldg_stream(w0 + k), b = ldg_stream(w1 + k);
#pragma unroll
    for (int m = 0; m < MR; ++m) {
      const float4 xa = *reinterpret_cast<const float4*>(xs + m * xld + k);
      const float4 xb = *reinterpret_cast<const float4*>(xs + m * xld + k + 4);
      s0[m] = dot8(a, xa, xb, s0[m]);
      s1[m] = dot8(b, xa, xb, s1[m]);
    }
  }
#pragma unroll
  for (int m = 0; m < MR; ++m)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s0[m] += __shfl_xor_sync(0xffffffffu, s0[m], o);
      s1[m] += __shfl_xor_sync(0xffffffffu, s1[m], o);
    }
}

// The projection phase of one CTA: pairs [0, npairs) of the matrix are split
// into contiguous ranges over the grid; rows(p, &w0, &w1) gives pair p's two
// weight rows, epi(p, m, y0, y1) consumes row m's two results. `red` is
// shared scratch of kDecWarps * 2 * MR floats.
template <int MR, typename Rows, typename Epi>
__device__ __forceinline__ void gemv_phase(int npairs, int K, const float* xs, int xld, float* red, Rows rows,
                                           Epi epi) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int p0, p1;
  cta_pairs(npairs, &p0, &p1);
  const int np = p1 - p0;
  if (np <= 0) return;
  if (np >= kDecWarps) {
    for (int p = p0 + warp; p < p1; p += kDecWarps) {
      const bf16 *w0, *w1;
      rows(p, &w0, &w1);
      float s0[MR], s1[MR];
      warp_dot2<MR>(w0, w1, xs, xld, 0, K, s0, s1);
#pragma unroll
      for (int m = 0; m < MR; ++m)
        if (lane == m) epi(p, m, s0[m], s1[m]);
    }
    return;
  }
  // Fewer pairs than warps: wpp warps per pair, each a contiguous slice of K.
  const int wpp = kDecWarps / np;
  const int pi = warp / wpp, part = warp - pi * wpp;
  const int k8 = K / 8;
  if (pi < np) {
    const int ka = 8 * (int)((long)k8 * part / wpp), kb = 8 * (int)((long)k8 * (part + 1) / wpp);
    const bf16 *w0, *w1;
    rows(p0 + pi, &w0, &w1);
    float s0[MR], s1[MR];
    warp_dot2<MR>(w0, w1, xs, xld, ka, kb, s0, s1);
    if (lane == 0)
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        red[(warp * MR + m) * 2] = s0[m];
        red[(warp * MR + m) * 2 + 1] = s1[m];
      }
  }
  __syncthreads();
  if (warp < np && lane < MR) {
    const int m = lane;
    float y0 = 0.f, y1 = 0.f;
    for (int q = 0; q < wpp; ++q) {
      y0 += red[((warp * wpp + q) * MR + m) * 2];
      y1 += red[((warp * wpp + q) * MR + m) * 2 + 1];
    }
    epi(p0 + warp, m, y0, y1);
  }
  __syncthreads();
}

// L2 prefetch of the weight rows of this CTA's pairs (K bf16 each), one
// pair per thread.
template <typename Rows>
__device__ __forceinline__ void prefetch_pairs(int npairs, int K, Rows rows) {
  int p0, p1;
  cta_pairs(npairs, &p0, &p1);
  for (int p = p0 + (int)threadIdx.x; p < p1; p += kDecThreads) {
    const bf16 *w0, *w1;
    rows(p, &w0, &w1);
    prefetch_l2(w0, (uint32_t)K * 2);
    prefetch_l2(w1, (uint32_t)K * 2);
  }
}

// x (global, MR rows of H) -> xs = x * rinv * gain in shared memory, every CTA
// the same way: warp m sums the squares of row m (lane-strided, butterfly).
template <int MR>
__device__ __forceinline__ void norm_rows(const float* x, int H, const bf16* gain, float eps, float* xs,
                                          float* s_rinv) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < MR) {
    float sq = 0.f;
    for (int i = lane; i < H; i += 32) {
      const float v = x[warp * H + i];
      sq = fmaf(v, v, sq);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0) s_rinv[warp] = 1.0f / sqrtf(sq / H + eps);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < MR * H; i += kDecThreads) {
    const int m = i / H, n = i - m * H;
    xs[i] = x[i] * s_rinv[m] * __bfloat162float(gain[n]);
  }
  __syncthreads();
}

}  // namespace

// Pair -> weight rows of each projection of layer lw (see gemv_phase).
struct QkvRows {
  const DecLayer* lw;
  int H, hd, nqp, nkp;
  __device__ void operator()(int p, const bf16** w0, const bf16** w1) const {
    const int half = hd / 2;
    if (p < nqp) {
      const int h = p / half, d = p - h * half;
      *w0 = lw->wq + (size_t)(h * hd + d) * H;
      *w1 = lw->wq + (size_t)(h * hd + d + half) * H;
    } else if (p < nqp + nkp) {
      const int p2 = p - nqp, h = p2 / half, d = p2 - h * half;
      *w0 = lw->wk + (size_t)(h * hd + d) * H;
      *w1 = lw->wk + (size_t)(h * hd + d + half) * H;
    } else {
      const int r = 2 * (p - nqp - nkp);
      *w0 = lw->wv + (size_t)r * H;
      *w1 = lw->wv + (size_t)(r + 1) * H;
    }
  }
};
struct PairRows {   // rows 2p and 2p + 1 of w (row length K)
  const bf16* w;
  int K;
  __device__ void operator()(int p, const bf16** w0, const bf16** w1) const {
    *w0 = w + (size_t)(2 * p) * K;
    *w1 = w + (size_t)(2 * p + 1) * K;
  }
};
struct GateUpRows {   // gate row f and up row f
  const bf16 *wg, *wu;
  int H;
  __device__ void operator()(int f, const bf16** w0, const bf16** w1) const {
    *w0 = wg + (size_t)f * H;
    *w1 = wu + (size_t)f * H;
  }
};

template <int MR>
__global__ void __launch_bounds__(kDecThreads, 1) k_decode(const __grid_constant__ DecArgs a) {
  extern __shared__ float dsm[];
  __shared__ float s_rinv[4];
  __shared__ int s_pos[4], s_b[4];
  __shared__ float red[kDecWarps * 2 * 4];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, hd = a.hd, half = hd / 2, nq = a.nq, nkv = a.nkv, F = a.F;
  const int QD = nq * hd, KVD = nkv * hd, group = nq / nkv;
  const int rps = a.rs.rps;
  const int nqp = QD / 2, nkp = KVD / 2, nqkv = nqp + nkp + KVD / 2;
  // Launch timeline (tracing on): phase k of the kernel stamps its start in
  // timeline slot trace_id + k, both entries (the time a phase adds to the
  // chain is the gap to the next slot's stamp).
  auto stamp = [&](int k) {
    if (a.rs.trace && blockIdx.x == 0 && tid == 0) {
      unsigned long long t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      const int slot = (a.rs.trace_id + k) % kTraceSlots;
      a.rs.trace[2 * slot] = t;
      a.rs.trace[2 * slot + 1] = t;
    }
  };
  // Weights are never written by the preceding kernels: layer 0's q, k, v
  // rows start towards L2 before the wait.
  trace_mark(a.rs, 0);
  prefetch_pairs(nqkv, H, QkvRows{&a.layers[0], H, hd, nqp, nkp});
  pdl_wait();
  trace_mark(a.rs, 1);
  if (tid < MR) {
    s_pos[tid] = row_slot(a.rs, tid);
    s_b[tid] = tid / rps;
  }
  // Embedding rows (bf16 -> fp32 residual stream).
  for (int i = blockIdx.x * kDecThreads + tid; i < MR * H; i += gridDim.x * kDecThreads) {
    const int m = i / H, n = i - m * H;
    const int b = m / rps, j = m - b * rps;
    const int tok = a.rs.tok[b * a.rs.tok_stride + a.rs.tok_off + j];
    float v = 0.f;
    if (tok >= 0 && tok < a.vocab) v = __bfloat162float(a.embed[(size_t)tok * a.embed_ld + n]);
    else if (n == 0) report_err(a.err, kErrCapacity);
    a.x[i] = v;
  }
  if (!grid_barrier(a.bar, a.err, a.expire_first_wait != 0)) return;

  const size_t seq_elems = (size_t)nkv * a.s_max * hd;
  const size_t layer_elems = 2 * (size_t)a.B * seq_elems;
  for (int l = 0; l < a.L; ++l) {
    const DecLayer& lw = a.layers[l];
    bf16* kc = a.kv + (size_t)l * layer_elems;
    bf16* vc = kc + layer_elems / 2;
    stamp(1 + 5 * l);
    // ---- A: q, k, v; this layer's O, gate/up and down rows start towards L2
    const PairRows o_rows{lw.wo, QD}, d_rows{lw.wd, F};
    const GateUpRows gu_rows{lw.wg, lw.wu, H};
    prefetch_pairs(H / 2, QD, o_rows);
    norm_rows<MR>(a.x, H, lw.ln1, a.eps, dsm, s_rinv);
    {
      const QkvRows rows{&lw, H, hd, nqp, nkp};
      auto epi = [&](int p, int m, float y0, float y1) {
        const int b = s_b[m], pos = s_pos[m];
        if (p < nqp + nkp) {
          const bool isq = p < nqp;
          const int p2 = isq ? p : p - nqp, h = p2 / half, d = p2 - h * half;
          const int r0 = h * hd + d, r1 = r0 + half;
          const bf16* bias = isq ? lw.bq : lw.bk;
          if (bias) {
            y0 += __bfloat162float(bias[r0]);
            y1 += __bfloat162float(bias[r1]);
          }
          const float2 cs = a.rope[(size_t)(pos - tree_gap(a.rs, m % rps)) * half + d];
          const float z0 = y0 * cs.x - y1 * cs.y, z1 = y1 * cs.x + y0 * cs.y;
          if (isq) {
            a.q[(size_t)m * QD + r0] = z0;
            a.q[(size_t)m * QD + r1] = z1;
          } else {
            bf16* kp = kc + ((size_t)b * nkv + h) * a.s_max * hd + (size_t)pos * hd;
            kp[d] = __float2bfloat16_rn(z0);
            kp[d + half] = __float2bfloat16_rn(z1);
          }
        } else {
          const int r = 2 * (p - nqp - nkp), h = r / hd, d = r - h * hd;
          if (lw.bv) {
            y0 += __bfloat162float(lw.bv[r]);
            y1 += __bfloat162float(lw.bv[r + 1]);
          }
          bf16* vp = vc + ((size_t)b * nkv + h) * a.s_max * hd + (size_t)pos * hd;
          vp[d] = __float2bfloat16_rn(y0);
          vp[d + 1] = __float2bfloat16_rn(y1);
        }
      };
      gemv_phase<MR>(nqkv, H, dsm, H, red, rows, epi);
    }
    if (!grid_barrier(a.bar, a.err)) return;

    stamp(2 + 5 * l);
    // The gate/up and down rows stream towards L2 while attention, which
    // moves little, runs.
    prefetch_pairs(F, H, gu_rows);
    prefetch_pairs(H / 2, F, d_rows);
    // ---- B: attention partials. Shared memory: keys (row pitch hd + 1, so
    // the 64 threads of a score row read 64 different banks) and values of
    // one chunk in fp32, the queries of the item, the chunk's probabilities.
    {
      const int nqv = rps * group;
      const int KP = hd + 1;
      float* ks = dsm;                        // [64][KP]
      float* vs = ks + 64 * KP;               // [64][hd]
      float* qs = vs + 64 * hd;               // [nqv][hd]
      float* ps = qs + nqv * hd;              // [nqv][64]
      float* mrun = ps + nqv * 64;            // [nqv]
      float* lrun = mrun + nqv;               // [nqv]
      float* alph = lrun + nqv;               // [nqv] this chunk's rescale factor; 1 / sum in the merge
      float* wts = alph + nqv;                // [nqv][n_ranges] the merge's range weights
      const int B = MR / rps;
      // Items: for each sequence and KV head, ranges of R chunks up to the
      // chunk of its last row.
      int total = 0;
      for (int b = 0; b < B; ++b) total += nkv * ((s_pos[b * rps + rps - 1] / 64) / a.R + 1);
      for (int item = blockIdx.x; item < total; item += gridDim.x) {
        int b = 0, rest = item;
        for (; b < B; ++b) {
          const int n = nkv * ((s_pos[b * rps + rps - 1] / 64) / a.R + 1);
          if (rest < n) break;
          rest -= n;
        }
        const int nr = (s_pos[b * rps + rps - 1] / 64) / a.R + 1;
        const int kvh = rest / nr, r = rest - kvh * nr;
        const int p_first = s_pos[b * rps], p_last = s_pos[b * rps + rps - 1];
        const int c0 = r * a.R, c1 = min(c0 + a.R, p_last / 64 + 1);
        for (int i = tid; i < nqv * hd; i += kDecThreads) {
          const int qv = i / hd, d = i - qv * hd;
          const int j = qv / group, hh = qv - j * group;
          qs[i] = a.q[(size_t)(b * rps + j) * QD + (kvh * group + hh) * hd + d];
        }
        if (tid < nqv) {
          mrun[tid] = -INFINITY;
          lrun[tid] = 0.f;
        }
        // Thread t owns output elements t, t + 512, ... of [nqv][hd].
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        const bf16* kbase = kc + ((size_t)b * nkv + kvh) * a.s_max * hd;
        const bf16* vbase = vc + ((size_t)b * nkv + kvh) * a.s_max * hd;
        for (int c = c0; c < c1; ++c) {
          const int nvalid = min(64, p_last - c * 64 + 1);
          __syncthreads();   // the previous chunk's keys, values and probabilities are consumed
          for (int i = tid; i < nvalid * hd / 8; i += kDecThreads) {
            const int s = i / (hd / 8), u = i - s * (hd / 8);
            const uint4 kv = *reinterpret_cast<const uint4*>(kbase + (size_t)(c * 64 + s) * hd + 8 * u);
            const uint4 vv = *reinterpret_cast<const uint4*>(vbase + (size_t)(c * 64 + s) * hd + 8 * u);
            const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w}, vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              ks[s * KP + 8 * u + 2 * e] = __uint_as_float(kw[e] << 16);
              ks[s * KP + 8 * u + 2 * e + 1] = __uint_as_float(kw[e] & 0xffff0000u);
              vs[s * hd + 8 * u + 2 * e] = __uint_as_float(vw[e] << 16);
              vs[s * hd + 8 * u + 2 * e + 1] = __uint_as_float(vw[e] & 0xffff0000u);
            }
          }
          __syncthreads();
          // Scores: element (qv, s) by thread qv * 64 + s (and + 512).
          for (int i = tid; i < nqv * 64; i += kDecThreads) {
            const int qv = i >> 6, s = i & 63;
            const int j = qv / group;
            const int last = p_first + j;   // row j sees slots <= its own position's slot
            float sc = -INFINITY;
            if (s < nvalid && c * 64 + s <= last) {
              float acc = 0.f;
              const float* qr = qs + qv * hd;
              const float* kr = ks + s * KP;
              for (int d = 0; d < hd; ++d) acc = fmaf(qr[d], kr[d], acc);
              sc = acc * a.scale;
            }
            ps[i] = sc;
          }
          __syncthreads();
          // Online softmax per query row: warp qv.
          if (warp < nqv) {
            const int qv = warp;
            float mx = -INFINITY;
            for (int s = lane; s < 64; s += 32) mx = fmaxf(mx, ps[qv * 64 + s]);
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
            const float m_old = mrun[qv];
            const float m_new = fmaxf(m_old, mx);
            const float alpha = m_new == -INFINITY ? 1.f : expf(m_old - m_new);
            float lsum = 0.f;
            for (int s = lane; s < 64; s += 32) {
              const float sc = ps[qv * 64 + s];
              const float p = sc == -INFINITY ? 0.f : expf(sc - m_new);
              ps[qv * 64 + s] = p;
              lsum += p;
            }
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o2);
            __syncwarp();
            if (lane == 0) {
              lrun[qv] = lrun[qv] * alpha + lsum;
              mrun[qv] = m_new;
              alph[qv] = alpha;
            }
          }
          __syncthreads();
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = tid + e * kDecThreads;
            if (i < nqv * hd) {
              const int qv = i / hd, d = i - qv * hd;
              float acc = 0.f;
              for (int s = 0; s < nvalid; ++s) acc = fmaf(ps[qv * 64 + s], vs[s * hd + d], acc);
              o[e] = o[e] * alph[qv] + acc;
            }
          }
        }
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = tid + e * kDecThreads;
          if (i < nqv * hd) {
            const int qv = i / hd, d = i - qv * hd;
            const int j = qv / group, hh = qv - j * group;
            const int m = b * rps + j, h = kvh * group + hh;
            if (c0 * 64 > p_first + j) continue;   // the row sees no slot of this range
            float* dst = a.part + (((size_t)m * nq + h) * a.n_ranges + r) * (hd + 2);
            dst[d] = o[e];
            if (d == 0) {
              dst[hd] = mrun[qv];
              dst[hd + 1] = lrun[qv];
            }
          }
        }
        // The last item of (b, kvh) to finish merges its ranges: every
        // (row, head) of the KV head, ranges in order, into the O
        // projection's input (over the queries, which nothing reads again).
        __shared__ int s_last;
        __syncthreads();
        if (tid == 0) {
          const unsigned done = atom_add_acq_rel(a.cnt + b * nkv + kvh, 1u);
          s_last = done == (unsigned)(nr - 1);
          if (s_last) st_relaxed_u32(a.cnt + b * nkv + kvh, 0u);
        }
        __syncthreads();
        if (s_last) {
          // Warp qv: the weights exp(m_r - max) / sum of every range of row
          // and head qv (lanes over ranges), into shared memory (the
          // probability scratch); then every output element sums its
          // ranges' values with those weights, in range order.
          const int nrmax = (p_last / 64) / a.R + 1;
          if (warp < nqv) {
            const int qv = warp, j = qv / group, hh = qv - j * group;
            const int m = b * rps + j, h = kvh * group + hh;
            const int nparts = (s_pos[m] / 64) / a.R + 1;
            const float* src = a.part + ((size_t)m * nq + h) * a.n_ranges * (hd + 2);
            float mx = -INFINITY;
            for (int r2 = lane; r2 < nparts; r2 += 32) mx = fmaxf(mx, src[r2 * (hd + 2) + hd]);
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
            float lsum = 0.f;
            for (int r2 = lane; r2 < nparts; r2 += 32) {
              const float w = expf(src[r2 * (hd + 2) + hd] - mx);
              wts[qv * nrmax + r2] = w;
              lsum = fmaf(w, src[r2 * (hd + 2) + hd + 1], lsum);
            }
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o2);
            if (lane == 0) alph[qv] = 1.0f / lsum;
          }
          __syncthreads();
          for (int i = tid; i < nqv * hd; i += kDecThreads) {
            const int qv = i / hd, d = i - qv * hd;
            const int j = qv / group, hh = qv - j * group;
            const int m = b * rps + j, h = kvh * group + hh;
            const int nparts = (s_pos[m] / 64) / a.R + 1;
            const float* src = a.part + ((size_t)m * nq + h) * a.n_ranges * (hd + 2) + d;
            float acc = 0.f;
#pragma unroll 8
            for (int r2 = 0; r2 < nparts; ++r2) acc = fmaf(wts[qv * nrmax + r2], src[r2 * (hd + 2)], acc);
            a.q[(size_t)m * QD + h * hd + d] = acc * alph[qv];
          }
        }
        __syncthreads();   // the running max and sum are reset by the next item
      }
    }
    if (!grid_barrier(a.bar, a.err)) return;

    stamp(3 + 5 * l);
    // ---- C: O + residual over the merged attention output.
    {
      float* as = dsm;   // [MR][QD]
      for (int i = tid; i < MR * QD; i += kDecThreads) as[i] = a.q[i];
      __syncthreads();
      auto epi = [&](int p, int m, float y0, float y1) {
        float* xr = a.x + (size_t)m * H + 2 * p;
        xr[0] += y0;
        xr[1] += y1;
      };
      gemv_phase<MR>(H / 2, QD, as, QD, red, o_rows, epi);
    }
    if (!grid_barrier(a.bar, a.err)) return;

    stamp(4 + 5 * l);
    // ---- D: gate / up + SwiGLU; the next layer's q, k, v rows start towards L2
    if (l + 1 < a.L) prefetch_pairs(nqkv, H, QkvRows{&a.layers[l + 1], H, hd, nqp, nkp});
    norm_rows<MR>(a.x, H, lw.ln2, a.eps, dsm, s_rinv);
    {
      auto epi = [&](int f, int m, float g, float u) { a.h[(size_t)m * F + f] = g / (1.0f + expf(-g)) * u; };
      gemv_phase<MR>(F, H, dsm, H, red, gu_rows, epi);
    }
    if (!grid_barrier(a.bar, a.err)) return;

    stamp(5 + 5 * l);
    // ---- E: down + residual
    for (int i = tid; i < MR * F; i += kDecThreads) dsm[i] = a.h[i];
    __syncthreads();
    {
      auto epi = [&](int p, int m, float y0, float y1) {
        float* xr = a.x + (size_t)m * H + 2 * p;
        xr[0] += y0;
        xr[1] += y1;
      };
      gemv_phase<MR>(H / 2, F, dsm, F, red, d_rows, epi);
    }
    if (!grid_barrier(a.bar, a.err)) return;
  }
  pdl_launch_next();

  // ---- the LM head's input: x * g (final norm) in fragment order, and the
  // sums of squares of every 128 features of x.
  const int T4 = (a.rs.M + 3) / 4;
  for (int i = blockIdx.x * kDecThreads + tid; i < MR * H; i += gridDim.x * kDecThreads) {
    const int m = i / H, n = i - m * H;
    act_store(a.frag, m, n, T4, a.x[i] * __bfloat162float(a.norm[n]), false);
  }
  for (int gq = blockIdx.x; gq < (H / 128) * MR; gq += gridDim.x) {
    const int g = gq / MR, m = gq - g * MR;
    if (warp == 0) {
      float sq = 0.f;
      for (int i = lane; i < 128; i += 32) {
        const float v = a.x[(size_t)m * H + 128 * g + i];
        sq = fmaf(v, v, sq);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      if (lane == 0) a.ssq[g * kRows + m] = sq;
    }
  }
}

// Shared memory of one CTA: the largest of the phases' needs.
int decode_smem_bytes(int MR, int H, int QD, int F, int hd, int group, int rps, int n_ranges) {
  int f = MR * H;
  f = max(f, MR * QD);
  f = max(f, MR * F);
  const int nqv = rps * group;
  f = max(f, 64 * (hd + 1) + 64 * hd + nqv * hd + nqv * 64 + 3 * nqv + nqv * n_ranges);
  return f * 4;
}

cudaError_t launch_decode(const DecArgs& a, int num_sms, cudaStream_t st) {
  const int MR = a.rs.M;
  if (MR < 1 || MR > 4 || a.hd % 8 || a.H % 128 || a.F % 8 || (a.nq * a.hd) % 8) return cudaErrorInvalidValue;
  const int smem = decode_smem_bytes(MR, a.H, a.nq * a.hd, a.F, a.hd, a.nq / a.nkv, a.rs.rps, a.n_ranges);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (MR) {
    case 1: return cudaLaunchKernelEx(&cfg, k_decode<1>, a);
    case 2: return cudaLaunchKernelEx(&cfg, k_decode<2>, a);
    case 3: return cudaLaunchKernelEx(&cfg, k_decode<3>, a);
    default: return cudaLaunchKernelEx(&cfg, k_decode<4>, a);
  }
}

cudaError_t decode_init(int max_smem) {
  const void* fns[] = {reinterpret_cast<const void*>(k_decode<1>), reinterpret_cast<const void*>(k_decode<2>),
                       reinterpret_cast<const void*>(k_decode<3>), reinterpret_cast<const void*>(k_decode<4>)};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace sf
