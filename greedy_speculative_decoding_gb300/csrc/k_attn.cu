// Embedding gather, GQA attention over the static KV cache, RoPE table.
//
// Attention is split over the cache ("flash decoding"): one work item is
// (sequence, KV head, 64-slot chunk). Its keys and values are contiguous in
// the cache, so one CTA brings them into shared memory with two bulk
// (TMA) copies completing on an mbarrier, and then serves every query that
// reads this KV head: all rows of the sequence times the query heads of the
// group. A query's scores come from one warp (two keys per lane, head
// dimension walked in a per-lane rotated order so the 16-byte shared reads
// never collide), with warp-shuffle max/sum; the chunk's partial result
// (max, sum of exponentials, unnormalised output) goes to scratch. A second
// kernel merges the chunks of every (row, head) in fixed chunk order.
//
// Chunk boundaries are fixed multiples of 64 slots and a row at position p
// reads slots 0..p, so a row's result does not depend on the other rows.
#include "sf_kernels.h"

namespace sf {

// ------------------------------------------------------------------ embedding
// x[m][:] = E[tok_m][:] in fp32, plus the per-128-feature sums of squares the
// next RMSNorm needs.
__global__ void __launch_bounds__(128) k_embed(const __grid_constant__ EmbedArgs a) {
  pdl_wait();
  pdl_launch_next();
  __shared__ float part[4];
  const int m = blockIdx.x, blk = blockIdx.y, i = threadIdx.x;
  const int b = m / a.rs.rps, j = m - b * a.rs.rps;
  int tok = a.rs.tok[b * a.rs.tok_stride + a.rs.tok_off + j];
  if (tok < 0 || tok >= a.vocab) {
    if (i == 0 && blk == 0) atomicOr(a.err, kErrCapacity);
    tok = 0;
  }
  const int n = blk * 128 + i;
  const float v = __bfloat162float(a.E[(size_t)tok * a.ld + n]);
  a.x[(size_t)m * a.H + n] = v;
  const float s = warp_sum(v * v);
  if ((i & 31) == 0) part[i >> 5] = s;
  __syncthreads();
  if (i == 0) a.ssq[blk * kRows + m] = ((part[0] + part[1]) + part[2]) + part[3];
}

cudaError_t launch_embed(const EmbedArgs& a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.rs.M, a.H / 128);
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_embed, a);
}

// ------------------------------------------------------------------ attention
constexpr uint32_t kWaitIters = 1u << 24;

template <int HD>
__global__ void __launch_bounds__(kAttnThreads) k_attn_chunks(const __grid_constant__ AttnArgs a) {
  constexpr int kUnits = HD / 8;            // 16-byte units per key row
  constexpr int kDims = HD / 32;            // output dims per lane
  __shared__ __align__(128) bf16 ks[kKvChunk * HD];
  __shared__ __align__(128) bf16 vs[kKvChunk * HD];
  __shared__ __align__(16) float qs[kAttnThreads / 32][HD];
  __shared__ __align__(8) uint64_t bar;

  pdl_wait();
  pdl_launch_next();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int group = a.nq / a.nkv;
  const int rps = a.rs.rps;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_proxy_async();
  }
  __syncthreads();

  // Work items: for each sequence b, nkv heads x chunks covering slots 0..p_last.
  int total = 0;
  for (int b = 0; b < a.B; ++b) {
    const int p_last = a.rs.pos_base[b] + a.rs.pos_off + rps - 1;
    total += a.nkv * (p_last / kKvChunk + 1);
  }
  uint32_t phase = 0;
  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    int b = 0, rest = item, nch = 0;
    for (; b < a.B; ++b) {
      const int p_last = a.rs.pos_base[b] + a.rs.pos_off + rps - 1;
      nch = p_last / kKvChunk + 1;
      if (rest < a.nkv * nch) break;
      rest -= a.nkv * nch;
    }
    const int kvh = rest / nch, c = rest - kvh * nch;
    const size_t off = (((size_t)b * a.nkv + kvh) * a.s_max + (size_t)c * kKvChunk) * HD;
    if (tid == 0) {
      fence_proxy_async();   // earlier generic reads of ks/vs before the async writes
      mbar_expect_tx(&bar, 2u * kKvChunk * HD * sizeof(bf16));
      bulk_g2s(ks, a.kc + off, kKvChunk * HD * sizeof(bf16), &bar);
      bulk_g2s(vs, a.vc + off, kKvChunk * HD * sizeof(bf16), &bar);
    }
    if (!mbar_wait(&bar, phase, kWaitIters)) {
      // The copy did not land: report, give it one more bounded chance, stop.
      if (tid == 0) atomicOr(a.err, kErrWait);
      mbar_wait(&bar, phase, kWaitIters);
      return;
    }
    phase ^= 1u;

    const int p0 = a.rs.pos_base[b] + a.rs.pos_off;
    for (int qi = warp; qi < rps * group; qi += kAttnThreads / 32) {
      const int j = qi / group, hh = qi - j * group;
      const int p = p0 + j;
      const int nk = min(kKvChunk, p - c * kKvChunk + 1);
      if (nk <= 0) continue;
      const int m = b * rps + j, h = kvh * group + hh;
      const float* qg = a.q + (size_t)m * a.nq * HD + (size_t)h * HD;
#pragma unroll
      for (int d = 0; d < kDims; ++d) qs[warp][lane + 32 * d] = qg[lane + 32 * d];
      __syncwarp();
      float s[2];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int kk = lane + 32 * half;
        float acc = 0.f;
        const uint4* krow = reinterpret_cast<const uint4*>(ks + kk * HD);
#pragma unroll
        for (int u0 = 0; u0 < kUnits; ++u0) {
          const int u = (u0 + lane) % kUnits;
          const uint4 kv = krow[u];
          const float4 qa = *reinterpret_cast<const float4*>(&qs[warp][8 * u]);
          const float4 qb = *reinterpret_cast<const float4*>(&qs[warp][8 * u + 4]);
          const float2 k01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kv.x));
          const float2 k23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kv.y));
          const float2 k45 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kv.z));
          const float2 k67 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kv.w));
          acc = fmaf(qa.x, k01.x, acc);
          acc = fmaf(qa.y, k01.y, acc);
          acc = fmaf(qa.z, k23.x, acc);
          acc = fmaf(qa.w, k23.y, acc);
          acc = fmaf(qb.x, k45.x, acc);
          acc = fmaf(qb.y, k45.y, acc);
          acc = fmaf(qb.z, k67.x, acc);
          acc = fmaf(qb.w, k67.y, acc);
        }
        s[half] = kk < nk ? acc * a.scale : -INFINITY;
      }
      const float mx = warp_max(fmaxf(s[0], s[1]));
      const float e0 = lane < nk ? expf(s[0] - mx) : 0.f;
      const float e1 = lane + 32 < nk ? expf(s[1] - mx) : 0.f;
      const float l = warp_sum(e0 + e1);
      float o[kDims];
#pragma unroll
      for (int d = 0; d < kDims; ++d) o[d] = 0.f;
      for (int kk = 0; kk < nk; ++kk) {
        const float pk = __shfl_sync(0xffffffffu, kk < 32 ? e0 : e1, kk & 31);
        const bf16* vrow = vs + kk * HD + lane * kDims;
        if (kDims == 4) {
          const uint2 vv = *reinterpret_cast<const uint2*>(vrow);
          const float2 v01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vv.x));
          const float2 v23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vv.y));
          o[0] = fmaf(pk, v01.x, o[0]);
          o[1] = fmaf(pk, v01.y, o[1]);
          o[2 % kDims] = fmaf(pk, v23.x, o[2 % kDims]);
          o[3 % kDims] = fmaf(pk, v23.y, o[3 % kDims]);
        } else {
          const float2 v01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(vrow));
          o[0] = fmaf(pk, v01.x, o[0]);
          o[1 % kDims] = fmaf(pk, v01.y, o[1 % kDims]);
        }
      }
      float* dst = a.part + (((size_t)m * a.nq + h) * a.n_kv_chunks + c) * (HD + 2);
#pragma unroll
      for (int d = 0; d < kDims; ++d) dst[lane * kDims + d] = o[d];
      if (lane == 0) {
        dst[HD] = mx;
        dst[HD + 1] = l;
      }
      __syncwarp();
    }
    __syncthreads();   // everyone is done with ks/vs before the next copy
  }
}

// out[m][h*hd + d] = sum_c o_c[d] e^(m_c - M) / sum_c l_c e^(m_c - M), chunks in order.
__global__ void k_attn_merge(const __grid_constant__ AttnArgs a) {
  pdl_wait();
  pdl_launch_next();
  const int m = blockIdx.x / a.nq, h = blockIdx.x - m * a.nq;
  const int d = threadIdx.x;
  const int p = row_pos(a.rs, m);
  const int nch = p / kKvChunk + 1;
  const float* src = a.part + ((size_t)m * a.nq + h) * a.n_kv_chunks * (a.hd + 2);
  float mx = -INFINITY;
  for (int c = 0; c < nch; ++c) mx = fmaxf(mx, src[(size_t)c * (a.hd + 2) + a.hd]);
  float l = 0.f, o = 0.f;
  for (int c = 0; c < nch; ++c) {
    const float* pc = src + (size_t)c * (a.hd + 2);
    const float w = expf(pc[a.hd] - mx);
    l = fmaf(pc[a.hd + 1], w, l);
    o = fmaf(pc[d], w, o);
  }
  a.out[(size_t)m * a.nq * a.hd + (size_t)h * a.hd + d] = o / l;
}

cudaError_t launch_attention(const AttnArgs& a, int num_sms, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  // Enough CTAs for the largest item count this launch can see (the count
  // itself lives on the device): B * nkv * chunks of the whole cache, capped.
  const int max_items = a.B * a.nkv * a.n_kv_chunks;
  cfg.gridDim = dim3(max(1, min(max_items, 2 * num_sms)));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e;
  if (a.hd == 128) e = cudaLaunchKernelEx(&cfg, k_attn_chunks<128>, a);
  else if (a.hd == 64) e = cudaLaunchKernelEx(&cfg, k_attn_chunks<64>, a);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg2 = {};
  cfg2.gridDim = dim3(a.rs.M * a.nq);
  cfg2.blockDim = dim3(a.hd);
  cfg2.stream = st;
  cfg2.attrs = attr;
  cfg2.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg2, k_attn_merge, a);
}

// ------------------------------------------------------------------ RoPE table
// table[p][i] = (cos(p * theta^(-2i/hd)), sin(...)), computed in double.
__global__ void k_rope_table(float2* t, int s_max, int hd, double theta) {
  const int half = hd / 2;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= s_max * half) return;
  const int p = idx / half, i = idx - p * half;
  const double inv = pow(theta, -2.0 * i / hd);
  double sn, cs;
  sincos((double)p * inv, &sn, &cs);
  t[idx] = make_float2((float)cs, (float)sn);
}

cudaError_t launch_rope_table(float2* table, int s_max, int hd, float theta, cudaStream_t st) {
  const int n = s_max * (hd / 2);
  k_rope_table<<<(n + 255) / 256, 256, 0, st>>>(table, s_max, hd, (double)theta);
  return cudaGetLastError();
}

}  // namespace sf
