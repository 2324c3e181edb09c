// Embedding gather, GQA attention over the static KV cache, RoPE table.
//
// Attention is split over the cache ("flash decoding"): one work item is
// (sequence, KV head, 64-slot chunk). Its keys and values are contiguous in
// the cache; one warp brings them into padded shared-memory rows with bulk
// (TMA) copies completing on an mbarrier, and the CTA then serves every
// query that reads this KV head (all rows of the sequence times the query
// heads of the group) on the tensor cores, 16 queries per warp. The chunk's
// partial result (row max, sum of exponentials, unnormalised output) goes to
// scratch; a second kernel merges the chunks of every (row, head) in fixed
// chunk order.
//
// Chunk boundaries are fixed multiples of 64 slots and a row at position p
// reads slots 0..p, so a row's result does not depend on the other rows.
#include "sf_kernels.h"

namespace sf {

// ------------------------------------------------------------------ embedding
// x[m][:] = E[tok_m][:] in fp32, plus the per-128-feature sums of squares the
// next RMSNorm needs.
__global__ void __launch_bounds__(128) k_embed(const __grid_constant__ EmbedArgs a) {
  trace_mark(a.rs, 0);
  pdl_wait();
  trace_mark(a.rs, 1);
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

__device__ __forceinline__ void ldsm_x2_trans(uint32_t& r0, uint32_t& r1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void split_bf16x2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const bf16 hx = __float2bfloat16_rn(x), hy = __float2bfloat16_rn(y);
  hi = pack_bf16x2(hx, hy);
  lo = pack_bf16x2(__float2bfloat16_rn(x - __bfloat162float(hx)), __float2bfloat16_rn(y - __bfloat162float(hy)));
}

// One work item = (sequence b, KV head, 64-slot chunk c). Each warp takes a
// tile of 16 queries (rows of the sequence x query heads of the group):
//   S = Q K^T with mma.sync m16n8k16 (Q as an fp32-accurate bf16 hi+lo pair,
//   the head dimension walked in an order that makes each thread's key
//   fragment one 8-byte shared load), masked to the slots each row may see,
//   row max / exp / row sum on the accumulators (quad shuffles), then
//   O = P V with P (hi+lo) taken straight from the S accumulators and V
//   fragments from ldmatrix.trans.
template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 2) k_attn_chunks(const __grid_constant__ AttnArgs a) {
  constexpr int KP = HD * 2 + 32;   // key row pitch: 8-bank shift per row for the 8-byte fragment loads
  constexpr int VP = HD * 2 + 16;   // value row pitch: 4-bank shift per row for ldmatrix
  constexpr int KS = HD / 16;       // k-steps over the head dimension
  constexpr int NT = HD / 8;        // n-tiles of the output
  __shared__ __align__(128) unsigned char ks[kKvChunk * KP];
  __shared__ __align__(128) unsigned char vs[kKvChunk * VP];
  __shared__ __align__(8) uint64_t bar;

  trace_mark(a.rs, 0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c4 = lane & 3;
  const int group = a.nq / a.nkv;
  const int rps = a.rs.rps;
  const int Mq = rps * group;
  if (tid == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // The lengths were written by kernels that finished before the preceding
  // one started, so they (and the cache slots below this pass's first
  // position) can be read before waiting on the preceding kernel.
  int total = 0;
  for (int b = 0; b < a.B; ++b) {
    const int p_last = a.rs.pos_base[b] + a.rs.pos_off + rps - 1;
    total += a.nkv * (p_last / kKvChunk + 1);
  }
  auto locate = [&](int item, int& b, int& kvh, int& c) {
    int rest = item, nch = 0;
    for (b = 0; b < a.B; ++b) {
      const int p_last = a.rs.pos_base[b] + a.rs.pos_off + rps - 1;
      nch = p_last / kKvChunk + 1;
      if (rest < a.nkv * nch) break;
      rest -= a.nkv * nch;
    }
    kvh = rest / nch;
    c = rest - kvh * nch;
  };
  auto issue = [&](int b, int kvh, int c) {
    const size_t off = (((size_t)b * a.nkv + kvh) * a.s_max + (size_t)c * kKvChunk) * HD;
    if (warp == 0) {
      if (lane == 0) mbar_expect_tx(&bar, 2u * kKvChunk * HD * sizeof(bf16));
      __syncwarp();
      fence_proxy_async();   // earlier generic accesses of ks/vs before the async writes
      for (int r = lane; r < kKvChunk; r += 32) {
        bulk_g2s(ks + r * KP, a.kc + off + (size_t)r * HD, HD * sizeof(bf16), &bar);
        bulk_g2s(vs + r * VP, a.vc + off + (size_t)r * HD, HD * sizeof(bf16), &bar);
      }
    }
  };
  bool issued = false;
  if ((int)blockIdx.x < total) {
    int b, kvh, c;
    locate(blockIdx.x, b, kvh, c);
    if ((c + 1) * kKvChunk <= a.rs.pos_base[b] + a.rs.pos_off) {   // no slot of this pass in the chunk
      issue(b, kvh, c);
      issued = true;
    }
  }
  pdl_wait();
  trace_mark(a.rs, 1);
  pdl_launch_next();

  uint32_t phase = 0;
  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    int b, kvh, c;
    locate(item, b, kvh, c);
    if (!issued) issue(b, kvh, c);
    issued = false;
    if (!mbar_wait(&bar, phase, kWaitIters)) {
      if (tid == 0) atomicOr(a.err, kErrWait);
      mbar_wait(&bar, phase, kWaitIters);
      return;
    }
    phase ^= 1u;

    const int p0 = a.rs.pos_base[b] + a.rs.pos_off;
    // Slots past the last row's position hold stale or never-written cache
    // entries; a zero probability times a NaN there would still be NaN in
    // the P V product, so clear those rows of the tile.
    const int nvalid = min(kKvChunk, p0 + rps - c * kKvChunk);
    if (nvalid < kKvChunk) {
      for (int i = tid; i < (kKvChunk - nvalid) * (HD / 8); i += kAttnThreads) {
        const int r = nvalid + i / (HD / 8), u = i % (HD / 8);
        *reinterpret_cast<uint4*>(ks + r * KP + 16 * u) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(vs + r * VP + 16 * u) = make_uint4(0, 0, 0, 0);
      }
      __syncthreads();
    }
    for (int qt = warp; qt * 16 < Mq; qt += kAttnThreads / 32) {
      // Rows g and g+8 of the tile.
      int nk[2];
      const float* qrow[2];
      int mrow[2], hrow[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int qi = qt * 16 + g + 8 * r;
        const int j = qi / group, hh = qi - j * group;
        mrow[r] = b * rps + j;
        hrow[r] = kvh * group + hh;
        nk[r] = qi < Mq ? min(kKvChunk, p0 + j - c * kKvChunk + 1) : 0;
        qrow[r] = a.q + ((size_t)mrow[r] * a.nq + hrow[r]) * HD;
      }
      // S = Q K^T
      float sacc[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
      for (int k = 0; k < KS; ++k) {
        uint32_t qh[4], ql[4];
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 q0 = nk[0] > 0 ? *reinterpret_cast<const float4*>(qrow[0] + 16 * k + 4 * c4) : z;
        const float4 q1 = nk[1] > 0 ? *reinterpret_cast<const float4*>(qrow[1] + 16 * k + 4 * c4) : z;
        split_bf16x2(q0.x, q0.y, qh[0], ql[0]);
        split_bf16x2(q1.x, q1.y, qh[1], ql[1]);
        split_bf16x2(q0.z, q0.w, qh[2], ql[2]);
        split_bf16x2(q1.z, q1.w, qh[3], ql[3]);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const uint2 kb = *reinterpret_cast<const uint2*>(ks + (8 * nt + g) * KP + 32 * k + 8 * c4);
          mma_bf16_16816(sacc[nt], qh[0], qh[1], qh[2], qh[3], kb.x, kb.y);
          mma_bf16_16816(sacc[nt], ql[0], ql[1], ql[2], ql[3], kb.x, kb.y);
        }
      }
      // Softmax pieces per row: max, exp, sum (rows g: e = 0,1; g+8: e = 2,3).
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = e >> 1, key = 8 * nt + 2 * c4 + (e & 1);
          sacc[nt][e] = key < nk[r] ? sacc[nt][e] * a.scale : -INFINITY;
          mx[r] = fmaxf(mx[r], sacc[nt][e]);
        }
      float l[2] = {0.f, 0.f};
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = e >> 1, key = 8 * nt + 2 * c4 + (e & 1);
          const float pe = key < nk[r] ? expf(sacc[nt][e] - mx[r]) : 0.f;
          sacc[nt][e] = pe;
          l[r] += pe;
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
        l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
      }
      // O = P V
      float oacc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) oacc[nt][0] = oacc[nt][1] = oacc[nt][2] = oacc[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < kKvChunk / 16; ++kk) {
        uint32_t ph[4], pl[4];
        split_bf16x2(sacc[2 * kk][0], sacc[2 * kk][1], ph[0], pl[0]);
        split_bf16x2(sacc[2 * kk][2], sacc[2 * kk][3], ph[1], pl[1]);
        split_bf16x2(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1], ph[2], pl[2]);
        split_bf16x2(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3], ph[3], pl[3]);
        const unsigned char* vrow = vs + (16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1)) * VP;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          uint32_t b0, b1;
          ldsm_x2_trans(b0, b1, vrow + 16 * nt);
          mma_bf16_16816(oacc[nt], ph[0], ph[1], ph[2], ph[3], b0, b1);
          mma_bf16_16816(oacc[nt], pl[0], pl[1], pl[2], pl[3], b0, b1);
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (nk[r] <= 0) continue;
        float* dst = a.part + (((size_t)mrow[r] * a.nq + hrow[r]) * a.n_kv_chunks + c) * (HD + 2);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          *reinterpret_cast<float2*>(dst + 8 * nt + 2 * c4) = make_float2(oacc[nt][2 * r], oacc[nt][2 * r + 1]);
        if (c4 == 0) {
          dst[HD] = mx[r];
          dst[HD + 1] = l[r];
        }
      }
    }
    __syncthreads();   // everyone is done with ks/vs before the next copy
  }
}

// out[m][h*hd + d] = sum_c o_c[d] e^(m_c - M) / sum_c l_c e^(m_c - M). One CTA
// per (row, head) of 256 threads: thread (g, d) with g = tid / hd adds the
// chunks g, g + G, g + 2G, ... (G = 256 / hd) in order, up to kMergeLoads of
// them loaded at once, and the G partial sums are then added in order g =
// 0, 1, ...; every chunk's (max, sum) pair is loaded in the same round, so a
// merge costs two dependent global loads, not one per few chunks.
constexpr int kMaxKvChunks = 256;
constexpr int kMergeThreads = 256;
constexpr int kMergeLoads = 24;

__global__ void __launch_bounds__(kMergeThreads) k_attn_merge(const __grid_constant__ AttnArgs a) {
  __shared__ float wgt[kMaxKvChunks];
  __shared__ float lw[kMaxKvChunks];
  __shared__ float opart[kMergeThreads];
  __shared__ float red[kMergeThreads / 32];
  __shared__ float s_mx, s_l;
  RowSet rs1 = a.rs;
  rs1.trace_id = a.merge_trace_id;
  trace_mark(rs1, 0);
  pdl_wait();
  trace_mark(rs1, 1);
  pdl_launch_next();
  const int m = blockIdx.x / a.nq, h = blockIdx.x - m * a.nq;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = kMergeThreads / a.hd;
  const int grp = tid / a.hd, d = tid - grp * a.hd;
  const int nch = row_pos(a.rs, m) / kKvChunk + 1;
  const int stride = a.hd + 2;
  const float* src = a.part + ((size_t)m * a.nq + h) * a.n_kv_chunks * stride;
  // Round one: every chunk's (max, sum) and this thread's first output terms.
  const float mc = tid < nch ? src[(size_t)tid * stride + a.hd] : -INFINITY;
  const float lc = tid < nch ? src[(size_t)tid * stride + a.hd + 1] : 0.f;
  float v[kMergeLoads];
#pragma unroll
  for (int q = 0; q < kMergeLoads; ++q) {
    const int c = grp + q * G;
    v[q] = c < nch ? src[(size_t)c * stride + d] : 0.f;
  }
  const float wm = warp_max(mc);
  if (lane == 0) red[warp] = wm;
  __syncthreads();
  if (tid == 0) {
    float x = red[0];
    for (int w = 1; w < kMergeThreads / 32; ++w) x = fmaxf(x, red[w]);
    s_mx = x;
  }
  __syncthreads();
  if (tid < nch) {
    wgt[tid] = expf(mc - s_mx);
    lw[tid] = lc;
  }
  __syncthreads();
  if (tid == 0) {
    float l = 0.f;
    for (int c = 0; c < nch; ++c) l = fmaf(lw[c], wgt[c], l);
    s_l = l;
  }
  float o = 0.f;
#pragma unroll
  for (int q = 0; q < kMergeLoads; ++q) {
    const int c = grp + q * G;
    if (c < nch) o = fmaf(v[q], wgt[c], o);
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
      if (c < nch) o = fmaf(v[q], wgt[c], o);
    }
  }
  opart[tid] = o;
  __syncthreads();
  if (grp == 0) {
    float t = opart[d];
    for (int g2 = 1; g2 < G; ++g2) t += opart[g2 * a.hd + d];
    a.out[(size_t)m * a.nq * a.hd + (size_t)h * a.hd + d] = t / s_l;
  }
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
  cfg2.blockDim = dim3(kMergeThreads);
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
