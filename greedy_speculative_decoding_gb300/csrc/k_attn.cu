// Embedding gather, GQA attention over the static KV cache, RoPE table.
//
// Attention is split over the cache ("flash decoding"): one work item is
// (sequence, KV head, 64-slot chunk, tile of 16 queries), the queries being
// all rows of the sequence times the query heads that read this KV head.
// The chunk's keys and values are contiguous in the cache; the CTA brings
// them into padded shared-memory rows and computes its tile on the tensor
// cores with all eight warps. The chunk's partial result (row max, sum of
// exponentials, unnormalised output) goes to scratch; a second kernel merges
// the chunks of every (row, head) in a fixed order (attn_merge.cuh).
//
// Chunk boundaries are fixed multiples of 64 slots and a row at position p
// reads slots 0..p, so a row's result does not depend on the other rows.
#include "attn_merge.cuh"

namespace sf {

// ------------------------------------------------------------------ embedding
// x[m][:] = E[tok_m][:] in fp32, the per-128-feature sums of squares the next
// RMSNorm needs, and x * gain in fragment order (that RMSNorm's GEMM input).
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
    if (i == 0 && blk == 0) report_err(a.err, kErrCapacity);
    tok = 0;
  }
  const int n = blk * 128 + i;
  const float v = __bfloat162float(a.E[(size_t)tok * a.ld + n]);
  a.x[(size_t)m * a.H + n] = v;
  act_store(a.frag, m, n, (a.rs.M + 3) / 4, v * __bfloat162float(a.gain[n]), a.umma);
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

// One work item = (sequence b, KV head, 64-slot chunk c). Its keys and values
// come into padded shared-memory rows with 16-byte asynchronous copies
// (slots past the last row's position are zero-filled instead: a zero
// probability times a stale NaN would still be NaN). The queries that read
// this KV head (rows of the sequence x query heads of the group) go through
// in tiles of 16, and all eight warps share each tile:
//   S = Q K^T   warp w computes the 8 keys 8w..8w+7 over the whole head
//               dimension (mma.sync m16n8k16, Q as an fp32-accurate bf16
//               hi+lo pair, the head dimension walked in an order that makes
//               each key fragment one 8-byte shared load);
//   softmax     row max and row sum combined across the warps through
//               shared memory (sums in warp order);
//   O = P V     P (hi+lo) through shared memory, warp w producing output
//               dimensions w*HD/8 .. (w+1)*HD/8 - 1 from all 64 keys.
// The split is the same for every tile and every launch, so a row's result
// does not depend on how many other rows the launch carries.
template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 2) k_attn_chunks(const __grid_constant__ AttnArgs a) {
  constexpr int KP = HD * 2 + 32;   // key row pitch (bytes): 8-bank shift per row for the 8-byte fragment loads
  constexpr int VP = HD * 2 + 16;   // value row pitch: 4-bank shift per row for ldmatrix
  constexpr int KS = HD / 16;       // k-steps over the head dimension
  constexpr int NTW = HD / 64;      // output n-tiles (8 dimensions each) per warp
  constexpr int HP = HD + 16;       // query hi / lo row pitch (bf16): 8-bank shift per row
  constexpr int PP = kKvChunk + 8;  // probability tile row pitch (bf16)
  constexpr int kPieces = kKvChunk * HD / 8;   // 16-byte pieces of a chunk's keys (and of its values)
  static_assert(kAttnThreads == 256 && kKvChunk == 64, "eight warps of eight keys");
  extern __shared__ __align__(128) unsigned char attn_smem[];
  unsigned char* ks = attn_smem;                                   // [64][KP]
  unsigned char* vs = ks + kKvChunk * KP;                          // [64][VP]
  bf16* sph = reinterpret_cast<bf16*>(vs + kKvChunk * VP);         // [16][PP] P hi
  bf16* spl = sph + 16 * PP;                                       // [16][PP] P lo
  __shared__ float red_mx[8][16], red_l[8][16];

  trace_mark(a.rs, 0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c4 = lane & 3;
  const int group = a.nq / a.nkv;
  const int rps = a.rs.rps;
  const int Mq = rps * group;
  const int ntiles = (Mq + 15) / 16;
  bf16* sqh = spl + 16 * PP;                                       // [16][HP] queries of the tile, hi
  bf16* sql = sqh + 16 * HP;                                       // [16][HP] queries of the tile, lo

  // The lengths were written by kernels that finished before the preceding
  // one started, so they (and the cache slots below this pass's first
  // position) can be read before waiting on the preceding kernel.
  // Work item = (sequence b, KV head, chunk c, query tile qt); the tiles of
  // one chunk are consecutive items (their CTAs share the chunk through L2).
  int total = 0;
  for (int b = 0; b < a.B; ++b) {
    const int p_last = a.rs.pos_base[b] + a.rs.pos_off + rps - 1;
    total += a.nkv * (p_last / kKvChunk + 1) * ntiles;
  }
  auto locate = [&](int item, int& b, int& kvh, int& c, int& qt) {
    int rest = item, nch = 0;
    for (b = 0; b < a.B; ++b) {
      const int p_last = a.rs.pos_base[b] + a.rs.pos_off + rps - 1;
      nch = p_last / kKvChunk + 1;
      if (rest < a.nkv * nch * ntiles) break;
      rest -= a.nkv * nch * ntiles;
    }
    kvh = rest / (nch * ntiles);
    rest -= kvh * nch * ntiles;
    c = rest / ntiles;
    qt = rest - c * ntiles;
  };
  // Copy slots [0, nvalid) of the chunk; zero the rest of the tile.
  auto issue = [&](int b, int kvh, int c, int nvalid) {
    const size_t off = (((size_t)b * a.nkv + kvh) * a.s_max + (size_t)c * kKvChunk) * HD;
    for (int i = tid; i < kPieces; i += kAttnThreads) {
      const int r = i / (HD / 8), u = i - r * (HD / 8);
      if (r < nvalid) {
        cp_async16(ks + r * KP + 16 * u, a.kc + off + (size_t)r * HD + 8 * u);
        cp_async16(vs + r * VP + 16 * u, a.vc + off + (size_t)r * HD + 8 * u);
      } else {
        *reinterpret_cast<uint4*>(ks + r * KP + 16 * u) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(vs + r * VP + 16 * u) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_commit();
  };
  bool issued = false;
  if ((int)blockIdx.x < total) {
    int b, kvh, c, qt;
    locate(blockIdx.x, b, kvh, c, qt);
    if ((c + 1) * kKvChunk <= a.rs.pos_base[b] + a.rs.pos_off) {   // no slot of this pass in the chunk
      issue(b, kvh, c, kKvChunk);
      issued = true;
    }
  }
  pdl_wait();
  trace_mark(a.rs, 1);
  pdl_launch_next();

  // The item's 16 query rows -> shared memory as bf16 hi + lo pairs (rows
  // past Mq are zero), all loads of a thread in flight at once.
  auto stage_q = [&](int b, int kvh, int qt) {
    constexpr int kBatch = 16 * (HD / 4) / kAttnThreads;
    const int n4 = 16 * (HD / 4);
    for (int i0 = 0; i0 < n4; i0 += kBatch * kAttnThreads) {
      float4 v[kBatch];
#pragma unroll
      for (int e = 0; e < kBatch; ++e) {
        const int i = i0 + tid + e * kAttnThreads;
        const int qi = qt * 16 + i / (HD / 4), u = i % (HD / 4);
        v[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < n4 && qi < Mq) {
          const int j = qi / group, hh = qi - j * group;
          v[e] = *reinterpret_cast<const float4*>(a.q + ((size_t)(b * rps + j) * a.nq + kvh * group + hh) * HD + 4 * u);
        }
      }
#pragma unroll
      for (int e = 0; e < kBatch; ++e) {
        const int i = i0 + tid + e * kAttnThreads;
        if (i >= n4) break;
        const int qi = i / (HD / 4), u = i - qi * (HD / 4);   // row within the tile
        uint2 h, l;
        split_bf16x2(v[e].x, v[e].y, h.x, l.x);
        split_bf16x2(v[e].z, v[e].w, h.y, l.y);
        *reinterpret_cast<uint2*>(sqh + qi * HP + 4 * u) = h;
        *reinterpret_cast<uint2*>(sql + qi * HP + 4 * u) = l;
      }
    }
  };

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    int b, kvh, c, qt;
    locate(item, b, kvh, c, qt);
    const int p0 = a.rs.pos_base[b] + a.rs.pos_off;
    if (!issued) issue(b, kvh, c, min(kKvChunk, p0 + rps - c * kKvChunk));
    issued = false;
    stage_q(b, kvh, qt);
    cp_async_wait_all();
    __syncthreads();

    {
      const bf16* qht = sqh;
      const bf16* qlt = sql;
      // Rows g and g+8 of the tile: slots this row may see within the chunk.
      int nk[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int qi = qt * 16 + g + 8 * r;
        const int j = qi / group;
        nk[r] = qi < Mq ? min(kKvChunk, p0 + j - c * kKvChunk + 1) : 0;
      }
      // S for keys 8w .. 8w+7: four independent accumulation chains (hi / lo
      // part of Q x even / odd k-step), added in a fixed order at the end.
      float sa[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sa[i][0] = sa[i][1] = sa[i][2] = sa[i][3] = 0.f;
      const unsigned char* krow = ks + (8 * warp + g) * KP + 8 * c4;
#pragma unroll
      for (int k = 0; k < KS; ++k) {
        // Elements 16k + 4c4 .. +3 of rows g and g+8: (a0, a2) and (a1, a3).
        const uint2 h0 = *reinterpret_cast<const uint2*>(qht + g * HP + 16 * k + 4 * c4);
        const uint2 h1 = *reinterpret_cast<const uint2*>(qht + (g + 8) * HP + 16 * k + 4 * c4);
        const uint2 l0 = *reinterpret_cast<const uint2*>(qlt + g * HP + 16 * k + 4 * c4);
        const uint2 l1 = *reinterpret_cast<const uint2*>(qlt + (g + 8) * HP + 16 * k + 4 * c4);
        const uint2 kb = *reinterpret_cast<const uint2*>(krow + 32 * k);
        mma_bf16_16816(sa[k & 1], h0.x, h1.x, h0.y, h1.y, kb.x, kb.y);
        mma_bf16_16816(sa[2 + (k & 1)], l0.x, l1.x, l0.y, l1.y, kb.x, kb.y);
      }
      float sacc[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[e] = (sa[0][e] + sa[1][e]) + (sa[2][e] + sa[3][e]);
      // sacc[e]: row g (e < 2) or g+8, key 8w + 2c4 + (e & 1).
      float mx[2];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = e >> 1, key = 8 * warp + 2 * c4 + (e & 1);
        sacc[e] = key < nk[r] ? sacc[e] * a.scale : -INFINITY;
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(sacc[2 * r], sacc[2 * r + 1]);
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        if (c4 == 0) red_mx[warp][g + 8 * r] = mx[r];
      }
      __syncthreads();   // red_mx complete
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float m8 = red_mx[0][g + 8 * r];
#pragma unroll
        for (int w = 1; w < 8; ++w) m8 = fmaxf(m8, red_mx[w][g + 8 * r]);
        mx[r] = m8;
      }
      float pe[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = e >> 1, key = 8 * warp + 2 * c4 + (e & 1);
        pe[e] = key < nk[r] ? expf(sacc[e] - mx[r]) : 0.f;
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float l = pe[2 * r] + pe[2 * r + 1];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        if (c4 == 0) red_l[warp][g + 8 * r] = l;
        uint32_t h, lo;
        split_bf16x2(pe[2 * r], pe[2 * r + 1], h, lo);
        *reinterpret_cast<uint32_t*>(sph + (g + 8 * r) * PP + 8 * warp + 2 * c4) = h;
        *reinterpret_cast<uint32_t*>(spl + (g + 8 * r) * PP + 8 * warp + 2 * c4) = lo;
      }
      __syncthreads();

      // O = P V for this warp's output dimensions (P hi and P lo in two
      // accumulation chains, added at the end).
      float oh[NTW][4], ol[NTW][4];
#pragma unroll
      for (int t = 0; t < NTW; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) oh[t][e] = ol[t][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < kKvChunk / 16; ++kk) {
        uint32_t ph[4], pl[4];
        const int k0 = 16 * kk + 2 * c4;
        ph[0] = *reinterpret_cast<const uint32_t*>(sph + g * PP + k0);
        ph[1] = *reinterpret_cast<const uint32_t*>(sph + (g + 8) * PP + k0);
        ph[2] = *reinterpret_cast<const uint32_t*>(sph + g * PP + k0 + 8);
        ph[3] = *reinterpret_cast<const uint32_t*>(sph + (g + 8) * PP + k0 + 8);
        pl[0] = *reinterpret_cast<const uint32_t*>(spl + g * PP + k0);
        pl[1] = *reinterpret_cast<const uint32_t*>(spl + (g + 8) * PP + k0);
        pl[2] = *reinterpret_cast<const uint32_t*>(spl + g * PP + k0 + 8);
        pl[3] = *reinterpret_cast<const uint32_t*>(spl + (g + 8) * PP + k0 + 8);
        const unsigned char* vrow = vs + (16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1)) * VP;
#pragma unroll
        for (int t = 0; t < NTW; ++t) {
          uint32_t b0, b1;
          ldsm_x2_trans(b0, b1, vrow + 16 * (warp * NTW + t));
          mma_bf16_16816(oh[t], ph[0], ph[1], ph[2], ph[3], b0, b1);
          mma_bf16_16816(ol[t], pl[0], pl[1], pl[2], pl[3], b0, b1);
        }
      }
      float oacc[NTW][4];
#pragma unroll
      for (int t = 0; t < NTW; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[t][e] = oh[t][e] + ol[t][e];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (nk[r] <= 0) continue;
        const int qi = qt * 16 + g + 8 * r;
        const int j = qi / group, hh = qi - j * group;
        const int m = b * rps + j, h = kvh * group + hh;
        float* dst = a.part + (((size_t)m * a.nq + h) * a.n_kv_chunks + c) * (HD + 2);
#pragma unroll
        for (int t = 0; t < NTW; ++t)
          *reinterpret_cast<float2*>(dst + 8 * (warp * NTW + t) + 2 * c4) =
              make_float2(oacc[t][2 * r], oacc[t][2 * r + 1]);
        if (warp == 0 && c4 == 0) {
          float l = red_l[0][g + 8 * r];
#pragma unroll
          for (int w = 1; w < 8; ++w) l += red_l[w][g + 8 * r];
          dst[HD] = mx[r];
          dst[HD + 1] = l;
        }
      }
      __syncthreads();   // P and red_* are free again
    }
  }
}

// The merge kernel: one CTA of kMergeThreads per (row, head); writes the
// output projection's input in fragment order.
__global__ void __launch_bounds__(kMergeThreads) k_attn_merge(const __grid_constant__ AttnArgs a) {
  __shared__ MergeSmem sm;
  RowSet rs1 = a.rs;
  rs1.trace_id = a.merge_trace_id;
  trace_mark(rs1, 0);
  pdl_wait();
  trace_mark(rs1, 1);
  pdl_launch_next();
  const int m = blockIdx.x / a.nq, h = blockIdx.x - m * a.nq;
  const int nch = row_pos(a.rs, m) / kKvChunk + 1;
  const float v = merge_row_head(a.part, a.nq, a.hd, a.n_kv_chunks, m, h, nch, sm);
  if ((int)threadIdx.x < a.hd) act_store(a.out, m, h * a.hd + threadIdx.x, (a.rs.M + 3) / 4, v, a.umma);
}

// Dynamic shared memory of the chunk kernel: keys, values, P hi + lo, and
// the item's query rows (padded to whole tiles of 16).
static int attn_smem_bytes(int hd) {
  return kKvChunk * (hd * 2 + 32) + kKvChunk * (hd * 2 + 16) + 2 * 16 * (kKvChunk + 8) * 2 + 2 * 16 * (hd + 16) * 2;
}

// Dynamic shared-memory limits of the chunk kernels and the largest
// shared-memory carve-out for every kernel of the chain.
cudaError_t attn_init() {
  cudaError_t e = cudaFuncSetAttribute(k_attn_chunks<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       attn_smem_bytes(128));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_attn_chunks<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, attn_smem_bytes(64));
  if (e != cudaSuccess) return e;
  // Largest shared-memory carve-out for every kernel of the chain (see gemm_init).
  const void* fns[] = {reinterpret_cast<const void*>(k_attn_chunks<128>),
                       reinterpret_cast<const void*>(k_attn_chunks<64>),
                       reinterpret_cast<const void*>(k_attn_merge), reinterpret_cast<const void*>(k_embed)};
  for (const void* f : fns)
    if ((e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
      return e;
  return cudaSuccess;
}

cudaError_t launch_attention(const AttnArgs& a, int num_sms, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  // Enough CTAs for the largest item count this launch can see (the count
  // itself lives on the device): B * nkv * chunks of the whole cache, capped.
  const int max_items = a.B * a.nkv * a.n_kv_chunks * ((a.rs.rps * (a.nq / a.nkv) + 15) / 16);
  cfg.gridDim = dim3(max(1, min(max_items, 2 * num_sms)));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e;
  cfg.dynamicSmemBytes = attn_smem_bytes(a.hd);
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
