// Skinny bf16 GEMM for decode (1-2 rows) and verify (K+1 rows) on sm_103a.
//
// The work is weight streaming: y[m][n] = sum_k a[m][k] W[n][k] with at most
// SF_MAX_ROWS token rows m, so every weight byte is read once and used by all
// rows. Each CTA owns 128 output rows (8 warps x 16) and one slice of K.
// Every warp runs its own TMA pipeline: a ring of kStages shared-memory
// tiles (16 weight rows x 64 k, 128-byte swizzle) filled by
// cp.async.bulk.tensor loads that complete on per-stage mbarriers, so about
// 80 KB of weights per CTA are in flight without holding registers. The tiles
// feed mma.sync m16n8k16 as the A operand ("swap AB": weights are the M
// side, tokens the N side). The token activations are staged in
// shared memory, converted to a bf16 pair (hi + lo) so that the product keeps
// about 16 mantissa bits of the fp32 activation; hi and lo of one token sit
// in adjacent columns of the n8 tile and are summed in the epilogue.
//
// Inside an MMA the order of k does not matter as long as A and B agree, so
// each thread takes 16 consecutive k of its rows and the activation tile is
// laid out in the matching "fragment order" (conflict-free 128-bit reads).
//
// Every row's arithmetic is independent of how many rows are present (same
// K split, same MMA sequence, same reduction order), so a verify row equals
// the decode of the same token at the same position bit for bit.
//
// Split-K partial tiles go to a global scratch area; the last CTA of a row
// block (arrival counter) adds them in fixed slice order and runs the
// epilogue, so results are deterministic without float atomics.
#include "sf_kernels.h"

namespace sf {

namespace {

constexpr uint32_t kWaitIters = 1u << 24;

// Tensor map and row coordinate of warp w's 16 rows in row block rb.
template <int EPI>
__device__ __forceinline__ int warp_tile_row(const GemmArgs& a, int rb, int w, int* seg) {
  if (EPI == EPI_SWIGLU) {           // warps 0-3: gate rows, 4-7: up rows of the same 64 features
    *seg = w >> 2;
    return rb * 64 + 16 * (w & 3);
  }
  const int n = rb * kBlockRows;     // segment boundaries are multiples of 128
  int s = 0;
  while (s < a.nseg - 1 && n >= a.seg_end[s]) ++s;
  *seg = s;
  return n - (s ? a.seg_end[s - 1] : 0) + 16 * w;
}

// Stage activation chunks [wc0, wc0 + nwc) of this CTA (absolute chunk index
// c0 + wc) into fragment order: [wc][t][h][lane][8] bf16, lane = 4*col + c
// with col = 2*(m%4) + {0: hi, 1: lo}, and k = 64*chunk + 16*c + 8*h + e.
template <int T>
__device__ __forceinline__ void stage_acts(const GemmArgs& a, uint2* act, const float* rinv, int cabs0,
                                           int nwc, int M) {
  constexpr int kItems = (4 * T * kWinChunks * 16 + kGemmThreads - 1) / kGemmThreads;
  const int per_m = nwc * 16;  // groups of 4 k per token row
  const int total = 4 * T * per_m;
  // All global loads of this thread first, so their latencies overlap.
  float4 v[kItems];
  uint2 gg[kItems];
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int idx = threadIdx.x + it * kGemmThreads;
    const int m = idx / per_m;
    const int k = cabs0 * kChunk + (idx - m * per_m) * 4;
    v[it] = make_float4(0.f, 0.f, 0.f, 0.f);
    gg[it] = make_uint2(0, 0);
    if (idx < total && m < M && k < a.K) {
      v[it] = *reinterpret_cast<const float4*>(a.in + (size_t)m * a.in_ld + k);
      if (a.gain) gg[it] = *reinterpret_cast<const uint2*>(a.gain + k);
    }
  }
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int idx = threadIdx.x + it * kGemmThreads;
    if (idx >= total) continue;
    const int m = idx / per_m;
    const int q4 = idx - m * per_m;
    float4 x = v[it];
    if (a.gain && m < M) {
      const float r = rinv[m];
      const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gg[it].x));
      const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gg[it].y));
      x.x = (x.x * r) * g01.x;
      x.y = (x.y * r) * g01.y;
      x.z = (x.z * r) * g23.x;
      x.w = (x.w * r) * g23.y;
    }
    const bf16 h0 = __float2bfloat16_rn(x.x), h1 = __float2bfloat16_rn(x.y);
    const bf16 h2 = __float2bfloat16_rn(x.z), h3 = __float2bfloat16_rn(x.w);
    const bf16 l0 = __float2bfloat16_rn(x.x - __bfloat162float(h0));
    const bf16 l1 = __float2bfloat16_rn(x.y - __bfloat162float(h1));
    const bf16 l2 = __float2bfloat16_rn(x.z - __bfloat162float(h2));
    const bf16 l3 = __float2bfloat16_rn(x.w - __bfloat162float(h3));
    const int wc = q4 >> 4;
    const int kk = (q4 & 15) * 4;
    const int c = kk >> 4, h = (kk >> 3) & 1, e = kk & 7;
    const int t = m >> 2, col = 2 * (m & 3);
    const int base = ((wc * T + t) * 2 + h) * 32;     // in 16-byte units
    // uint2 index: 16-byte unit * 2 + (e / 4)
    act[(base + 4 * col + c) * 2 + (e >> 2)] = make_uint2(pack_bf16x2(h0, h1), pack_bf16x2(h2, h3));
    act[(base + 4 * (col + 1) + c) * 2 + (e >> 2)] = make_uint2(pack_bf16x2(l0, l1), pack_bf16x2(l2, l3));
  }
}

template <int T>
__device__ __forceinline__ void mma_chunk(float (&acc)[T][4], const uint4 (&w)[4], const uint4* act, int wc,
                                          int lane) {
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const uint4 b0 = act[((wc * T + t) * 2 + 0) * 32 + lane];
    const uint4 b1 = act[((wc * T + t) * 2 + 1) * 32 + lane];
    mma_bf16_16816(acc[t], w[0].x, w[2].x, w[0].y, w[2].y, b0.x, b0.y);
    mma_bf16_16816(acc[t], w[0].z, w[2].z, w[0].w, w[2].w, b0.z, b0.w);
    mma_bf16_16816(acc[t], w[1].x, w[3].x, w[1].y, w[3].y, b1.x, b1.y);
    mma_bf16_16816(acc[t], w[1].z, w[3].z, w[1].w, w[3].w, b1.z, b1.w);
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

// ---------------------------------------------------------------- epilogues
template <int T>
__device__ void epi_resid(const GemmArgs& a, float* ys, int rb, int M) {
  constexpr int kE = (4 * T * kBlockRows + kGemmThreads - 1) / kGemmThreads;
  float old[kE];
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    const int i = threadIdx.x + e * kGemmThreads;
    const int m = i / kBlockRows, n = rb * kBlockRows + (i - m * kBlockRows);
    old[e] = (m < M && n < a.N) ? a.out[(size_t)m * a.out_ld + n] : 0.f;
  }
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    const int i = threadIdx.x + e * kGemmThreads;
    if (i >= M * kBlockRows) continue;
    const int m = i / kBlockRows, n = rb * kBlockRows + (i - m * kBlockRows);
    float v = 0.f;
    if (n < a.N) {
      v = old[e] + ys[i];
      a.out[(size_t)m * a.out_ld + n] = v;
    }
    ys[i] = v;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int m = warp; m < M; m += kGemmThreads / 32) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float v = ys[m * kBlockRows + lane + 32 * j];
      s = fmaf(v, v, s);
    }
    s = warp_sum(s);
    if (lane == 0) a.ssq_out[rb * kRows + m] = s;
  }
}

template <int T>
__device__ void epi_qkv(const GemmArgs& a, const float* ys, int rb, int M) {
  constexpr int kE = (4 * T * kBlockRows + kGemmThreads - 1) / kGemmThreads;
  const int half = a.hd >> 1;
  const int n0 = rb * kBlockRows;
  const int s = n0 < a.seg_end[0] ? 0 : (n0 < a.seg_end[1] ? 1 : 2);   // one segment per block
  const int seg0 = s ? a.seg_end[s - 1] : 0;
  const bf16* bias = a.bias[s];
  // Gather every global operand first (bias pairs, rotation factors, positions).
  float b1[kE], b2[kE];
  float2 cs[kE];
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    const int i = threadIdx.x + e * kGemmThreads;
    const int m = i / kBlockRows, r = i - m * kBlockRows;
    const int local = n0 + r - seg0;
    const int d = local % a.hd;
    b1[e] = b2[e] = 0.f;
    cs[e] = make_float2(1.f, 0.f);
    if (m < M && n0 + r < a.N) {
      if (bias) b1[e] = __bfloat162float(bias[local]);
      if (s < 2 && d < half) {
        if (bias) b2[e] = __bfloat162float(bias[local + half]);
        cs[e] = a.rope[(size_t)row_pos(a.rs, m) * half + d];
      }
    }
  }
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    const int i = threadIdx.x + e * kGemmThreads;
    const int m = i / kBlockRows, r = i - m * kBlockRows;
    if (m >= M || n0 + r >= a.N) continue;
    const int local = n0 + r - seg0;
    const int d = local % a.hd;
    const int b = m / a.rs.rps;
    const int pos = row_pos(a.rs, m);
    if (s == 2) {
      const int kvh = local / a.hd;
      a.vc[(((size_t)b * a.nkv + kvh) * a.s_max + pos) * a.hd + d] = __float2bfloat16_rn(ys[i] + b1[e]);
      continue;
    }
    if (d >= half) continue;
    const float x1 = ys[i] + b1[e];
    const float x2 = ys[i + half] + b2[e];
    const float y1 = x1 * cs[e].x - x2 * cs[e].y;
    const float y2 = x2 * cs[e].x + x1 * cs[e].y;
    if (s == 0) {
      float* q = a.out + (size_t)m * a.out_ld + local;
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

__device__ void epi_swiglu(const GemmArgs& a, const float* ys, int rb, int M) {
  for (int i = threadIdx.x; i < M * 64; i += kGemmThreads) {
    const int m = i >> 6, j = i & 63;
    const int f = rb * 64 + j;
    if (f >= a.N) continue;
    const float gte = ys[m * kBlockRows + j];
    const float up = ys[m * kBlockRows + 64 + j];
    a.out[(size_t)m * a.out_ld + f] = gte / (1.0f + expf(-gte)) * up;
  }
}

__device__ void epi_store(const GemmArgs& a, const float* ys, int rb, int M) {
  for (int i = threadIdx.x; i < M * kBlockRows; i += kGemmThreads) {
    const int m = i / kBlockRows, r = i - m * kBlockRows;
    const int n = rb * kBlockRows + r;
    if (n < a.N) a.out[(size_t)m * a.out_ld + n] = ys[i];
  }
}

__device__ void epi_argmax(const GemmArgs& a, const float* ys, int rb, int M, int* s_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int m = warp; m < M; m += kGemmThreads / 32) {
    unsigned long long best = 0ull;
    bool bad = false;
    const int mb = m / a.rs.rps, mj = m - mb * a.rs.rps;
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
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.err, kErrNonfinite);
    if (lane == 0) atomicMax(a.keys + m, best);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *s_flag = (atomicAdd(a.done, 1) == a.nblocks - 1);
  __syncthreads();
  if (!*s_flag) return;
  __threadfence();
  if (threadIdx.x < M) {
    const int m = threadIdx.x;
    const unsigned long long k = atomicExch(a.keys + m, 0ull);
    const int b = m / a.rs.rps, j = m - b * a.rs.rps;
    if (j >= a.tok_skip) a.tok_out[b * a.tok_stride + a.tok_off + j - a.tok_skip] = key_index(k);
  }
  if (threadIdx.x == 0) *a.done = 0;
}

}  // namespace

template <int T, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 2) k_gemm(const __grid_constant__ GemmArgs a) {
  extern __shared__ unsigned char smem_raw[];
  // The swizzled TMA tiles need a 1024-byte aligned base.
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  unsigned char* ring = smem;                                            // [8][kStages][kTileBytes]
  uint4* act = reinterpret_cast<uint4*>(smem + 8 * kStages * kTileBytes);
  float* ys = reinterpret_cast<float*>(smem + 8 * kStages * kTileBytes + kWinChunks * T * 1024);
  float* rinv = ys + 4 * T * kBlockRows;
  uint64_t* bars = reinterpret_cast<uint64_t*>(rinv + 4 * T);           // [8][kStages]
  __shared__ int s_flag;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int rb = blockIdx.x / a.nsplit, sp = blockIdx.x - rb * a.nsplit;
  const int nch_total = (a.K + kChunk - 1) / kChunk;
  const int c0 = sp * a.cps;
  const int nch = min(a.cps, nch_total - c0);

  int seg = 0;
  const int trow = warp_tile_row<EPI>(a, rb, warp, &seg);
  const CUtensorMap* map = &a.tm[seg];
  unsigned char* my_ring = ring + warp * kStages * kTileBytes;
  uint64_t* my_bar = bars + warp * kStages;
  uint64_t policy = 0;
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&my_bar[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    policy = policy_evict_first();
    // Weights are never written by the preceding kernels: start streaming
    // them before waiting on the producer of the activations.
    for (int s = 0; s < kStages && s < nch; ++s) {
      mbar_expect_tx(&my_bar[s], kTileBytes);
      tma_load_2d(my_ring + s * kTileBytes, map, (c0 + s) * kChunk, trow, &my_bar[s], policy);
    }
  }
  __syncwarp();

  pdl_wait();
  pdl_launch_next();
  const int M = a.rs.M;
  if (a.gain) {
    // 1 / rms of each token row from the per-128-feature sums of squares:
    // one warp per row, one load per lane (at most 64 partial sums).
    for (int m = warp; m < M; m += kGemmThreads / 32) {
      float s0 = lane < a.nssq ? a.ssq[lane * kRows + m] : 0.f;
      float s1 = lane + 32 < a.nssq ? a.ssq[(lane + 32) * kRows + m] : 0.f;
      const float s = warp_sum(s0 + s1);
      if (lane == 0) rinv[m] = 1.0f / sqrtf(s * a.inv_k + a.eps);
    }
  }
  __syncthreads();
  stage_acts<T>(a, reinterpret_cast<uint2*>(act), rinv, c0, min(nch, kWinChunks), M);
  __syncthreads();

  float acc[T][4];
#pragma unroll
  for (int t = 0; t < T; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  // Row g / g+8 of the tile, 16-byte units 2c and 2c+1 (k = 16c .. 16c+15),
  // at their 128-byte-swizzled positions.
  const int sw = g & 7;
  const int off_lo = g * 128 + (((2 * c) ^ sw) << 4);
  const int off_hi = g * 128 + (((2 * c + 1) ^ sw) << 4);
  bool timed_out = false;
  for (int ch = 0; ch < nch; ++ch) {
    if (ch > 0 && (ch % kWinChunks) == 0) {
      __syncthreads();
      stage_acts<T>(a, reinterpret_cast<uint2*>(act), rinv, c0 + ch, min(nch - ch, kWinChunks), M);
      __syncthreads();
    }
    const int s = ch % kStages;
    if (!mbar_wait(&my_bar[s], (ch / kStages) & 1, kWaitIters)) timed_out = true;
    const unsigned char* tile = my_ring + s * kTileBytes;
    uint4 w[4];
    w[0] = *reinterpret_cast<const uint4*>(tile + off_lo);
    w[1] = *reinterpret_cast<const uint4*>(tile + off_hi);
    w[2] = *reinterpret_cast<const uint4*>(tile + 8 * 128 + off_lo);
    w[3] = *reinterpret_cast<const uint4*>(tile + 8 * 128 + off_hi);
    __syncwarp();
    if (lane == 0 && ch + kStages < nch) {
      fence_proxy_async();   // the warp's reads of this stage before the async refill
      mbar_expect_tx(&my_bar[s], kTileBytes);
      tma_load_2d(my_ring + s * kTileBytes, map, (c0 + ch + kStages) * kChunk, trow, &my_bar[s], policy);
    }
    mma_chunk<T>(acc, w, act, ch % kWinChunks, lane);
  }
  if (timed_out) {
    // A tile never arrived: report, and give every copy of this warp one more
    // bounded chance to land before the CTA's shared memory is released.
    if (lane == 0) atomicOr(a.err, kErrWait);
    for (int ch = max(0, nch - kStages); ch < nch; ++ch)
      mbar_wait(&my_bar[ch % kStages], (ch / kStages) & 1, kWaitIters);
  }

  // Token m = 4t + c: hi in column 2c, lo in column 2c + 1.
  const int r0 = warp * 16 + g;
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const int m = 4 * t + c;
    ys[m * kBlockRows + r0] = acc[t][0] + acc[t][1];
    ys[m * kBlockRows + r0 + 8] = acc[t][2] + acc[t][3];
  }
  __syncthreads();

  if (a.nsplit > 1) {
    float* mine = a.part + ((size_t)rb * a.nsplit + sp) * (kRows * kBlockRows);
    for (int i = tid; i < M * kBlockRows; i += kGemmThreads) __stcg(mine + i, ys[i]);
    __threadfence();
    __syncthreads();
    if (tid == 0) s_flag = (atomicAdd(a.counter + rb, 1) == a.nsplit - 1);
    __syncthreads();
    if (!s_flag) return;
    __threadfence();
    // Sum the slices in fixed order 0, 1, ..., loading four slices' worth of
    // this thread's elements at a time so the loads overlap.
    const float* src = a.part + (size_t)rb * a.nsplit * (kRows * kBlockRows);
    constexpr int kE = (4 * T * kBlockRows + kGemmThreads - 1) / kGemmThreads;
    float sum[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) sum[e] = 0.f;
    for (int p0 = 0; p0 < a.nsplit; p0 += 4) {
      float v[4][kE];
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int e = 0; e < kE; ++e) {
          const int i = tid + e * kGemmThreads;
          v[q][e] = (p0 + q < a.nsplit && i < M * kBlockRows)
                        ? __ldcg(src + (size_t)(p0 + q) * (kRows * kBlockRows) + i)
                        : 0.f;
        }
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int e = 0; e < kE; ++e) sum[e] += v[q][e];
    }
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      const int i = tid + e * kGemmThreads;
      if (i < M * kBlockRows) ys[i] = sum[e];
    }
    if (tid == 0) a.counter[rb] = 0;
    __syncthreads();
  }

  if (EPI == EPI_RESID) epi_resid<T>(a, ys, rb, M);
  else if (EPI == EPI_QKV) epi_qkv<T>(a, ys, rb, M);
  else if (EPI == EPI_SWIGLU) epi_swiglu(a, ys, rb, M);
  else if (EPI == EPI_STORE) epi_store(a, ys, rb, M);
  else epi_argmax(a, ys, rb, M, &s_flag);
}

int gemm_smem_bytes(int M) {
  const int T = (M + 3) / 4;
  return 1024 /* alignment slack */ + 8 * kStages * kTileBytes + kWinChunks * T * 1024 + 4 * T * kBlockRows * 4 +
         4 * T * 4 + 8 * kStages * 8;
}

cudaError_t make_weight_map(CUtensorMap* map, const void* w, int rows, int K, int ld) {
  typedef CUresult (*encode_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static encode_fn encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
    encode = reinterpret_cast<encode_fn>(fn);
  }
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kChunk, 16};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int T, int EPI>
static cudaError_t launch_t(const GemmArgs& a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nblocks * a.nsplit);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = gemm_smem_bytes(4 * T);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_gemm<T, EPI>, a);
}

template <int T>
static cudaError_t init_t() {
  const int smem = gemm_smem_bytes(4 * T);
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_gemm<T, EPI_QKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem))) return e;
  if ((e = cudaFuncSetAttribute(k_gemm<T, EPI_RESID>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem))) return e;
  if ((e = cudaFuncSetAttribute(k_gemm<T, EPI_SWIGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem))) return e;
  if ((e = cudaFuncSetAttribute(k_gemm<T, EPI_STORE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem))) return e;
  return cudaFuncSetAttribute(k_gemm<T, EPI_ARGMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

// Raise the dynamic shared-memory limit of every instantiation (current device).
cudaError_t gemm_init() {
  cudaError_t e;
  if ((e = init_t<1>())) return e;
  if ((e = init_t<2>())) return e;
  if ((e = init_t<3>())) return e;
  return init_t<4>();
}

template <int EPI>
static cudaError_t launch_e(const GemmArgs& a, cudaStream_t st, bool pdl) {
  switch ((a.rs.M + 3) / 4) {
    case 1: return launch_t<1, EPI>(a, st, pdl);
    case 2: return launch_t<2, EPI>(a, st, pdl);
    case 3: return launch_t<3, EPI>(a, st, pdl);
    case 4: return launch_t<4, EPI>(a, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm(const GemmArgs& a, int epi, cudaStream_t st, bool pdl) {
  if (a.rs.M < 1 || a.rs.M > kRows) return cudaErrorInvalidValue;
  switch (epi) {
    case EPI_QKV: return launch_e<EPI_QKV>(a, st, pdl);
    case EPI_RESID: return launch_e<EPI_RESID>(a, st, pdl);
    case EPI_SWIGLU: return launch_e<EPI_SWIGLU>(a, st, pdl);
    case EPI_ARGMAX: return launch_e<EPI_ARGMAX>(a, st, pdl);
    case EPI_STORE: return launch_e<EPI_STORE>(a, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sf
