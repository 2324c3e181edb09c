// Skinny bf16 GEMM for decode (1-2 rows) and verify (K+1 rows) on sm_103a.
//
// The work is weight streaming: y[m][n] = sum_k a[m][k] W[n][k] with at most
// 16 token rows m per CTA, so every weight byte is read once and used by all
// rows. Each CTA owns 128 output rows (8 warps x 16) and one slice of K. A
// launch of more rows (up to SF_MAX_ROWS) runs one CTA per 16-row group,
// neighbours in launch order: the first to ask for a weight tile brings it
// from HBM, the others find it in L2 (normal eviction priority instead of
// evict-first).
// Every warp runs its own TMA pipeline: a ring of kStages shared-memory
// tiles (16 weight rows x 64 k, 128-byte swizzle) filled by
// cp.async.bulk.tensor loads that complete on per-stage mbarriers, so about
// 80 KB of weights per CTA are in flight without holding registers. The tiles
// feed mma.sync m16n8k16 as the A operand ("swap AB": weights are the M
// side, tokens the N side). The token activations arrive from the producing
// kernel already as bf16 pairs (hi + lo, about 16 mantissa bits of the fp32
// value) in "fragment order": each lane reads its B operand for a 64-k chunk
// with two 16-byte loads per token tile, straight from global memory (L1
// serves the other warps of the CTA), one chunk ahead of the MMAs, so no
// warp ever waits for the others inside the main loop. hi and lo of one
// token sit in adjacent columns of the n8 tile and are summed at the end.
// An RMSNorm input is stored as x * gain; the 1 / rms(x) row factor is
// applied to the finished dot products.
//
// Inside an MMA the order of k does not matter as long as A and B agree, so
// each thread takes 16 consecutive k of its rows and the activations are
// laid out in the matching order (frag_index).
//
// Every row's arithmetic is independent of how many rows are present (same
// K split, same MMA sequence, same reduction order), so a verify row equals
// the decode of the same token at the same position bit for bit.
//
// Split K: the slices of a row block are one thread-block cluster; every
// rank but 0 pushes its partial tile into rank 0's shared memory with
// asynchronous remote stores (or, when that area does not fit, rank 0 pulls
// the tiles after a cluster barrier), and rank 0 adds them in rank order and
// runs the epilogue. sf_linear splits without clusters: partial tiles go to
// a global scratch area and the last CTA of a row block (arrival counter)
// adds them in slice order. Either way results are deterministic without
// float atomics.
#include <algorithm>
#include <mutex>

#include "gemm_epi.cuh"

namespace sf {

namespace {

constexpr int kMaxDevices = 64;

constexpr uint32_t kWaitIters = 1u << 24;
constexpr int kScaleTileBytes = 16 * 8 * 2;   // NF4: 16 rows x 8 block scales (fp16)

__constant__ float c_nf4_levels[16];

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

// B operand of chunk j for this lane: per token tile, the two 16-byte units
// of halves h = 0, 1. Chunks are `stride` units apart; tiles t >= tl (past
// the last token tile of the layout, in the last row group) read as zero.
template <int T>
__device__ __forceinline__ void load_b(uint4 (&b)[T][2], const uint4* in, size_t stride, int j, int tl, int lane) {
  const uint4* p = in + (size_t)j * stride + lane;
#pragma unroll
  for (int t = 0; t < T; ++t) {
    if (t < tl) {
      b[t][0] = p[(2 * t) * 32];
      b[t][1] = p[(2 * t + 1) * 32];
    } else {
      b[t][0] = b[t][1] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Copy the B operand of chunks [c0, c0 + nch) of this CTA's token tiles into
// shared memory (T tiles per chunk, contiguous); tiles t >= tl become zero.
template <int T>
__device__ __forceinline__ void stage_b_copy(uint4* dst, const uint4* src, size_t stride, int nch, int tl) {
  for (int i = threadIdx.x; i < nch * T * 64; i += kGemmThreads) {
    const int ci = i / (T * 64), r = i - ci * (T * 64);
    if (r / 64 < tl) cp_async16(dst + i, src + (size_t)ci * stride + r);
    else dst[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
}

template <int T>
__device__ __forceinline__ void mma_chunk(float (&acc)[T][4], const uint4 (&w)[4], const uint4 (&b)[T][2]) {
#pragma unroll
  for (int t = 0; t < T; ++t) {
    mma_bf16_16816(acc[t], w[0].x, w[2].x, w[0].y, w[2].y, b[t][0].x, b[t][0].y);
    mma_bf16_16816(acc[t], w[0].z, w[2].z, w[0].w, w[2].w, b[t][0].z, b[t][0].w);
    mma_bf16_16816(acc[t], w[1].x, w[3].x, w[1].y, w[3].y, b[t][1].x, b[t][1].y);
    mma_bf16_16816(acc[t], w[1].z, w[3].z, w[1].w, w[3].w, b[t][1].z, b[t][1].w);
  }
}


}  // namespace

// GRP: the launch has more than 16 token rows (T = 4, one CTA per row group);
// without it the row-group arithmetic folds away at compile time.
template <int T, int EPI, bool NF4, bool GRP>
__global__ void __launch_bounds__(kGemmThreads, (T <= 3 || (!NF4 && EPI != EPI_QKV) ? 2 : 1)) k_gemm(const __grid_constant__ GemmArgs a) {
  extern __shared__ unsigned char smem_raw[];
  // The swizzled TMA tiles need a 1024-byte aligned base.
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  unsigned char* ring = smem;                                            // [8][kStages][kTileBytes]
  const int kStages = a.stages;
  // NF4: each stage also carries the block scales of its rows ([16][8] fp16).
  unsigned char* sring = smem + 8 * kStages * kTileBytes;                // [8][kStages][kScaleTileBytes]
  unsigned char* after_ring = sring + (NF4 ? 8 * kStages * kScaleTileBytes : 0);
  float* ys = reinterpret_cast<float*>(after_ring);
  float* rinv = ys + 4 * T * kBlockRows;
  uint64_t* bars = reinterpret_cast<uint64_t*>(rinv + 4 * T);           // [8][kStages]
  uint4* bstage = reinterpret_cast<uint4*>(bars + 8 * kStages);         // staged B operand (if any)
  const int sb = a.stage_b ? staged_b_bytes(T, a.cps) : 0;             // staged B operand bytes
  float* recv = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(bstage) + sb);   // push landing area
  __shared__ int s_flag;
  __shared__ int s_pos[kGroupRows];
  __shared__ __align__(8) uint64_t recv_bar;   // push: the other ranks' tiles have landed
  // NF4: byte (two codes) -> bf16 pair of levels, one copy of the 256-entry
  // table per lane (entry b of lane l at 32 b + l: every lookup of a warp
  // hits its own bank, whatever the codes).
  __shared__ uint32_t lut[NF4 ? 256 * 32 : 1];
  trace_mark(a.rs, 0);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  // Block = (row block rb, token row group gi, K slice sp). The slices of one
  // (rb, gi) are consecutive (one cluster), and the row groups of a row block
  // are neighbours in launch order, so they read its weight tiles at about
  // the same time: from HBM once, then from L2.
  const int G = GRP ? (a.rs.M + kGroupRows - 1) / kGroupRows : 1;
  const int Tt = GRP ? (a.rs.M + 3) / 4 : T;        // token tiles of the fragment layout
  const int qb = blockIdx.x / a.nsplit, sp = blockIdx.x - qb * a.nsplit;
  const int rb = GRP ? qb / G : qb, gi = GRP ? qb - rb * G : 0;
  const int m0 = gi * kGroupRows;
  const int M = GRP ? min(kGroupRows, a.rs.M - m0) : a.rs.M;   // token rows of this CTA
  const int tl = GRP ? min(T, Tt - 4 * gi) : T;     // token tiles present in this group
  const int nch_total = (a.K + kChunk - 1) / kChunk;
  const int c0 = sp * a.cps;
  const int nch = min(a.cps, nch_total - c0);

  int seg = 0;
  const int trow = warp_tile_row<EPI>(a, rb, warp, &seg);
  const CUtensorMap* map = &a.tm[seg];
  const CUtensorMap* smap = &a.tms[seg];
  unsigned char* my_ring = ring + warp * kStages * kTileBytes;
  unsigned char* my_sring = sring + warp * kStages * kScaleTileBytes;
  uint64_t* my_bar = bars + warp * kStages;
  // bf16: one stage = one 64-k chunk; NF4: one stage = four chunks (16 rows x
  // 128 bytes of codes) plus the 8-block scale group that holds them.
  const int per_stage = NF4 ? 4 : 1;
  const int nst = (nch + per_stage - 1) / per_stage;
  const uint64_t pol = GRP ? policy_evict_normal() : policy_evict_first();
  auto issue = [&](int s, int st) {
    if (NF4) {
      const int cabs = c0 + 4 * st;
      mbar_expect_tx(&my_bar[s], kTileBytes + kScaleTileBytes);
      tma_load_2d(my_ring + s * kTileBytes, map, cabs * (kChunk / 2), trow, &my_bar[s], pol);
      tma_load_2d(my_sring + s * kScaleTileBytes, smap, (cabs / 8) * 8, trow, &my_bar[s], pol);
    } else {
      mbar_expect_tx(&my_bar[s], kTileBytes);
      tma_load_2d(my_ring + s * kTileBytes, map, (c0 + st) * kChunk, trow, &my_bar[s], pol);
    }
  };
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&my_bar[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // Weights are never written by the preceding kernels: start streaming
    // them before waiting on the producer of the activations.
    for (int s = 0; s < kStages && s < nst; ++s) issue(s, s);
  }
  if (NF4) {
    for (int i = tid; i < 256 * 32; i += kGemmThreads) {
      const int b = i >> 5;
      lut[i] = pack_bf16x2(__float2bfloat16_rn(c_nf4_levels[b & 15]), __float2bfloat16_rn(c_nf4_levels[b >> 4]));
    }
  }
  // Token positions (QKV: RoPE angle and cache slot), read before the wait:
  // the sequence lengths are written only by the acceptance and reset
  // kernels and by host copies, never by the kernel that directly precedes a
  // projection (the only one that can still be running at this point).
  if (EPI == EPI_QKV && tid < M) s_pos[tid] = row_slot(a.rs, m0 + tid);
  if (a.push) {
    // Rank 0's landing barrier expects every other rank's tile; the cluster
    // barrier that starts here (and is waited on only after the main loop)
    // publishes its initialisation before any rank stores into it.
    if (cluster_rank() == 0 && tid == 0) {
      mbar_init(&recv_bar, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      mbar_expect_tx(&recv_bar, (uint32_t)push_bytes(a.nsplit, M));
    }
    __syncthreads();
    cluster_arrive();
  } else {
    __syncthreads();
  }

  pdl_wait();
  trace_mark(a.rs, 1);
  pdl_launch_next();
  // The CTAs that run the epilogue: all of them, except that in a cluster
  // split only rank 0 does.
  const bool finisher = !(a.cluster && a.nsplit > 1) || cluster_rank() == 0;
  // First chunk's activations, then the epilogue's operands and the RMSNorm
  // partial sums (rows warp and warp + 8, one or two per lane), all in
  // flight together; the sums are only needed after the main loop.
  // B operand source: global memory, or this CTA's chunks staged in shared
  // memory (short K slices: one copy instead of a global round trip per chunk).
  const uint4* bsrc = a.in + (size_t)(4 * gi) * 64;   // this group's first token tile
  size_t bstride = (size_t)Tt * 64;                    // 16-byte units per chunk
  int jb = 0;                                          // chunk index of bsrc[0]
  if (sb && nch > 0) {
    stage_b_copy<T>(bstage, bsrc + (size_t)c0 * bstride, bstride, nch, tl);
    bsrc = bstage;
    bstride = (size_t)T * 64;
    jb = c0;
  }
  uint4 bq[T][2];
  if (nch > 0) load_b<T>(bq, bsrc, bstride, c0 - jb, tl, lane);
  EpiPre<T> pre;
  if (finisher) epi_prefetch<T, EPI>(a, rb, m0, M, pre, s_pos);
  float ssq_part[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  if (a.ssq && finisher) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int m = warp + 8 * j;
      if (m < M) {
        ssq_part[j][0] = lane < a.nssq ? a.ssq[lane * kRows + m0 + m] : 0.f;
        ssq_part[j][1] = lane + 32 < a.nssq ? a.ssq[(lane + 32) * kRows + m0 + m] : 0.f;
      }
    }
  }

  float acc[T][4];
#pragma unroll
  for (int t = 0; t < T; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  // Row g / g+8 of the tile, 16-byte units 2c and 2c+1 (k = 16c .. 16c+15),
  // at their 128-byte-swizzled positions.
  const int sw = g & 7;
  const int off_lo = g * 128 + (((2 * c) ^ sw) << 4);
  const int off_hi = g * 128 + (((2 * c + 1) ^ sw) << 4);
  bool timed_out = false;
  for (int st = 0; st < nst; ++st) {
    const int s = st % kStages;
    // Test hook for the error path: a first wait with no iterations always
    // gives up; the full wait that follows keeps the data and the flow intact.
    if (st == 0 && a.expire_first_wait && !mbar_wait(&my_bar[s], 0, 0)) timed_out = true;
    if (!mbar_wait(&my_bar[s], (st / kStages) & 1, kWaitIters)) timed_out = true;
    const unsigned char* tile = my_ring + s * kTileBytes;
    if (!NF4) {
      uint4 bn[T][2];
      if (st + 1 < nch) load_b<T>(bn, bsrc, bstride, c0 + st + 1 - jb, tl, lane);
      uint4 w[4];
      w[0] = *reinterpret_cast<const uint4*>(tile + off_lo);
      w[1] = *reinterpret_cast<const uint4*>(tile + off_hi);
      w[2] = *reinterpret_cast<const uint4*>(tile + 8 * 128 + off_lo);
      w[3] = *reinterpret_cast<const uint4*>(tile + 8 * 128 + off_hi);
      __syncwarp();
      if (lane == 0 && st + kStages < nst) {
        fence_proxy_async();   // the warp's reads of this stage before the async refill
        issue(s, st + kStages);
      }
      mma_chunk<T>(acc, w, bq);
      if (st + 1 < nch) {
#pragma unroll
        for (int t = 0; t < T; ++t) {
          bq[t][0] = bn[t][0];
          bq[t][1] = bn[t][1];
        }
      }
    } else {
      const __half* sct = reinterpret_cast<const __half*>(my_sring + s * kScaleTileBytes);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int ch = 4 * st + q;
        if (ch >= nch) break;
        uint4 bn[T][2];
        if (ch + 1 < nch) load_b<T>(bn, bsrc, bstride, c0 + ch + 1 - jb, tl, lane);
        // 8 code bytes (k = 16c .. 16c+15 of this chunk) of rows g and g+8,
        // at their 128-byte-swizzled positions; the scale of each row.
        const int cofs = ((((2 * q + (c >> 1)) ^ sw) << 4) + 8 * (c & 1));
        const uint2 b0 = *reinterpret_cast<const uint2*>(tile + g * 128 + cofs);
        const uint2 b1 = *reinterpret_cast<const uint2*>(tile + (g + 8) * 128 + cofs);
        const int scol = (c0 + ch) & 7;
        const float s_lo = __half2float(sct[g * 8 + scol]);
        const float s_hi = __half2float(sct[(g + 8) * 8 + scol]);
        uint4 w[4];
        const uint32_t* lt = lut + lane;
        w[0] = make_uint4(lt[(b0.x & 255) << 5], lt[((b0.x >> 8) & 255) << 5], lt[((b0.x >> 16) & 255) << 5],
                          lt[(b0.x >> 24) << 5]);
        w[1] = make_uint4(lt[(b0.y & 255) << 5], lt[((b0.y >> 8) & 255) << 5], lt[((b0.y >> 16) & 255) << 5],
                          lt[(b0.y >> 24) << 5]);
        w[2] = make_uint4(lt[(b1.x & 255) << 5], lt[((b1.x >> 8) & 255) << 5], lt[((b1.x >> 16) & 255) << 5],
                          lt[(b1.x >> 24) << 5]);
        w[3] = make_uint4(lt[(b1.y & 255) << 5], lt[((b1.y >> 8) & 255) << 5], lt[((b1.y >> 16) & 255) << 5],
                          lt[(b1.y >> 24) << 5]);
        // Levels are unscaled; one chunk shares one scale per row, applied
        // to the chunk's product before it joins the running sum.
        float part[T][4];
#pragma unroll
        for (int t = 0; t < T; ++t) part[t][0] = part[t][1] = part[t][2] = part[t][3] = 0.f;
        mma_chunk<T>(part, w, bq);
        if (ch + 1 < nch) {
#pragma unroll
          for (int t = 0; t < T; ++t) {
            bq[t][0] = bn[t][0];
            bq[t][1] = bn[t][1];
          }
        }
#pragma unroll
        for (int t = 0; t < T; ++t) {
          acc[t][0] = fmaf(s_lo, part[t][0], acc[t][0]);
          acc[t][1] = fmaf(s_lo, part[t][1], acc[t][1]);
          acc[t][2] = fmaf(s_hi, part[t][2], acc[t][2]);
          acc[t][3] = fmaf(s_hi, part[t][3], acc[t][3]);
        }
      }
      __syncwarp();
      if (lane == 0 && st + kStages < nst) {
        fence_proxy_async();
        issue(s, st + kStages);
      }
    }
  }
  if (timed_out) {
    // A tile never arrived: report, and give every copy of this warp one more
    // bounded chance to land before the CTA's shared memory is released.
    if (lane == 0) report_err(a.err, kErrWait);
    for (int st = max(0, nst - kStages); st < nst; ++st)
      mbar_wait(&my_bar[st % kStages], (st / kStages) & 1, kWaitIters);
  }

  // RMSNorm input: 1 / rms(x_m) of rows warp and warp + 8 (visible to the
  // CTA after the barrier below).
  if (a.ssq && finisher) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int m = warp + 8 * j;
      if (m < M) {
        const float sq = warp_sum(ssq_part[j][0] + ssq_part[j][1]);
        if (lane == 0) rinv[m] = 1.0f / sqrtf(sq * a.inv_k + a.eps);
      }
    }
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

  if (a.push) {
    // The K slices of this row block are the CTAs of one cluster. Every other
    // rank stores its tile into rank 0's landing area with asynchronous
    // remote stores counted on rank 0's barrier and leaves; rank 0 adds the
    // tiles in rank order.
    const uint32_t rank = cluster_rank();
    cluster_wait();
    if (rank != 0) {
      const uint32_t dst = dsmem_addr(smem_u32(recv), 0) + (rank - 1) * (uint32_t)(M * kBlockRows * 4);
      const uint32_t bar = dsmem_addr(smem_u32(&recv_bar), 0);
      const float4* mine = reinterpret_cast<const float4*>(ys);
      for (int i = tid; i < M * (kBlockRows / 4); i += kGemmThreads) st_async_v4(dst + 16 * i, mine[i], bar);
      return;
    }
    if (!mbar_wait_cluster(&recv_bar, 0, kWaitIters)) {
      // A tile never arrived: report, give the stores one more bounded
      // chance to land in this CTA's shared memory, and skip the epilogue.
      if (tid == 0) report_err(a.err, kErrWait);
      mbar_wait_cluster(&recv_bar, 0, kWaitIters);
      return;
    }
    for (int i = tid; i < M * kBlockRows; i += kGemmThreads) {
      float v = ys[i];
      for (int r = 1; r < a.nsplit; ++r) v += recv[(r - 1) * (M * kBlockRows) + i];
      ys[i] = a.ssq ? v * rinv[i / kBlockRows] : v;
    }
    __syncthreads();
  } else if (a.nsplit > 1 && a.cluster) {
    // The K slices of this row block are the CTAs of one cluster: after the
    // barrier every partial tile sits in its CTA's shared memory and rank 0
    // adds them in rank order, loading up to kG slices per round. The other
    // CTAs keep their shared memory alive until rank 0 has arrived on the
    // second barrier, which rank 0 does as soon as it has read them.
    // Rank 0 publishes nothing in the first phase: its arrival is relaxed (a
    // releasing one would also wait for its epilogue prefetch loads).
    const uint32_t rank = cluster_rank();
    if (rank != 0) {
      cluster_sync();
      cluster_arrive();
      cluster_wait();
      return;
    }
    cluster_arrive_relaxed();
    cluster_wait();
    constexpr int kE = (4 * T * kBlockRows + kGemmThreads - 1) / kGemmThreads;
    constexpr int kG = kE <= 2 ? 16 : (kE <= 4 ? 8 : 4);   // at most 32 loads in flight per thread
    const uint32_t ys_s = smem_u32(ys);
    float sum[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) sum[e] = 0.f;
    for (int p0 = 0; p0 < a.nsplit; p0 += kG) {
      float v[kG][kE];
#pragma unroll
      for (int q = 0; q < kG; ++q)
#pragma unroll
        for (int e = 0; e < kE; ++e) {
          const int i = tid + e * kGemmThreads;
          v[q][e] = (p0 + q < a.nsplit && i < M * kBlockRows) ? ld_dsmem(dsmem_addr(ys_s + 4 * i, p0 + q)) : 0.f;
        }
#pragma unroll
      for (int q = 0; q < kG; ++q)
#pragma unroll
        for (int e = 0; e < kE; ++e) sum[e] += v[q][e];
    }
    // Each thread rewrites only the elements it summed (its own loads of
    // this CTA's tile are done); the stores consume every loaded value, so
    // once they have issued the other CTAs may go (relaxed arrival).
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      const int i = tid + e * kGemmThreads;
      if (i < M * kBlockRows) ys[i] = a.ssq ? sum[e] * rinv[i / kBlockRows] : sum[e];
    }
    cluster_arrive_relaxed();
    __syncthreads();
  } else if (a.nsplit > 1) {
    float* mine = a.part + ((size_t)qb * a.nsplit + sp) * (kGroupRows * kBlockRows);
    for (int i = tid; i < M * kBlockRows; i += kGemmThreads) __stcg(mine + i, ys[i]);
    __threadfence();
    __syncthreads();
    if (tid == 0) s_flag = (atomicAdd(a.counter + qb, 1) == a.nsplit - 1);
    __syncthreads();
    if (!s_flag) return;
    __threadfence();
    // Sum the slices in fixed order 0, 1, ..., loading four slices' worth of
    // this thread's elements at a time so the loads overlap.
    const float* src = a.part + (size_t)qb * a.nsplit * (kGroupRows * kBlockRows);
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
                        ? __ldcg(src + (size_t)(p0 + q) * (kGroupRows * kBlockRows) + i)
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
      if (i < M * kBlockRows) ys[i] = a.ssq ? sum[e] * rinv[i / kBlockRows] : sum[e];
    }
    if (tid == 0) a.counter[qb] = 0;
    __syncthreads();
  }

  if (a.ssq && a.nsplit == 1) {
    // RMSNorm input without a K split: scale row m by 1 / rms(x_m) here.
    for (int i = tid; i < M * kBlockRows; i += kGemmThreads) ys[i] *= rinv[i / kBlockRows];
    __syncthreads();
  }
  if (EPI == EPI_RESID) epi_resid<T>(a, ys, rb, m0, M, Tt, pre);
  else if (EPI == EPI_QKV) epi_qkv<T>(a, ys, rb, m0, M, pre, s_pos);
  else if (EPI == EPI_SWIGLU) epi_swiglu(a, ys, rb, m0, M, Tt);
  else if (EPI == EPI_STORE) epi_store(a, ys, rb, m0, M);
  else epi_argmax(a, ys, rb, m0, M, a.nblocks * G, &s_flag);
  if (a.nsplit > 1 && a.cluster && !a.push) cluster_wait();
}

// ------------------------------------------------------------------ LM head
// Persistent form of the GEMM with the argmax epilogue, for the vocabulary
// projection (one K slice, far more 128-row blocks than CTAs): CTA b of G
// takes row blocks b, b + G, b + 2G, ...; each warp's TMA ring runs over the
// concatenated (block, chunk) sequence, so the weight stream never drains at
// a block boundary; the running best (value, index) of every token row stays
// in shared memory and is merged into the global keys once per CTA. The
// per-row arithmetic is that of k_gemm with one K slice (same chunk order,
// same MMA sequence, same 1 / rms scaling), so logits are bit-identical.
// A forward of more than 16 token rows runs one set of CTAs per 16-row group,
// interleaved in launch order (CTA i of every group side by side), so the
// groups walk the same row blocks together and share them through L2.
template <int T, bool GRP>
__global__ void __launch_bounds__(kGemmThreads, (T <= 3 ? 2 : 1)) k_lmhead(const __grid_constant__ GemmArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int kStages = a.stages;
  unsigned char* ring = smem;                                            // [8][kStages][kTileBytes]
  float* ys = reinterpret_cast<float*>(smem + 8 * kStages * kTileBytes);   // [4T][128]
  float* rinv = ys + 4 * T * kBlockRows;
  uint64_t* bars = reinterpret_cast<uint64_t*>(rinv + 4 * T);            // [8][kStages]
  uint4* bstage = reinterpret_cast<uint4*>(bars + 8 * kStages);          // staged B operand (if any)
  __shared__ unsigned long long s_best[kGroupRows];
  __shared__ int s_flag;
  trace_mark(a.rs, 0);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int nch = (a.K + kChunk - 1) / kChunk;
  const int G = GRP ? (a.rs.M + kGroupRows - 1) / kGroupRows : 1;   // token row groups
  const int Tt = GRP ? (a.rs.M + 3) / 4 : T;                     // token tiles of the fragment layout
  const int cta = GRP ? blockIdx.x / G : blockIdx.x, gi = GRP ? blockIdx.x - cta * G : 0;
  const int m0 = gi * kGroupRows;
  const int M = GRP ? min(kGroupRows, a.rs.M - m0) : a.rs.M;     // token rows of this CTA
  const int tl = GRP ? min(T, Tt - 4 * gi) : T;
  const int nc = GRP ? gridDim.x / G : gridDim.x;                // CTAs per group (launch: <= nblocks)
  const int nmine = (a.nblocks - cta + nc - 1) / nc;
  const long total = (long)nmine * nch;                             // this warp's tiles, all blocks
  unsigned char* my_ring = ring + warp * kStages * kTileBytes;
  uint64_t* my_bar = bars + warp * kStages;
  const uint64_t pol = GRP ? policy_evict_normal() : policy_evict_first();
  auto issue = [&](int s, long q) {
    const int i = (int)(q / nch), j = (int)(q - (long)i * nch);
    const int rb = cta + i * nc;
    mbar_expect_tx(&my_bar[s], kTileBytes);
    tma_load_2d(my_ring + s * kTileBytes, &a.tm[0], j * kChunk, rb * kBlockRows + 16 * warp, &my_bar[s], pol);
  };
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&my_bar[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int s = 0; s < kStages && s < total; ++s) issue(s, s);   // weights: before the wait
  }
  if (tid < kGroupRows) s_best[tid] = 0ull;
  __syncthreads();

  pdl_wait();
  trace_mark(a.rs, 1);
  pdl_launch_next();
  float ssq_part[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  if (a.ssq) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int m = warp + 8 * j;
      if (m < M) {
        ssq_part[j][0] = lane < a.nssq ? a.ssq[lane * kRows + m0 + m] : 0.f;
        ssq_part[j][1] = lane + 32 < a.nssq ? a.ssq[(lane + 32) * kRows + m0 + m] : 0.f;
      }
    }
  }
  // The B operand is the same for every block: staged once when it is small.
  const uint4* bsrc = a.in + (size_t)(4 * gi) * 64;
  size_t bstride = (size_t)Tt * 64;
  if (staged_b_bytes(T, nch)) {
    stage_b_copy<T>(bstage, bsrc, bstride, nch, tl);
    bsrc = bstage;
    bstride = (size_t)T * 64;
  }
  uint4 bq[T][2];
  load_b<T>(bq, bsrc, bstride, 0, tl, lane);

  const int sw = g & 7;
  const int off_lo = g * 128 + (((2 * c) ^ sw) << 4);
  const int off_hi = g * 128 + (((2 * c + 1) ^ sw) << 4);
  bool timed_out = false;
  long q = 0;
  for (int i = 0; i < nmine; ++i) {
    const int rb = cta + i * nc;
    float acc[T][4];
#pragma unroll
    for (int t = 0; t < T; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    for (int j = 0; j < nch; ++j, ++q) {
      const int s = (int)(q % kStages);
      const bool more = j + 1 < nch || i + 1 < nmine;
      uint4 bn[T][2];
      if (more) load_b<T>(bn, bsrc, bstride, j + 1 < nch ? j + 1 : 0, tl, lane);
      if (!mbar_wait(&my_bar[s], (uint32_t)((q / kStages) & 1), kWaitIters)) timed_out = true;
      const unsigned char* tile = my_ring + s * kTileBytes;
      uint4 w[4];
      w[0] = *reinterpret_cast<const uint4*>(tile + off_lo);
      w[1] = *reinterpret_cast<const uint4*>(tile + off_hi);
      w[2] = *reinterpret_cast<const uint4*>(tile + 8 * 128 + off_lo);
      w[3] = *reinterpret_cast<const uint4*>(tile + 8 * 128 + off_hi);
      __syncwarp();
      if (lane == 0 && q + kStages < total) {
        fence_proxy_async();   // the warp's reads of this stage before the async refill
        issue(s, q + kStages);
      }
      mma_chunk<T>(acc, w, bq);
      if (more) {
#pragma unroll
        for (int t = 0; t < T; ++t) {
          bq[t][0] = bn[t][0];
          bq[t][1] = bn[t][1];
        }
      }
    }
    if (i == 0 && a.ssq) {
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int m = warp + 8 * jj;
        if (m < M) {
          const float sq = warp_sum(ssq_part[jj][0] + ssq_part[jj][1]);
          if (lane == 0) rinv[m] = 1.0f / sqrtf(sq * a.inv_k + a.eps);
        }
      }
    }
    const int r0 = warp * 16 + g;
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const int m = 4 * t + c;
      ys[m * kBlockRows + r0] = acc[t][0] + acc[t][1];
      ys[m * kBlockRows + r0 + 8] = acc[t][2] + acc[t][3];
    }
    __syncthreads();
    for (int m = warp; m < M; m += kGemmThreads / 32) {
      unsigned long long best = 0ull;
      bool bad = false;
      const int mb = (m0 + m) / a.rs.rps, mj = (m0 + m) - mb * a.rs.rps;
      const int lg_row = mj >= a.tok_skip ? mb * a.lg_stride + a.lg_off + mj - a.tok_skip : -1;
      const float sc = a.ssq ? rinv[m] : 1.f;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int r = lane + 32 * jj;
        const int n = rb * kBlockRows + r;
        if (n < a.N) {
          const float v = a.ssq ? ys[m * kBlockRows + r] * sc : ys[m * kBlockRows + r];
          if (a.logits && lg_row >= 0) a.logits[(size_t)lg_row * a.N + n] = v;
          bad |= !isfinite(v);
          const unsigned long long k = argmax_key(v, n);
          best = k > best ? k : best;
        }
      }
      best = shfl_max_u64(best);
      if (__any_sync(0xffffffffu, bad) && lane == 0) report_err(a.err, kErrNonfinite);
      if (lane == 0 && best > s_best[m]) s_best[m] = best;
    }
    __syncthreads();   // ys is free for the next block
  }
  if (timed_out) {
    if (lane == 0) report_err(a.err, kErrWait);
    for (long st = (total > kStages ? total - kStages : 0); st < total; ++st)
      mbar_wait(&my_bar[st % kStages], (uint32_t)((st / kStages) & 1), kWaitIters);
  }
  // Merge the CTA's bests; the last CTA to arrive writes the tokens and
  // leaves the keys and the counter at zero for the next launch.
  if (tid < M) atomicMax(a.keys + m0 + tid, s_best[tid]);
  __threadfence();
  __syncthreads();
  if (tid == 0) s_flag = (atomicAdd(a.done, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!s_flag) return;
  __threadfence();
  if (tid < a.rs.M) {
    const int m = tid;
    const unsigned long long k = atomicExch(a.keys + m, 0ull);
    const int b = m / a.rs.rps, j = m - b * a.rs.rps;
    if (j >= a.tok_skip) a.tok_out[b * a.tok_stride + a.tok_off + j - a.tok_skip] = key_index(k);
  }
  if (tid == 0) *a.done = 0;
}

int gemm_smem_bytes(int M, int stages, bool nf4, int cps, int push) {
  const int T = (std::min(M, kGroupRows) + 3) / 4;   // token tiles of one row group
  return 1024 /* alignment slack */ + 8 * stages * (kTileBytes + (nf4 ? kScaleTileBytes : 0)) +
         4 * T * kBlockRows * 4 + 4 * T * 4 + 8 * stages * 8 + staged_b_bytes(T, cps) + push;
}

cudaError_t set_nf4_levels(const float levels[16]) {
  return cudaMemcpyToSymbol(c_nf4_levels, levels, 16 * sizeof(float));
}

static cudaError_t encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                             uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                             CUtensorMapSwizzle sw) {
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
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_weight_map(CUtensorMap* map, const void* w, int rows, int K, int ld, int box_rows) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w, K, rows, (uint64_t)ld * 2, kChunk, box_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

int nf4_scale_ld(int K) { return ((K / 64 + 7) / 8) * 8; }

cudaError_t make_kv_map(CUtensorMap* map, const void* kv, long rows, int hd, int box_rows) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kv, hd, (uint64_t)rows, (uint64_t)hd * 2, 64, box_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t make_nf4_maps(CUtensorMap* codes_map, CUtensorMap* scale_map, const void* codes, const void* scales,
                          int rows, int K, int box_rows) {
  cudaError_t e = encode_2d(codes_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, K / 2, rows, K / 2, 128, box_rows,
                            CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  return encode_2d(scale_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, scales, K / 64, rows, (uint64_t)nf4_scale_ld(K) * 2,
                   8, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int T, int EPI, bool NF4, bool GRP>
static cudaError_t launch_t(const GemmArgs& a, cudaStream_t st, bool pdl) {
  const int G = (a.rs.M + kGroupRows - 1) / kGroupRows;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nblocks * a.nsplit * G);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = gemm_smem_bytes(4 * T, a.stages, NF4, a.stage_b ? a.cps : 0,
                                         a.push ? push_bytes(a.nsplit, std::min(a.rs.M, kGroupRows)) : 0);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (a.cluster && a.nsplit > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = a.nsplit;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, k_gemm<T, EPI, NF4, GRP>, a);
}

template <int T, int EPI, bool NF4, bool GRP>
static cudaError_t init_one() {
  const int smem = gemm_smem_bytes(4 * T, NF4 ? kMaxStagesNF4 : kMaxStages, NF4, 0, kMaxPushBytes) + kMaxStagedB;
  cudaError_t e = cudaFuncSetAttribute(k_gemm<T, EPI, NF4, GRP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // Every kernel of the chain asks for the largest shared-memory carve-out,
  // so an SM running one of them can take the next kernel's CTAs early
  // (programmatic dependent launch) without first changing its L1 / shared split.
  e = cudaFuncSetAttribute(k_gemm<T, EPI, NF4, GRP>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_gemm<T, EPI, NF4, GRP>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <int T, bool NF4, bool GRP = false>
static cudaError_t init_t() {
  cudaError_t e;
  if ((e = init_one<T, EPI_QKV, NF4, GRP>()) || (e = init_one<T, EPI_RESID, NF4, GRP>()) ||
      (e = init_one<T, EPI_SWIGLU, NF4, GRP>()) || (e = init_one<T, EPI_STORE, NF4, GRP>()))
    return e;
  return init_one<T, EPI_ARGMAX, NF4, GRP>();
}

// Largest number of clusters of `csize` CTAs that can be resident at once
// for a launch with this shared-memory footprint (clusters are placed within
// GPCs, so this can be below SMs x CTAs per SM / csize). Measured on the
// 9..12-row instantiation with the QKV epilogue (the most registers of the
// two-CTAs-per-SM kernels); 0 if the query fails.
int gemm_max_clusters(int csize, int M, int stages, int cps) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize * 512);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = gemm_smem_bytes(M, stages, false, cps);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = csize;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  return cudaOccupancyMaxActiveClusters(&n, k_gemm<3, EPI_QKV, false, false>, &cfg) == cudaSuccess ? n : 0;
}

template <int T, bool GRP = false>
static cudaError_t init_lm() {
  const int smem = gemm_smem_bytes(4 * T, kMaxStages, false, 0) + kMaxStagedB;
  cudaError_t e = cudaFuncSetAttribute(k_lmhead<T, GRP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_lmhead<T, GRP>, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

// Raise the dynamic shared-memory limit of every instantiation (current device).
static cudaError_t gemm_init_all() {
  cudaError_t e;
  if ((e = init_lm<1>()) || (e = init_lm<2>()) || (e = init_lm<3>()) || (e = init_lm<4>()) ||
      (e = init_lm<4, true>()))
    return e;
  if ((e = init_t<1, false>()) || (e = init_t<2, false>()) || (e = init_t<3, false>()) ||
      (e = init_t<4, false>()) || (e = init_t<1, true>()) || (e = init_t<2, true>()) ||
      (e = init_t<3, true>()) || (e = init_t<4, true>()) || (e = init_t<4, false, true>()) ||
      (e = init_t<4, true, true>()))
    return e;
  if ((e = f32_init()) != cudaSuccess) return e;
  return umma_init();
}

// Once per device (the attributes persist for the process): about 130
// attribute calls, too slow to repeat before every sf_linear launch.
cudaError_t gemm_init() {
  static std::mutex mu;
  static bool done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return gemm_init_all();
  std::lock_guard<std::mutex> lk(mu);
  if (done[dev]) return cudaSuccess;
  if ((e = gemm_init_all()) != cudaSuccess) return e;
  done[dev] = true;
  return cudaSuccess;
}

template <int EPI, bool NF4>
static cudaError_t launch_e(const GemmArgs& a, cudaStream_t st, bool pdl) {
  if (a.rs.M > kGroupRows) return launch_t<4, EPI, NF4, true>(a, st, pdl);
  switch ((a.rs.M + 3) / 4) {
    case 1: return launch_t<1, EPI, NF4, false>(a, st, pdl);
    case 2: return launch_t<2, EPI, NF4, false>(a, st, pdl);
    case 3: return launch_t<3, EPI, NF4, false>(a, st, pdl);
    case 4: return launch_t<4, EPI, NF4, false>(a, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <bool NF4>
static cudaError_t launch_f(const GemmArgs& a, int epi, cudaStream_t st, bool pdl) {
  switch (epi) {
    case EPI_QKV: return launch_e<EPI_QKV, NF4>(a, st, pdl);
    case EPI_RESID: return launch_e<EPI_RESID, NF4>(a, st, pdl);
    case EPI_SWIGLU: return launch_e<EPI_SWIGLU, NF4>(a, st, pdl);
    case EPI_ARGMAX: return launch_e<EPI_ARGMAX, NF4>(a, st, pdl);
    case EPI_STORE: return launch_e<EPI_STORE, NF4>(a, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

// One thread per 16-byte unit of the output: fragment order, or (umma) the
// tensor-core operand order (umma_index).
__global__ void k_to_frag(const float* x, int M, int K, int ld, int T, uint4* out, long units, int umma) {
  const long u = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  int m, k0, lo;
  if (umma) {   // T counts 8-token tiles here
    const int pos = (int)(u & 7), row = (int)((u >> 3) & 7);
    const long r = u >> 6;
    const int t = (int)(r % T), j = (int)(r / T);
    m = 8 * t + row;
    lo = 0;
    k0 = 64 * j + 8 * (pos ^ row);
  } else {
    const int lane = (int)(u & 31);
    const int h = (int)((u >> 5) & 1);
    const long r = u >> 6;
    const int t = (int)(r % T), j = (int)(r / T);
    const int col = lane >> 2, c = lane & 3;
    m = 4 * t + (col >> 1);
    lo = col & 1;
    k0 = 64 * j + 16 * c + 8 * h;
  }
  uint32_t p[4];
#pragma unroll
  for (int e2 = 0; e2 < 4; ++e2) {
    bf16 v2[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int k = k0 + 2 * e2 + q;
      const float v = (m < M && k < K) ? x[(size_t)m * ld + k] : 0.f;
      const bf16 hi = __float2bfloat16_rn(v);
      v2[q] = lo ? __float2bfloat16_rn(v - __bfloat162float(hi)) : hi;
    }
    p[e2] = pack_bf16x2(v2[0], v2[1]);
  }
  out[u] = make_uint4(p[0], p[1], p[2], p[3]);
}

cudaError_t launch_to_frag(const float* x, int M, int K, int ld, bf16* out, cudaStream_t st) {
  const int umma = M >= umma_min_rows() ? 1 : 0;
  const int T = umma ? (M + 7) / 8 : (M + 3) / 4;
  const long units = (long)frag_bytes(K, T) / 16;
  k_to_frag<<<(unsigned)((units + 255) / 256), 256, 0, st>>>(x, M, K, ld, T, reinterpret_cast<uint4*>(out), units,
                                                            umma);
  return cudaGetLastError();
}

// ctas: CTAs of the whole launch (per row group x row groups).
template <int T, bool GRP>
static cudaError_t launch_lm_t(const GemmArgs& a, int ctas, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = gemm_smem_bytes(4 * T, a.stages, false, (a.K + kChunk - 1) / kChunk);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_lmhead<T, GRP>, a);
}

cudaError_t launch_lmhead(const GemmArgs& a, int num_sms, cudaStream_t st, bool pdl) {
  const int T = (std::min(a.rs.M, kGroupRows) + 3) / 4;
  const int G = (a.rs.M + kGroupRows - 1) / kGroupRows;
  if (a.rs.M < 1 || a.rs.M > kRows || a.nf4 || a.stages < 2 || a.stages > kMaxStages) return cudaErrorInvalidValue;
  const int ctas = G * std::max(1, std::min(a.nblocks, (T <= 3 ? 2 : 1) * num_sms / G));
  if (G > 1) return launch_lm_t<4, true>(a, ctas, st, pdl);
  switch (T) {
    case 1: return launch_lm_t<1, false>(a, ctas, st, pdl);
    case 2: return launch_lm_t<2, false>(a, ctas, st, pdl);
    case 3: return launch_lm_t<3, false>(a, ctas, st, pdl);
    default: return launch_lm_t<4, false>(a, ctas, st, pdl);
  }
}

cudaError_t launch_gemm(const GemmArgs& a, int epi, cudaStream_t st, bool pdl) {
  if (a.rs.M < 1 || a.rs.M > kRows) return cudaErrorInvalidValue;
  if (a.cluster && a.nsplit > kMaxClusterSplit) return cudaErrorInvalidValue;
  if (a.stages < 2 || a.stages > (a.nf4 ? kMaxStagesNF4 : kMaxStages)) return cudaErrorInvalidValue;
  if (a.nf4 && (a.K % 64 || (a.cps * a.nsplit > 1 && a.cps % 4))) return cudaErrorInvalidValue;
  // Push when the landing area fits and keeps the CTA within half an SM's
  // shared memory (two CTAs per SM: this kernel's and the next one's, or two
  // of this kernel's); otherwise rank 0 pulls the tiles.
  // Staging the B operand and the landing area compete for that space; the
  // push reduction wins when both do not fit.
  GemmArgs b = a;
  const int mg = std::min(a.rs.M, kGroupRows);   // token rows of one CTA
  const int pb = push_bytes(a.nsplit, mg);
  const bool split = a.cluster && a.nsplit > 1 && pb <= kMaxPushBytes;
  b.stage_b = staged_b_bytes((mg + 3) / 4, a.cps) > 0;
  b.push = split && gemm_smem_bytes(a.rs.M, a.stages, a.nf4, a.cps, pb) <= kHalfSmBytes;
  if (split && !b.push && gemm_smem_bytes(a.rs.M, a.stages, a.nf4, 0, pb) <= kHalfSmBytes) {
    b.stage_b = 0;
    b.push = 1;
  }
  return b.nf4 ? launch_f<true>(b, epi, st, pdl) : launch_f<false>(b, epi, st, pdl);
}

}  // namespace sf
