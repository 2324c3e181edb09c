// The weight-streaming GEMM on the tcgen05 tensor cores, for forwards of more
// than 16 token rows (the verify pass of a batch of sequences, prefill
// chunks) and for every forward with NF4 weights: y[m][n] = sum_k x[m][k]
// W[n][k] for every token row m (up to SF_MAX_ROWS) in one CTA per (128
// weight rows, K slice).
//
// The mma.sync kernel (k_gemm.cu) covers at most 16 token rows per CTA, so a
// 72-row verify ran as five row groups that each streamed (from L2) and, for
// NF4 weights, dequantised every weight tile again. Here the whole token
// block is the N side of one MMA: M = 128 weight rows, N = one column per
// token (bf16 activations; rounded up to a multiple of 16), accumulated in
// tensor memory, so every weight tile is read and dequantised once.
//
// Warp roles, 256 threads (bf16 weights) or 384 (NF4):
//   thread 0      producer: weight tiles by TMA (two 64-row boxes, 128-byte
//                 swizzle) or NF4 code tiles + block scales, and the token
//                 operand of each 64-k chunk by one bulk copy (the producers
//                 of the activations store them in exactly the tile layout
//                 the MMA reads: umma_index in sf_common.cuh);
//   thread 32     MMA issuer: four tcgen05.mma (K = 16 each) per chunk,
//                 tcgen05.commit to the stage's "empty" barrier;
//   warps 4-11    NF4 only: dequantise each chunk's codes (thread r of warps
//                 4-7 and of warps 8-11 = weight row r, the first group the
//                 chunk's elements 0-31, the second 32-63: one lookup of a
//                 per-lane table of bf16 level pairs and one bf16x2 multiply
//                 by the block scale per two codes) and write the bf16 tile
//                 straight into tensor memory (tcgen05.st), four chunks deep;
//                 the MMA reads A from there;
//   warps 4-7(11) afterwards: read the accumulator (tcgen05.ld, one weight
//                 row per thread, one column per token; NF4: the two groups
//                 take alternate 16-column blocks) and write the CTA's tile
//                 ys[m][128] in shared memory.
// Then all threads sum the K slices (thread-block cluster, rank 0 reads the
// other ranks' tiles; or global partial tiles and an arrival counter) and
// apply the RMSNorm row factor; the first 256 run the same epilogues as
// k_gemm, one 16-row group at a time.
#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "gemm_epi.cuh"
#include "umma.cuh"

namespace sf {

namespace {

constexpr uint32_t kUWaitIters = 1u << 24;
constexpr int kUThreads = 256;              // bf16 weights
constexpr int kUThreadsNf4 = 384;           // NF4: eight dequantising warps
template <bool NF4> __host__ __device__ constexpr int uthreads() { return NF4 ? kUThreadsNf4 : kUThreads; }
constexpr int kUMaxStages = 6;
constexpr int kATileBytes = 128 * 128;      // 128 weight rows x 64 k bf16 (also 128 rows x 256 k of NF4 codes)
constexpr int kUScaleBytes = 128 * 16;      // NF4: 128 rows x 8 fp16 block scales
constexpr int kCodeStage = kATileBytes + kUScaleBytes;
constexpr int kCodeStages = 2;
constexpr int kDeqStages = 4;               // NF4: dequantised chunks in tensor memory
constexpr int kLutBytes = 256 * 32 * 4;     // NF4: byte -> bf16 level pair, one copy per lane
constexpr int kAccCols = 128;               // tensor-memory columns of the accumulator (N <= 128)
constexpr int kNf4Cols = 256;               // NF4: accumulator + kDeqStages x 32 columns of A

__constant__ float c_levels[16];

struct USmem {
  uint64_t full[kUMaxStages], empty[kUMaxStages];   // token operand (+ bf16 weights) ring
  uint64_t cfull[kCodeStages], cempty[kCodeStages];   // NF4 code ring
  uint64_t afull[kDeqStages], aempty[kDeqStages];     // NF4 dequantised weight ring
  uint64_t acc;                                       // accumulator complete
  uint32_t tmem;
  int flag;
  int pos[kRows];
  float rinv[kRows];
};

__device__ __forceinline__ int tiles_padded(int T) { return (T + 1) & ~1; }

// Tensor map, first weight row and row of the second 64-row box of row block
// rb: SwiGLU blocks are 64 gate rows then the same 64 features' up rows.
template <int EPI>
__device__ __forceinline__ void block_rows(const GemmArgs& a, int rb, int* seg_lo, int* row_lo, int* seg_hi,
                                           int* row_hi) {
  if (EPI == EPI_SWIGLU) {
    *seg_lo = 0;
    *seg_hi = 1;
    *row_lo = *row_hi = rb * 64;
    return;
  }
  const int n = rb * kBlockRows;
  int s = 0;
  while (s < a.nseg - 1 && n >= a.seg_end[s]) ++s;
  *seg_lo = *seg_hi = s;
  *row_lo = n - (s ? a.seg_end[s - 1] : 0);
  *row_hi = *row_lo + 64;
}

}  // namespace

template <int EPI, bool NF4>
__global__ void __launch_bounds__(uthreads<NF4>(), 2) k_umma(const __grid_constant__ GemmArgs a) {
  constexpr int kThr = uthreads<NF4>();
  extern __shared__ unsigned char usmem_raw[];
  unsigned char* base = usmem_raw + ((1024 - (smem_u32(usmem_raw) & 1023)) & 1023);
  __shared__ USmem sm;
  trace_mark(a.rs, 0);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int M = a.rs.M;
  const int T = (M + 7) / 8;              // 8-token tiles of the operand layout
  const int T4 = (M + 3) / 4;             // the fragment layout's tile count (epilogue stores)
  const int Tp = tiles_padded(T);         // MMA N = 8 * Tp (a multiple of 16)
  const int N = 8 * Tp;
  const int ncols = NF4 ? kNf4Cols : (N <= 32 ? 32 : (N <= 64 ? 64 : (N <= 128 ? 128 : 256)));
  const int S = a.stages;
  const int rb = blockIdx.x / a.nsplit, sp = blockIdx.x - rb * a.nsplit;
  const int nch_total = (a.K + kChunk - 1) / kChunk;
  const int c0 = sp * a.cps;
  const int nch = min(a.cps, nch_total - c0);
  const uint32_t btile = (uint32_t)T * 1024;   // bytes of one chunk's token operand

  // Shared memory: bf16: S stages of [weights 16 KB | tokens Tp KB];
  // NF4: 2 code stages [codes 16 KB | scales 2 KB], the level-pair table
  // (32 KB), S token stages of Tp KB. The result tile ys aliases it.
  const int bstage = Tp * 1024;
  auto wtile = [&](int s) -> unsigned char* { return base + (size_t)s * (kATileBytes + bstage); };
  auto btile_p = [&](int s) -> unsigned char* {
    return NF4 ? base + kCodeStages * kCodeStage + kLutBytes + (size_t)s * bstage : wtile(s) + kATileBytes;
  };
  auto ctile = [&](int s) -> unsigned char* { return base + (size_t)s * kCodeStage; };
  uint32_t* lut = reinterpret_cast<uint32_t*>(base + kCodeStages * kCodeStage);   // [256][32]
  float* ys = reinterpret_cast<float*>(base);

  int seg_lo, row_lo, seg_hi, row_hi;
  block_rows<EPI>(a, rb, &seg_lo, &row_lo, &seg_hi, &row_hi);

  if (warp == 0) {
    tmem_alloc(&sm.tmem, ncols);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < kCodeStages; ++s) {
      mbar_init(&sm.cfull[s], 1);
      mbar_init(&sm.cempty[s], 8);   // one arrival per dequantising warp
    }
    for (int s = 0; s < kDeqStages; ++s) {
      mbar_init(&sm.afull[s], 8);
      mbar_init(&sm.aempty[s], 1);
    }
    mbar_init(&sm.acc, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // An odd tile count leaves the last tile of every token stage unwritten by
  // the copies: it reads as zero columns.
  if (Tp > T)
    for (int i = tid; i < S * 64; i += kThr)
      reinterpret_cast<uint4*>(btile_p(i / 64) + (size_t)T * 1024)[i % 64] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async();
  // Token positions (QKV epilogue), read before the wait: lengths are never
  // written by the kernel that directly precedes a projection.
  if (EPI == EPI_QKV && tid < M) sm.pos[tid] = row_slot(a.rs, tid);
  if (NF4) {
    // Entry b of lane l at 32 b + l: every lookup of a warp hits its own bank.
    for (int i = tid; i < 256 * 32; i += kThr) {
      const int b = i >> 5;
      lut[i] = pack_bf16x2(__float2bfloat16_rn(c_levels[b & 15]), __float2bfloat16_rn(c_levels[b >> 4]));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;

  const uint64_t pol_w = policy_evict_first();
  const uint64_t pol_b = policy_evict_normal();
  const int ncg = (nch + 3) / 4;          // NF4 code groups of this slice
  (void)ncg;
  auto issue_codes = [&](int q) {
    const int s = q % kCodeStages;
    const int cabs = c0 + 4 * q;
    mbar_expect_tx(&sm.cfull[s], kCodeStage);
    tma_load_2d(ctile(s), &a.tm[seg_lo], cabs * (kChunk / 2), row_lo, &sm.cfull[s], pol_w);
    tma_load_2d(ctile(s) + kATileBytes / 2, &a.tm[seg_hi], cabs * (kChunk / 2), row_hi, &sm.cfull[s], pol_w);
    tma_load_2d(ctile(s) + kATileBytes, &a.tms[seg_lo], (cabs / 8) * 8, row_lo, &sm.cfull[s], pol_w);
    tma_load_2d(ctile(s) + kATileBytes + kUScaleBytes / 2, &a.tms[seg_hi], (cabs / 8) * 8, row_hi, &sm.cfull[s],
                pol_w);
  };
  auto issue_w = [&](int st) {
    const int s = st % S;
    tma_load_2d(wtile(s), &a.tm[seg_lo], (c0 + st) * kChunk, row_lo, &sm.full[s], pol_w);
    tma_load_2d(wtile(s) + kATileBytes / 2, &a.tm[seg_hi], (c0 + st) * kChunk, row_hi, &sm.full[s], pol_w);
  };
  auto issue_b = [&](int st) {
    bulk_load(btile_p(st % S), reinterpret_cast<const unsigned char*>(a.in) + (size_t)(c0 + st) * btile, btile,
              &sm.full[st % S], pol_b);
  };
  const int pre = min(S, nch);
  // Weights are never written by the preceding kernels: start them first.
  if (tid == 0) {
    if (NF4) {
      for (int q = 0; q < kCodeStages && q < ncg; ++q) issue_codes(q);
      for (int st = 0; st < pre; ++st) mbar_expect_tx(&sm.full[st], btile);
    } else {
      for (int st = 0; st < pre; ++st) {
        mbar_expect_tx(&sm.full[st], kATileBytes + btile);
        issue_w(st);
      }
    }
  }
  pdl_wait();
  trace_mark(a.rs, 1);
  pdl_launch_next();

  bool timed_out = false;
  if (tid == 0) {
    // ---- producer. NF4 code group q (chunks 4q .. 4q+3) reuses code stage
    // q % 2 once the dequantisers released group q - 2; token stage s is
    // refilled once the MMAs of chunk st - S committed.
    for (int st = 0; st < nch; ++st) {
      const int s = st % S;
      if (NF4 && (st & 3) == 0 && st / 4 >= kCodeStages) {
        const int q = st / 4;
        if (!mbar_wait(&sm.cempty[q % kCodeStages], ((q / kCodeStages) + 1) & 1, kUWaitIters)) timed_out = true;
        issue_codes(q);
      }
      if (st >= pre) {
        if (!mbar_wait(&sm.empty[s], ((st / S) + 1) & 1, kUWaitIters)) timed_out = true;
        mbar_expect_tx(&sm.full[s], NF4 ? btile : kATileBytes + btile);
        if (!NF4) issue_w(st);
      }
      issue_b(st);
    }
  } else if (tid == 32) {
    // ---- MMA issuer
    const uint32_t idesc = umma_idesc_bf16(128, N);
    for (int st = 0; st < nch; ++st) {
      const int s = st % S;
      // Test hook for the error path (as in k_gemm): the first wait gives up at once.
      if (st == 0 && a.expire_first_wait && !mbar_wait(&sm.full[s], 0, 0)) timed_out = true;
      if (!mbar_wait(&sm.full[s], (st / S) & 1, kUWaitIters)) timed_out = true;
      const int ds = st % kDeqStages;
      if (NF4 && !mbar_wait(&sm.afull[ds], (st / kDeqStages) & 1, kUWaitIters)) timed_out = true;
      tc_fence_after();
      const uint32_t bw = smem_u32(btile_p(s));
      if (NF4) {
        const uint32_t at = tmem + kAccCols + 32 * ds;   // A: 64 k = 32 columns per chunk
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_tmem_a(tmem, at + 8 * kk, sw128_desc(bw + 32 * kk), idesc, (st | kk) != 0);
      } else {
        const uint32_t aw = smem_u32(wtile(s));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem, sw128_desc(aw + 32 * kk), sw128_desc(bw + 32 * kk), idesc, (st | kk) != 0);
      }
      umma_commit(&sm.empty[s]);
      if (NF4) umma_commit(&sm.aempty[ds]);
    }
    umma_commit(&sm.acc);
  } else if (NF4 && warp >= 4) {
    // ---- dequantisers: warps 4-7 and 8-11; thread r of a group owns weight
    // row r = tensor-memory lane r, the first group columns 0-15 of every
    // chunk (elements 0-31), the second columns 16-31 (elements 32-63).
    const int quarter = warp & 3, h = (warp - 4) >> 2;
    const int r = 32 * quarter + lane;
    const int sw = r & 7;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
    const uint32_t lut_lane = smem_u32(lut) + 4 * lane;
    for (int st = 0; st < nch; ++st) {
      const int q = st >> 2, sub = st & 3, cs = q % kCodeStages, ds = st % kDeqStages;
      if (sub == 0 && !mbar_wait(&sm.cfull[cs], (q / kCodeStages) & 1, kUWaitIters)) timed_out = true;
      if (!mbar_wait(&sm.aempty[ds], ((st / kDeqStages) + 1) & 1, kUWaitIters)) timed_out = true;
      tc_fence_after();
      const unsigned char* crow = ctile(cs) + (r >> 3) * 1024 + sw * 128;
      const uint4 bw = *reinterpret_cast<const uint4*>(crow + (((2 * sub + h) ^ sw) << 4));
      const __half* sc = reinterpret_cast<const __half*>(ctile(cs) + kATileBytes) + r * 8;
      const bf16 sb = __float2bfloat16_rn(__half2float(sc[(c0 + st) & 7]));
      const uint32_t scale2 = pack_bf16x2(sb, sb);
      // Column j of the chunk: elements 2j (low nibble of code byte j) and
      // 2j + 1. Table entry b of this lane at shared address lut_lane + 128 b.
      const uint32_t cw[4] = {bw.x, bw.y, bw.z, bw.w};
      uint32_t av[16];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t idx, v;
          asm("bfe.u32 %0, %1, %2, 8;" : "=r"(idx) : "r"(cw[c]), "r"(8 * e));
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(lut_lane + (idx << 7)));
          av[4 * c + e] = bf16x2_mul(v, scale2);
        }
      tmem_st16(lane_addr + kAccCols + 32 * ds + 16 * h, av);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.afull[ds]);
        if (sub == 3 || st == nch - 1) mbar_arrive(&sm.cempty[cs]);
      }
    }
  }

  // ---- accumulator -> ys[m][128] (warps 4-7, and 8-11 with NF4 taking every
  // other 16 columns: lane 32 * (warp % 4) + lane = weight row)
  if (warp >= 4) {
    if (!mbar_wait(&sm.acc, 0, kUWaitIters)) {
      timed_out = true;
      mbar_wait(&sm.acc, 0, kUWaitIters);
    }
    tc_fence_after();
    const int row = 32 * (warp & 3) + lane;
    const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const int ngroups = kThr / 128 - 1;   // drain groups of four warps: 1 (bf16) or 2 (NF4)
    for (int c16 = (warp - 4) >> 2; c16 < N / 16; c16 += ngroups) {
      uint32_t v[16];
      tmem_ld16(taddr + 16 * c16, v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int m = 16 * c16 + i;
        if (m < M) ys[m * kBlockRows + row] = __uint_as_float(v[i]);
      }
    }
  }
  if (timed_out) report_err(a.err, kErrWait);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }

  // ---- RMSNorm row factors 1 / rms(x_m)
  if (a.ssq)
    for (int m = warp; m < M; m += kThr / 32) {
      float sq = (lane < a.nssq ? a.ssq[lane * kRows + m] : 0.f) + (lane + 32 < a.nssq ? a.ssq[(lane + 32) * kRows + m] : 0.f);
      sq = warp_sum(sq);
      if (lane == 0) sm.rinv[m] = 1.0f / sqrtf(sq * a.inv_k + a.eps);
    }
  __syncthreads();

  // ---- sum the K slices in slice order, scale rows by 1 / rms, epilogue
  const int nel = M * kBlockRows;
  const int G = (M + kGroupRows - 1) / kGroupRows;
  auto epilogue = [&](int m0) {   // one 16-row group (the k_gemm epilogues)
    const int Mg = min(kGroupRows, M - m0);
    float* yg = ys + m0 * kBlockRows;
    EpiPre<4> pre_g;
    epi_prefetch<4, EPI>(a, rb, m0, Mg, pre_g, sm.pos + m0);
    if (EPI == EPI_RESID) epi_resid<4>(a, yg, rb, m0, Mg, T4, pre_g);
    else if (EPI == EPI_QKV) epi_qkv<4>(a, yg, rb, m0, Mg, pre_g, sm.pos + m0);
    else if (EPI == EPI_SWIGLU) epi_swiglu(a, yg, rb, m0, Mg, T4);
    else if (EPI == EPI_ARGMAX) epi_argmax(a, yg, rb, m0, Mg, a.nblocks * G, &sm.flag);   // every (block, group) once
    else epi_store(a, yg, rb, m0, Mg);
  };
  if (a.nsplit > 1 && a.cluster) {
    // The K slices of this row block are the CTAs of one cluster. The sum is
    // spread over the ranks: rank r adds 16-row groups r, r + nsplit, ...
    // from every rank's tile (ranks in order, 16-byte remote loads all in
    // flight together), writes them into its own tile and runs their
    // epilogue; a last barrier keeps every tile alive until all have read.
    cluster_sync();
    const uint32_t rank = cluster_rank();
    const uint32_t ys_s = smem_u32(ys);
    for (int g = (int)rank; g < G; g += a.nsplit) {
      const int m0 = g * kGroupRows, Mg = min(kGroupRows, M - m0);
      for (int i = tid; i < Mg * (kBlockRows / 4); i += kThr) {
        const int e = m0 * (kBlockRows / 4) + i;   // float4 index in the tile
        float4 v[8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r < a.nsplit) v[r] = ld_dsmem_v4(dsmem_addr(ys_s + 16 * e, r));
        float4 acc = v[0];
#pragma unroll
        for (int r = 1; r < 8; ++r)
          if (r < a.nsplit) {
            acc.x += v[r].x;
            acc.y += v[r].y;
            acc.z += v[r].z;
            acc.w += v[r].w;
          }
        if (a.ssq) {
          const float f = sm.rinv[(4 * e) / kBlockRows];
          acc.x *= f;
          acc.y *= f;
          acc.z *= f;
          acc.w *= f;
        }
        reinterpret_cast<float4*>(ys)[e] = acc;
      }
    }
    __syncthreads();
    if (tid < kGemmThreads)   // the epilogues' own barriers count kGemmThreads threads
      for (int g = (int)rank; g < G; g += a.nsplit) epilogue(g * kGroupRows);
    cluster_sync();
    return;
  }
  if (a.nsplit > 1) {
    for (int i = tid; i < nel; i += kThr) {
      const int m = i / kBlockRows, g = m / kGroupRows;
      __stcg(a.part + (((size_t)(rb * G + g) * a.nsplit + sp) * kGroupRows + (m - g * kGroupRows)) * kBlockRows +
                 (i - m * kBlockRows),
             ys[i]);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) sm.flag = (atomicAdd(a.counter + rb * G, 1) == a.nsplit - 1);
    __syncthreads();
    if (!sm.flag) return;
    __threadfence();
    // The last CTA of the row block adds the slices in order, 16-byte loads
    // of up to eight slices in flight at once.
    const int n4 = nel / 4;
    for (int i = tid; i < n4; i += kThr) {
      const int m = (4 * i) / kBlockRows, g = m / kGroupRows;
      const float4* src = reinterpret_cast<const float4*>(
          a.part + ((size_t)(rb * G + g) * a.nsplit * kGroupRows + (m - g * kGroupRows)) * kBlockRows +
          (4 * i - m * kBlockRows));
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int p0 = 0; p0 < a.nsplit; p0 += 8) {
        float4 v[8];
#pragma unroll
        for (int p = 0; p < 8; ++p)
          if (p0 + p < a.nsplit) v[p] = __ldcg(src + (size_t)(p0 + p) * (kGroupRows * kBlockRows / 4));
#pragma unroll
        for (int p = 0; p < 8; ++p)
          if (p0 + p < a.nsplit) {
            acc.x += v[p].x;
            acc.y += v[p].y;
            acc.z += v[p].z;
            acc.w += v[p].w;
          }
      }
      const float f = a.ssq ? sm.rinv[m] : 1.f;
      reinterpret_cast<float4*>(ys)[i] = make_float4(acc.x * f, acc.y * f, acc.z * f, acc.w * f);
    }
    if (tid == 0) a.counter[rb * G] = 0;
  } else if (a.ssq) {
    for (int i = tid; i < nel; i += kThr) ys[i] *= sm.rinv[i / kBlockRows];
  }
  __syncthreads();
  if (tid < kGemmThreads)   // the epilogues' own barriers count kGemmThreads threads
    for (int m0 = 0; m0 < M; m0 += kGroupRows) epilogue(m0);
}

// Dynamic shared memory of a launch (plus 1 KB for the 1024-byte alignment).
int umma_smem_bytes(int M, int stages, bool nf4) {
  const int Tp = ((M + 7) / 8 + 1) & ~1;
  const int ring = nf4 ? kCodeStages * kCodeStage + kLutBytes + stages * Tp * 1024
                       : stages * (kATileBytes + Tp * 1024);
  return 1024 + std::max(ring, M * kBlockRows * 4);
}

// Deepest token ring that keeps two CTAs on an SM (each at most kHalfSmBytes).
int umma_stages(int M, bool nf4) {
  int s = kUMaxStages;
  while (s > 2 && umma_smem_bytes(M, s, nf4) > kHalfSmBytes) --s;
  return s;
}

cudaError_t set_umma_nf4_levels(const float levels[16]) {
  return cudaMemcpyToSymbol(c_levels, levels, 16 * sizeof(float));
}

template <int EPI, bool NF4>
static cudaError_t launch_ut(const GemmArgs& a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nblocks * a.nsplit);
  cfg.blockDim = dim3(uthreads<NF4>());
  cfg.dynamicSmemBytes = umma_smem_bytes(a.rs.M, a.stages, NF4);
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
  return cudaLaunchKernelEx(&cfg, k_umma<EPI, NF4>, a);
}

template <bool NF4>
static cudaError_t launch_uf(const GemmArgs& a, int epi, cudaStream_t st, bool pdl) {
  switch (epi) {
    case EPI_QKV: return launch_ut<EPI_QKV, NF4>(a, st, pdl);
    case EPI_RESID: return launch_ut<EPI_RESID, NF4>(a, st, pdl);
    case EPI_SWIGLU: return launch_ut<EPI_SWIGLU, NF4>(a, st, pdl);
    case EPI_STORE: return launch_ut<EPI_STORE, NF4>(a, st, pdl);
    case EPI_ARGMAX: return NF4 ? cudaErrorInvalidValue : launch_ut<EPI_ARGMAX, false>(a, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

// Token-row count from which the projections run on this kernel: 17 (above
// one 16-row group of the mma.sync kernel), or SF_UMMA_MIN_ROWS from the
// environment (1..81; read once per process), for comparing the two kernels.
int umma_min_rows() {
  static const int v = [] {
    const char* e = getenv("SF_UMMA_MIN_ROWS");
    const int n = e ? atoi(e) : kGroupRows + 1;
    return n < 1 ? 1 : (n > kRows + 1 ? kRows + 1 : n);
  }();
  return v;
}

// The same threshold for forwards with NF4 weights (SF_UMMA_MIN_ROWS_NF4).
// Default 1: every NF4 forward dequantises each weight tile once into tensor
// memory (the batch-1 14B-shape NF4 verify: 7.2 ms against 8.6 ms on the
// mma.sync kernel on GB300).
int umma_min_rows_nf4() {
  static const int v = [] {
    const char* e = getenv("SF_UMMA_MIN_ROWS_NF4");
    const int n = e ? atoi(e) : 1;
    return n < 1 ? 1 : (n > kRows + 1 ? kRows + 1 : n);
  }();
  return v;
}

cudaError_t launch_umma(const GemmArgs& a, int epi, cudaStream_t st, bool pdl) {
  if (a.rs.M < 1 || a.rs.M > kRows) return cudaErrorInvalidValue;
  if (a.nsplit > (a.cluster ? 8 : 16)) return cudaErrorInvalidValue;
  if (a.stages < 2 || a.stages > kUMaxStages) return cudaErrorInvalidValue;
  if (umma_smem_bytes(a.rs.M, a.stages, a.nf4) > 227 * 1024) return cudaErrorInvalidValue;
  if (a.nf4 && (a.K % 64 || (a.nsplit > 1 && a.cps % 4))) return cudaErrorInvalidValue;
  return a.nf4 ? launch_uf<true>(a, epi, st, pdl) : launch_uf<false>(a, epi, st, pdl);
}

template <int EPI, bool NF4>
static cudaError_t uinit_one() {
  const int smem = umma_smem_bytes(kRows, kUMaxStages, NF4);
  cudaError_t e = cudaFuncSetAttribute(k_umma<EPI, NF4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       std::min(smem, 227 * 1024));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_umma<EPI, NF4>, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

template <bool NF4>
static cudaError_t uinit_t() {
  cudaError_t e;
  if ((e = uinit_one<EPI_QKV, NF4>()) || (e = uinit_one<EPI_RESID, NF4>()) || (e = uinit_one<EPI_SWIGLU, NF4>()))
    return e;
  if (!NF4 && (e = uinit_one<EPI_ARGMAX, false>())) return e;
  return uinit_one<EPI_STORE, NF4>();
}

// Attributes of every instantiation on the current device (called from
// gemm_init, once per device).
cudaError_t umma_init() {
  cudaError_t e = uinit_t<false>();
  if (e != cudaSuccess) return e;
  return uinit_t<true>();
}

// Largest number of clusters of `csize` CTAs resident at once for this
// launch footprint (0 if the query fails).
int umma_max_clusters(int csize, int M, int stages, bool nf4) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize * 512);
  cfg.blockDim = dim3(nf4 ? kUThreadsNf4 : kUThreads);
  cfg.dynamicSmemBytes = umma_smem_bytes(M, stages, nf4);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = csize;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t e = nf4 ? cudaOccupancyMaxActiveClusters(&n, k_umma<EPI_QKV, true>, &cfg)
                            : cudaOccupancyMaxActiveClusters(&n, k_umma<EPI_QKV, false>, &cfg);
  return e == cudaSuccess ? n : 0;
}

}  // namespace sf
