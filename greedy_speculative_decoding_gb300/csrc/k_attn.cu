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

constexpr uint32_t kAttnWaitIters = 1u << 24;

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
  const float v = ldw(a.E, (size_t)tok * a.ld + n, a.f32);
  a.x[(size_t)m * a.H + n] = v;
  act_store(a.frag, m, n, (a.rs.M + 3) / 4, v * ldw(a.gain, n, a.f32), a.umma);
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

// One work item = (sequence b, KV head, range r of R consecutive 64-slot
// chunks, group of up to kTG 16-query tiles); the queries are all rows of the
// sequence times the query heads that read this KV head. The chunks' keys and
// values arrive by 2-D TMA (box 64 dims x 64 slots, 128-byte swizzle) into a
// two-stage ring that runs across the CTA's items, so the next chunk is in
// flight while this one is computed; every query tile of the group is
// computed from one copy. The eight warps split into kTG teams of
// W = 8 / kTG, one per query tile, all tiles at once:
//   S = Q K^T   a team's warp computes 64 / W keys over the whole head
//               dimension (mma.sync m16n8k16, Q as an fp32-accurate bf16
//               hi+lo pair), 8 keys per MMA tile;
//   softmax     online over the range: row max and row sum combined across
//               the team through shared memory (the sums of every 8 keys
//               added in key order), the running max and sum rescaled per
//               chunk;
//   O = P V     P (hi+lo) through shared memory, a team's warp producing
//               HD / W output dimensions from all 64 keys, the running
//               output rescaled per chunk.
// Every score, sum and output element is the same sequence of operations
// whatever W is (W only decides which warp performs it), so kTG can follow
// the row count of each launch. The range's unnormalised output, running max
// and sum go to scratch; the merge kernel combines the ranges of every
// (row, head) in order. R is fixed per model and engine and the ranges start
// at fixed multiples of R chunks, so a row's result does not depend on how
// many other rows the launch carries.
template <int HD, int kTG>
__global__ void __launch_bounds__(kAttnThreads, kTG == 4 ? 1 : 2) k_attn_chunks(const __grid_constant__ AttnArgs a) {
  constexpr int kBox = kKvChunk * 128;          // one TMA box: 64 slots x 64 dims (8 KB)
  constexpr int kHalf = HD / 64;                // boxes per chunk of keys (or values)
  constexpr int kKV = kHalf * kBox;             // one chunk's keys (or values)
  constexpr int kStage = 2 * kKV;
  constexpr int KS = HD / 16;                   // k-steps over the head dimension
  constexpr int WPT = 8 / kTG;                  // warps per query tile
  constexpr int KPW = kKvChunk / WPT;           // keys per warp in S = Q K^T
  constexpr int NKT = KPW / 8;                  // key n-tiles (8 keys each) per warp
  constexpr int NTW = HD / 8 / WPT;             // output n-tiles (8 dimensions each) per warp
  constexpr int HP = HD + 16;                   // query hi / lo row pitch (bf16): 8-bank shift per row
  constexpr int PP = kKvChunk + 8;              // probability tile row pitch (bf16)
  static_assert(kAttnThreads == 256 && kKvChunk == 64 && 8 % kTG == 0, "eight warps over kTG tiles");
  extern __shared__ unsigned char attn_smem_raw[];
  unsigned char* base = attn_smem_raw + ((1024 - (smem_u32(attn_smem_raw) & 1023)) & 1023);
  bf16* sph = reinterpret_cast<bf16*>(base + a.stages * kStage); // [TG][16][PP] P hi
  bf16* spl = sph + kTG * 16 * PP;                               // [TG][16][PP] P lo
  bf16* sq = spl + kTG * 16 * PP;                                // [TG][2][16][HP] queries hi / lo
  __shared__ float red_mx[8][16];                                // per warp: row max of its keys
  __shared__ float red_l[kTG][8][16];                            // per tile and 8 keys: row sums
  __shared__ float m_run[kTG][16], l_run[kTG][16];
  __shared__ __align__(8) uint64_t full[2];

  trace_mark(a.rs, 0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c4 = lane & 3;
  const int ti = warp / WPT, wq = warp % WPT;   // this warp's query tile within the item, its rank there
  // The warps of one query tile meet at a named barrier of their own.
  auto tile_sync = [](int t) { asm volatile("bar.sync %0, %1;" ::"r"(1 + t), "r"(WPT * 32) : "memory"); };
  const int group = a.nq / a.nkv;
  const int rps = a.rs.rps;
  const int Mq = rps * group;
  const int ntiles = (Mq + 15) / 16;
  constexpr int TG = kTG;   // query tiles per item (a.TG)
  const int ntg = (ntiles + TG - 1) / TG;
  const int R = a.R;
  const int NS = a.stages;

  // The lengths were written by kernels that finished before the preceding
  // one started, so they (and the cache slots below this pass's first
  // position) can be read before waiting on the preceding kernel.
  int total = 0;
  for (int b = 0; b < a.B; ++b) {
    const int nch = (a.rs.pos_base[b] + a.rs.pos_off + rps - 1) / kKvChunk + 1;
    total += a.nkv * ((nch + R - 1) / R) * ntg;
  }
  struct Item {
    int b, kvh, r, tg, c0, c1, p0, p_last;
  };
  auto locate = [&](int item) {
    Item it;
    int rest = item;
    for (it.b = 0; it.b < a.B; ++it.b) {
      it.p0 = a.rs.pos_base[it.b] + a.rs.pos_off;
      it.p_last = it.p0 + rps - 1;
      const int n = a.nkv * ((it.p_last / kKvChunk + 1 + R - 1) / R) * ntg;
      if (rest < n) break;
      rest -= n;
    }
    const int nr = (it.p_last / kKvChunk + 1 + R - 1) / R;
    it.kvh = rest / (nr * ntg);
    rest -= it.kvh * nr * ntg;
    it.r = rest / ntg;
    it.tg = rest - it.r * ntg;
    it.c0 = it.r * R;
    it.c1 = min(it.c0 + R, it.p_last / kKvChunk + 1);
    return it;
  };
  auto kv_row = [&](const Item& it, int c) { return a.kv_row0 + it.b * a.kv_brows + it.kvh * a.s_max + c * kKvChunk; };

  // Producer (thread 0): a cursor over (item, chunk) steps of this CTA.
  int is_item = blockIdx.x, is_c = 0, issued = 0;
  Item is_it;
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (is_item < total) {
      is_it = locate(is_item);
      is_c = is_it.c0;
    }
  }
  auto issue_next = [&]() {   // thread 0: load the cursor's chunk into stage issued % NS, advance
    if (is_item >= total) return;
    const int s = issued % NS;
    unsigned char* st = base + s * kStage;
    fence_proxy_async();
    const int row = kv_row(is_it, is_c);
    // Slots past the sequence's last row hold nothing of this pass: with
    // box8 a partly filled last chunk loads only the 8-slot boxes that hold
    // valid slots.
    const int nvalid = min(kKvChunk, is_it.p_last - is_c * kKvChunk + 1);
    if (nvalid < kKvChunk && a.box8) {
      const int nb = (nvalid + 7) / 8;
      mbar_expect_tx(&full[s], 2 * kHalf * nb * 8 * 128);
      for (int h = 0; h < kHalf; ++h)
        for (int i = 0; i < nb; ++i) {
          tma_load_2d(st + h * kBox + i * 1024, &a.kvmap8, 64 * h, row + 8 * i, &full[s], policy_evict_first());
          tma_load_2d(st + kKV + h * kBox + i * 1024, &a.kvmap8, 64 * h, row + a.kv_vrows + 8 * i, &full[s],
                      policy_evict_first());
        }
    } else {
      mbar_expect_tx(&full[s], kStage);
#pragma unroll
      for (int h = 0; h < kHalf; ++h) {
        tma_load_2d(st + h * kBox, &a.kvmap, 64 * h, row, &full[s], policy_evict_first());
        tma_load_2d(st + kKV + h * kBox, &a.kvmap, 64 * h, row + a.kv_vrows, &full[s], policy_evict_first());
      }
    }
    ++issued;
    if (++is_c >= is_it.c1) {
      is_item += gridDim.x;
      if (is_item < total) {
        is_it = locate(is_item);
        is_c = is_it.c0;
      }
    }
  };
  __syncthreads();
  // The first chunk, before the wait when it holds no slot of this pass.
  if (tid == 0 && is_item < total && (is_c + 1) * kKvChunk <= is_it.p0) issue_next();
  pdl_wait();
  trace_mark(a.rs, 1);
  pdl_launch_next();
  if (tid == 0 && issued == 0) issue_next();

  int step = 0;
  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    const Item it = locate(item);
    const int t0 = it.tg * TG, nt = min(TG, ntiles - t0);
    // The item's query tiles -> shared memory as bf16 hi + lo pairs (rows
    // past Mq are zero); the running max and sum start empty.
    {
      // All of a thread's query loads in flight at once, then the splits.
      constexpr int kQB = (kTG * 16 * (HD / 4) + kAttnThreads - 1) / kAttnThreads;
      const int n4 = nt * 16 * (HD / 4);
      float4 qv[kQB];
#pragma unroll
      for (int e = 0; e < kQB; ++e) {
        const int i = tid + e * kAttnThreads;
        qv[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < n4) {
          const int qt = i / (16 * (HD / 4)), rem = i - qt * (16 * (HD / 4));
          const int qr = rem / (HD / 4), u = rem - qr * (HD / 4);
          const int qi = (t0 + qt) * 16 + qr;
          if (qi < Mq) {
            const int j = qi / group, hh = qi - j * group;
            qv[e] = *reinterpret_cast<const float4*>(a.q + ((size_t)(it.b * rps + j) * a.nq + it.kvh * group + hh) * HD +
                                                     4 * u);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < kQB; ++e) {
        const int i = tid + e * kAttnThreads;
        if (i >= n4) break;
        const int qt = i / (16 * (HD / 4)), rem = i - qt * (16 * (HD / 4));
        const int qr = rem / (HD / 4), u = rem - qr * (HD / 4);
        uint2 h, l;
        split_bf16x2(qv[e].x, qv[e].y, h.x, l.x);
        split_bf16x2(qv[e].z, qv[e].w, h.y, l.y);
        *reinterpret_cast<uint2*>(sq + ((2 * qt) * 16 + qr) * HP + 4 * u) = h;
        *reinterpret_cast<uint2*>(sq + ((2 * qt + 1) * 16 + qr) * HP + 4 * u) = l;
      }
      if (tid < kTG * 16) {
        m_run[tid >> 4][tid & 15] = -INFINITY;
        l_run[tid >> 4][tid & 15] = 0.f;
      }
    }
    float oacc[NTW][4];
#pragma unroll
    for (int t2 = 0; t2 < NTW; ++t2) oacc[t2][0] = oacc[t2][1] = oacc[t2][2] = oacc[t2][3] = 0.f;
    __syncthreads();

    for (int c = it.c0; c < it.c1; ++c, ++step) {
      const int s = step % NS;
      // Two stages: the next step's chunk goes into the other one now; one
      // stage: after this step has released it (end of the step).
      if (tid == 0 && NS == 2) issue_next();
      if (!mbar_wait(&full[s], (step / NS) & 1, kAttnWaitIters)) {
        report_err(a.err, kErrWait);
        mbar_wait(&full[s], (step / NS) & 1, kAttnWaitIters);
      }
      const unsigned char* ks = base + s * kStage;
      unsigned char* vs = base + s * kStage + kKV;
      // Slots past the sequence's last row were not written by anyone this
      // pass: zero their values (a zero probability times a stale NaN would
      // still be NaN); their scores are masked below.
      const int nvalid = min(kKvChunk, it.p_last - c * kKvChunk + 1);
      if (nvalid < kKvChunk) {
        for (int i = tid; i < (kKvChunk - nvalid) * 8 * kHalf; i += kAttnThreads) {
          const int r = nvalid + i / (8 * kHalf), rem = i % (8 * kHalf);
          *reinterpret_cast<uint4*>(vs + (rem >> 3) * kBox + r * 128 + (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async();   // ordered before the next copy into this stage
        // Ordered before every team's P V reads: by the team's first barrier
        // when one team is the whole block, else by a block barrier.
        if (kTG > 1) __syncthreads();
      }
      if (ti < nt) {
        const bf16* qht = sq + (2 * ti) * 16 * HP;
        const bf16* qlt = sq + (2 * ti + 1) * 16 * HP;
        bf16* tph = sph + ti * 16 * PP;
        bf16* tpl = spl + ti * 16 * PP;
        // Row j sees the chunk's keys below nk, except [gl, gh): in a
        // multi-candidate verify, the slots of the candidates before its own.
        int nk[2], gl[2], gh[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int qi = (t0 + ti) * 16 + g + 8 * r;
          const int j = qi / group;
          nk[r] = qi < Mq ? min(kKvChunk, it.p0 + j - c * kKvChunk + 1) : 0;
          gl[r] = it.p0 + 1 - c * kKvChunk;
          gh[r] = gl[r] + tree_gap(a.rs, j);
        }
        // S for this warp's keys, 8 at a time (n8 tile t: keys
        // wq*KPW + 8t .. +7): per tile four independent chains (hi / lo part
        // of Q x even / odd k-step), added in a fixed order at the end. Key
        // row `key` of the swizzled tile: dims 8q .. 8q+7 at 16-byte piece
        // q ^ (key & 7).
        float sa[NKT][4][4];
#pragma unroll
        for (int t = 0; t < NKT; ++t)
#pragma unroll
          for (int i = 0; i < 4; ++i) sa[t][i][0] = sa[t][i][1] = sa[t][i][2] = sa[t][i][3] = 0.f;
#pragma unroll
        for (int k = 0; k < KS; ++k) {
          const uint2 h0 = *reinterpret_cast<const uint2*>(qht + g * HP + 16 * k + 4 * c4);
          const uint2 h1 = *reinterpret_cast<const uint2*>(qht + (g + 8) * HP + 16 * k + 4 * c4);
          const uint2 l0 = *reinterpret_cast<const uint2*>(qlt + g * HP + 16 * k + 4 * c4);
          const uint2 l1 = *reinterpret_cast<const uint2*>(qlt + (g + 8) * HP + 16 * k + 4 * c4);
          const int q16 = 2 * (k & 3) + (c4 >> 1);
#pragma unroll
          for (int t = 0; t < NKT; ++t) {
            const int key = wq * KPW + 8 * t + g;
            const uint2 kb = *reinterpret_cast<const uint2*>(ks + (k >> 2) * kBox + key * 128 +
                                                             ((q16 ^ (key & 7)) << 4) + 8 * (c4 & 1));
            mma_bf16_16816(sa[t][k & 1], h0.x, h1.x, h0.y, h1.y, kb.x, kb.y);
            mma_bf16_16816(sa[t][2 + (k & 1)], l0.x, l1.x, l0.y, l1.y, kb.x, kb.y);
          }
        }
        float sacc[NKT][4];
#pragma unroll
        for (int t = 0; t < NKT; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = e >> 1, kk = wq * KPW + 8 * t + 2 * c4 + (e & 1);
            const float v = (sa[t][0][e] + sa[t][1][e]) + (sa[t][2][e] + sa[t][3][e]);
            sacc[t][e] = (kk < nk[r] && (kk < gl[r] || kk >= gh[r])) ? v * a.scale : -INFINITY;
          }
        // Row maxima (exact, so the order of combination does not matter).
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float mx = -INFINITY;
#pragma unroll
          for (int t = 0; t < NKT; ++t) mx = fmaxf(mx, fmaxf(sacc[t][2 * r], sacc[t][2 * r + 1]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          if (c4 == 0) red_mx[warp][g + 8 * r] = mx;
        }
        tile_sync(ti);   // the tile's red_mx complete
        float m_new[2], alpha[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float m8 = red_mx[ti * WPT][g + 8 * r];
#pragma unroll
          for (int w = 1; w < WPT; ++w) m8 = fmaxf(m8, red_mx[ti * WPT + w][g + 8 * r]);
          const float m_old = m_run[ti][g + 8 * r];
          m_new[r] = fmaxf(m_old, m8);
          alpha[r] = m_new[r] == -INFINITY ? 1.f : expf(m_old - m_new[r]);
        }
        // Probabilities; the row sum of every 8 keys (summed over the 64 in
        // key order below); P as bf16 hi + lo through shared memory.
#pragma unroll
        for (int t = 0; t < NKT; ++t) {
          float pe[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) pe[e] = sacc[t][e] != -INFINITY ? expf(sacc[t][e] - m_new[e >> 1]) : 0.f;
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            float l = pe[2 * r] + pe[2 * r + 1];
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            if (c4 == 0) red_l[ti][wq * NKT + t][g + 8 * r] = l;
            uint32_t h, lo;
            split_bf16x2(pe[2 * r], pe[2 * r + 1], h, lo);
            const int col = wq * KPW + 8 * t + 2 * c4;
            *reinterpret_cast<uint32_t*>(tph + (g + 8 * r) * PP + col) = h;
            *reinterpret_cast<uint32_t*>(tpl + (g + 8 * r) * PP + col) = lo;
          }
        }
        tile_sync(ti);   // the tile's P and red_l complete

        // O = O * alpha + P V for this warp's output dimensions (P hi and P lo
        // in two chains, added at the end). Value row `slot`, dims 8n .. 8n+7:
        // 16-byte piece (n & 7) ^ (slot & 7) of box n >> 3.
        float oh[NTW][4], ol[NTW][4];
#pragma unroll
        for (int t2 = 0; t2 < NTW; ++t2)
#pragma unroll
          for (int e = 0; e < 4; ++e) oh[t2][e] = ol[t2][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < kKvChunk / 16; ++kk) {
          uint32_t ph[4], pl[4];
          const int k0 = 16 * kk + 2 * c4;
          ph[0] = *reinterpret_cast<const uint32_t*>(tph + g * PP + k0);
          ph[1] = *reinterpret_cast<const uint32_t*>(tph + (g + 8) * PP + k0);
          ph[2] = *reinterpret_cast<const uint32_t*>(tph + g * PP + k0 + 8);
          ph[3] = *reinterpret_cast<const uint32_t*>(tph + (g + 8) * PP + k0 + 8);
          pl[0] = *reinterpret_cast<const uint32_t*>(tpl + g * PP + k0);
          pl[1] = *reinterpret_cast<const uint32_t*>(tpl + (g + 8) * PP + k0);
          pl[2] = *reinterpret_cast<const uint32_t*>(tpl + g * PP + k0 + 8);
          pl[3] = *reinterpret_cast<const uint32_t*>(tpl + (g + 8) * PP + k0 + 8);
          const int slot = 16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
          for (int t2 = 0; t2 < NTW; ++t2) {
            const int n = wq * NTW + t2;
            uint32_t b0, b1;
            ldsm_x2_trans(b0, b1, vs + (n >> 3) * kBox + slot * 128 + (((n & 7) ^ (slot & 7)) << 4));
            mma_bf16_16816(oh[t2], ph[0], ph[1], ph[2], ph[3], b0, b1);
            mma_bf16_16816(ol[t2], pl[0], pl[1], pl[2], pl[3], b0, b1);
          }
        }
#pragma unroll
        for (int t2 = 0; t2 < NTW; ++t2)
#pragma unroll
          for (int e = 0; e < 4; ++e) oacc[t2][e] = oacc[t2][e] * alpha[e >> 1] + (oh[t2][e] + ol[t2][e]);
        if (wq == 0 && c4 == 0) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            float l = red_l[ti][0][g + 8 * r];
#pragma unroll
            for (int w = 1; w < 8; ++w) l += red_l[ti][w][g + 8 * r];
            l_run[ti][g + 8 * r] = l_run[ti][g + 8 * r] * alpha[r] + l;
            m_run[ti][g + 8 * r] = m_new[r];
          }
        }
      }
      __syncthreads();   // the stage, P, red_* free; running max / sum updated
      if (tid == 0 && NS == 1) issue_next();
    }

    // The range's partial result of every row of this warp's tile that sees a slot of it.
    if (ti < nt) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int qi = (t0 + ti) * 16 + g + 8 * r;
        if (qi >= Mq) continue;
        const int j = qi / group, hh = qi - j * group;
        if (it.p0 + j < it.c0 * kKvChunk) continue;
        const int m = it.b * rps + j, h = it.kvh * group + hh;
        float* dst = a.part + (((size_t)m * a.nq + h) * a.n_kv_chunks + it.r) * (HD + 2);
#pragma unroll
        for (int t2 = 0; t2 < NTW; ++t2)
          *reinterpret_cast<float2*>(dst + 8 * (wq * NTW + t2) + 2 * c4) =
              make_float2(oacc[t2][2 * r], oacc[t2][2 * r + 1]);
        if (wq == 0 && c4 == 0) {
          dst[HD] = m_run[ti][g + 8 * r];
          dst[HD + 1] = l_run[ti][g + 8 * r];
        }
      }
    }
    __syncthreads();   // the query tiles and running state are reused by the next item
  }
}

// One-chunk, one-tile items (a small cache load: R = 1, TG = 1) without the
// TMA ring: work item = (sequence b, KV head, 64-slot chunk c, 16-query tile
// qt); the chunk's keys and values come into padded shared-memory rows with
// 16-byte asynchronous copies issued by every thread (slots past the last
// row's position are zero-filled instead: a zero probability times a stale
// NaN would still be NaN), the first item's before the wait on the
// producing kernel when the chunk holds no slot of this pass. Per tile, the
// same arithmetic as k_attn_chunks with one team of eight warps and an empty
// running state: S by eight keys per warp (Q as bf16 hi + lo, four
// accumulation chains), the chunk's row max and the 8-key sums combined in
// warp order, P (hi + lo) through shared memory, warp w producing output
// dimensions w*HD/8 .. from all 64 keys. Measured faster than the ring
// kernel for these launches (the draft step's and the batch-1 verify's).
template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 2) k_attn_chunk1(const __grid_constant__ AttnArgs a) {
  constexpr int KP = HD * 2 + 32;   // key row pitch (bytes): 8-bank shift per row for the 8-byte fragment loads
  constexpr int VP = HD * 2 + 16;   // value row pitch: 4-bank shift per row for ldmatrix
  constexpr int KS = HD / 16;       // k-steps over the head dimension
  constexpr int NTW = HD / 64;      // output n-tiles (8 dimensions each) per warp
  constexpr int HP = HD + 16;       // query hi / lo row pitch (bf16)
  constexpr int PP = kKvChunk + 8;  // probability tile row pitch (bf16)
  constexpr int kPieces = kKvChunk * HD / 8;   // 16-byte pieces of a chunk's keys (and of its values)
  static_assert(kAttnThreads == 256 && kKvChunk == 64, "eight warps of eight keys");
  extern __shared__ __align__(128) unsigned char attn1_smem[];
  unsigned char* ks = attn1_smem;                                  // [64][KP]
  unsigned char* vs = ks + kKvChunk * KP;                          // [64][VP]
  bf16* sph = reinterpret_cast<bf16*>(vs + kKvChunk * VP);         // [16][PP] P hi
  bf16* spl = sph + 16 * PP;                                       // [16][PP] P lo
  bf16* sqh = spl + 16 * PP;                                       // [16][HP] queries of the tile, hi
  bf16* sql = sqh + 16 * HP;                                       // [16][HP] queries of the tile, lo
  __shared__ float red_mx[8][16], red_l[8][16];

  trace_mark(a.rs, 0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c4 = lane & 3;
  const int group = a.nq / a.nkv;
  const int rps = a.rs.rps;
  const int Mq = rps * group;
  const int ntiles = (Mq + 15) / 16;
  // Lengths and the cache slots below this pass's first position may be
  // read before the wait (see k_attn_chunks).
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

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    int b, kvh, c, qt;
    locate(item, b, kvh, c, qt);
    const int p0 = a.rs.pos_base[b] + a.rs.pos_off;
    if (!issued) issue(b, kvh, c, min(kKvChunk, p0 + rps - c * kKvChunk));
    issued = false;
    // The tile's 16 query rows -> bf16 hi + lo (rows past Mq are zero), all
    // of a thread's loads in flight at once.
    {
      constexpr int kQB = 16 * (HD / 4) / kAttnThreads;
      float4 qv[kQB];
#pragma unroll
      for (int e = 0; e < kQB; ++e) {
        const int i = tid + e * kAttnThreads;
        const int qi = qt * 16 + i / (HD / 4), u = i % (HD / 4);
        qv[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (qi < Mq) {
          const int j = qi / group, hh = qi - j * group;
          qv[e] = *reinterpret_cast<const float4*>(a.q + ((size_t)(b * rps + j) * a.nq + kvh * group + hh) * HD +
                                                   4 * u);
        }
      }
#pragma unroll
      for (int e = 0; e < kQB; ++e) {
        const int i = tid + e * kAttnThreads;
        const int qr = i / (HD / 4), u = i - qr * (HD / 4);
        uint2 h, l;
        split_bf16x2(qv[e].x, qv[e].y, h.x, l.x);
        split_bf16x2(qv[e].z, qv[e].w, h.y, l.y);
        *reinterpret_cast<uint2*>(sqh + qr * HP + 4 * u) = h;
        *reinterpret_cast<uint2*>(sql + qr * HP + 4 * u) = l;
      }
    }
    cp_async_wait_all();
    __syncthreads();

    // Row j sees the chunk's keys below nk, except [gl, gh): in a
    // multi-candidate verify, the slots of the candidates before its own.
    int nk[2], gl[2], gh[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int qi = qt * 16 + g + 8 * r;
      const int j = qi / group;
      nk[r] = qi < Mq ? min(kKvChunk, p0 + j - c * kKvChunk + 1) : 0;
      gl[r] = p0 + 1 - c * kKvChunk;
      gh[r] = gl[r] + tree_gap(a.rs, j);
    }
    float sa[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) sa[i][0] = sa[i][1] = sa[i][2] = sa[i][3] = 0.f;
    const unsigned char* krow = ks + (8 * warp + g) * KP + 8 * c4;
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      const uint2 h0 = *reinterpret_cast<const uint2*>(sqh + g * HP + 16 * k + 4 * c4);
      const uint2 h1 = *reinterpret_cast<const uint2*>(sqh + (g + 8) * HP + 16 * k + 4 * c4);
      const uint2 l0 = *reinterpret_cast<const uint2*>(sql + g * HP + 16 * k + 4 * c4);
      const uint2 l1 = *reinterpret_cast<const uint2*>(sql + (g + 8) * HP + 16 * k + 4 * c4);
      const uint2 kb = *reinterpret_cast<const uint2*>(krow + 32 * k);
      mma_bf16_16816(sa[k & 1], h0.x, h1.x, h0.y, h1.y, kb.x, kb.y);
      mma_bf16_16816(sa[2 + (k & 1)], l0.x, l1.x, l0.y, l1.y, kb.x, kb.y);
    }
    float sacc[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = e >> 1, kk = 8 * warp + 2 * c4 + (e & 1);
      const float v = (sa[0][e] + sa[1][e]) + (sa[2][e] + sa[3][e]);
      sacc[e] = (kk < nk[r] && (kk < gl[r] || kk >= gh[r])) ? v * a.scale : -INFINITY;
    }
    float mx[2];
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
    for (int e = 0; e < 4; ++e) pe[e] = sacc[e] != -INFINITY ? expf(sacc[e] - mx[e >> 1]) : 0.f;
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
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (nk[r] <= 0) continue;   // the row sees no slot of this chunk
      const int qi = qt * 16 + g + 8 * r;
      const int j = qi / group, hh = qi - j * group;
      const int m = b * rps + j, h = kvh * group + hh;
      float* dst = a.part + (((size_t)m * a.nq + h) * a.n_kv_chunks + c) * (HD + 2);
#pragma unroll
      for (int t = 0; t < NTW; ++t)
        *reinterpret_cast<float2*>(dst + 8 * (warp * NTW + t) + 2 * c4) =
            make_float2(oh[t][2 * r] + ol[t][2 * r], oh[t][2 * r + 1] + ol[t][2 * r + 1]);
      if (warp == 0 && c4 == 0) {
        float l = red_l[0][g + 8 * r];
#pragma unroll
        for (int w = 1; w < 8; ++w) l += red_l[w][g + 8 * r];
        dst[HD] = mx[r];
        dst[HD + 1] = l;
      }
    }
    __syncthreads();   // keys, values, P and red_* are free again
  }
}

static int attn1_smem_bytes(int hd) {
  return kKvChunk * (hd * 2 + 32) + kKvChunk * (hd * 2 + 16) + 2 * 16 * (kKvChunk + 8) * 2 + 2 * 16 * (hd + 16) * 2;
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
  const int nparts = (row_slot(a.rs, m) / kKvChunk) / a.R + 1;   // ranges of R chunks the row sees
  const float v = merge_row_head(a.part, a.nq, a.hd, a.n_kv_chunks, m, h, nparts, sm);
  if ((int)threadIdx.x < a.hd) act_store(a.out, m, h * a.hd + threadIdx.x, (a.rs.M + 3) / 4, v, a.umma);
}

// Dynamic shared memory of the chunk kernel: `stages` stages of keys + values
// (1024-byte aligned for the swizzled TMA boxes), P hi + lo, and TG query
// tiles (hi + lo).
static int attn_smem_bytes(int hd, int stages, int tg) {
  return 1024 + stages * 2 * kKvChunk * hd * 2 + tg * 2 * 16 * (kKvChunk + 8) * 2 + tg * 2 * 16 * (hd + 16) * 2;
}

// Dynamic shared-memory limits of the chunk kernels and the largest
// shared-memory carve-out for every kernel of the chain.
cudaError_t attn_init() {
  cudaError_t e;
  const void* chunk_fns[] = {reinterpret_cast<const void*>(k_attn_chunks<128, 1>),
                             reinterpret_cast<const void*>(k_attn_chunks<128, 2>),
                             reinterpret_cast<const void*>(k_attn_chunks<128, 4>),
                             reinterpret_cast<const void*>(k_attn_chunks<64, 1>),
                             reinterpret_cast<const void*>(k_attn_chunks<64, 2>),
                             reinterpret_cast<const void*>(k_attn_chunks<64, 4>)};
  const int hd_of[] = {128, 128, 128, 64, 64, 64}, tg_of[] = {1, 2, 4, 1, 2, 4};
  for (int i = 0; i < 6; ++i)
    if ((e = cudaFuncSetAttribute(chunk_fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  attn_smem_bytes(hd_of[i], 2, tg_of[i]))) != cudaSuccess)
      return e;
  // Largest shared-memory carve-out for every kernel of the chain (see gemm_init).
  for (const void* f : chunk_fns)
    if ((e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
      return e;
  if ((e = cudaFuncSetAttribute(k_attn_chunk1<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn1_smem_bytes(128))) != cudaSuccess ||
      (e = cudaFuncSetAttribute(k_attn_chunk1<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn1_smem_bytes(64))) != cudaSuccess)
    return e;
  const void* fns[] = {reinterpret_cast<const void*>(k_attn_chunk1<128>),
                       reinterpret_cast<const void*>(k_attn_chunk1<64>),
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
  // itself lives on the device): B * nkv * ranges of the whole cache, capped.
  const int ntiles = (a.rs.rps * (a.nq / a.nkv) + 15) / 16;
  const int max_items = a.B * a.nkv * ((a.n_kv_chunks + a.R - 1) / a.R) * ((ntiles + a.TG - 1) / a.TG);
  if (a.TG < 1 || a.TG > 4 || a.stages < 1 || a.stages > 2 || a.R < 1) return cudaErrorInvalidValue;
  cfg.gridDim = dim3(max(1, min(max_items, 2 * num_sms)));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e;
  if (a.TG != 1 && a.TG != 2 && a.TG != 4) return cudaErrorInvalidValue;
  if (a.R == 1 && a.TG == 1 && a.kc && a.vc) {
    // One chunk, one tile per item: the copy kernel (same arithmetic).
    cfg.dynamicSmemBytes = attn1_smem_bytes(a.hd);
    if (a.hd == 128) e = cudaLaunchKernelEx(&cfg, k_attn_chunk1<128>, a);
    else if (a.hd == 64) e = cudaLaunchKernelEx(&cfg, k_attn_chunk1<64>, a);
    else return cudaErrorInvalidValue;
  } else {
    cfg.dynamicSmemBytes = attn_smem_bytes(a.hd, a.stages, a.TG);
    if (a.hd == 128)
      e = a.TG == 4   ? cudaLaunchKernelEx(&cfg, k_attn_chunks<128, 4>, a)
          : a.TG == 2 ? cudaLaunchKernelEx(&cfg, k_attn_chunks<128, 2>, a)
                      : cudaLaunchKernelEx(&cfg, k_attn_chunks<128, 1>, a);
    else if (a.hd == 64)
      e = a.TG == 4   ? cudaLaunchKernelEx(&cfg, k_attn_chunks<64, 4>, a)
          : a.TG == 2 ? cudaLaunchKernelEx(&cfg, k_attn_chunks<64, 2>, a)
                      : cudaLaunchKernelEx(&cfg, k_attn_chunks<64, 1>, a);
    else
      return cudaErrorInvalidValue;
  }
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
